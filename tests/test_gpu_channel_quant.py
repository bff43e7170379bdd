"""GPU parity of the per-channel group quantiser (paperlayer summary, "C. Experiments on
per-channel quantization of keys": group size 64, keys per channel) against the oracle:
codes and (scale, zero) bit-exact for every full group; the pending keys are left alone."""
import numpy as np
import pytest
import torch

from gpu_helpers import dev, to_np
from mixed_precision_kv_balancer_gb300 import _lib
from oracle import channel_quant as cq
from oracle import quant as oq

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("bits,units,n", [(2, 3, 200), (4, 2, 128), (8, 1, 64), (2, 5, 1000), (4, 1, 63)])
def test_channel_quantize_bit_exact(bits, units, n):
    rng = np.random.default_rng(bits * 100 + n)
    k = (rng.standard_normal((units, n, 128)) * np.linspace(0.5, 3, 128)).astype(np.float16)
    if n >= 64:
        k[0, 10, 7] = np.float16(300.0)          # an outlier in one channel of group 0
        k[-1, :64, 3] = np.float16(-2.0)         # a constant channel in group 0 of the last unit
    rb = 128 * bits // 8
    codes = torch.full((units, n, rb), 0xAB, dtype=torch.uint8, device=dev())
    meta = torch.zeros((units, max(n // 64, 1), 128, 2), dtype=torch.float16, device=dev())
    _lib.mikv_channel_quantize(torch.from_numpy(k).to(dev()), bits, codes, meta)
    torch.cuda.synchronize()
    gc, gm = to_np(codes), to_np(meta.view(torch.int16)).view(np.uint16)
    for u in range(units):
        for gi in range(n // 64):
            c_o, m_o = cq.quantize_channel_group(k[u, 64 * gi:64 * gi + 64], bits)
            np.testing.assert_array_equal(gc[u, 64 * gi:64 * gi + 64], oq.pack_codes(c_o, bits))
            np.testing.assert_array_equal(gm[u, gi], m_o)
        # rows of the pending keys are not written
        assert np.all(gc[u, 64 * (n // 64):] == 0xAB)


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_channel_quantize_near_ties_bit_exact(bits):
    """Every channel's 64 values on, or one fp16 step beside, the half-integer points of the
    channel's own grid (both ends present), so the quotient (x - z) / s meets rounding ties:
    the packed fast path and its exact-division fallback must match the oracle."""
    from test_gpu_parity import _tie_rows
    rng = np.random.default_rng(90 + bits)
    qmax = 2 ** bits - 1
    units = 3
    k = np.stack([_tie_rows(rng, 128, qmax)[:, :64].T for _ in range(units)]).astype(np.float16)  # [u][64][128]
    rb = 128 * bits // 8
    codes = torch.zeros((units, 64, rb), dtype=torch.uint8, device=dev())
    meta = torch.zeros((units, 1, 128, 2), dtype=torch.float16, device=dev())
    _lib.mikv_channel_quantize(torch.from_numpy(np.ascontiguousarray(k)).to(dev()), bits, codes, meta)
    torch.cuda.synchronize()
    gc, gm = to_np(codes), to_np(meta.view(torch.int16)).view(np.uint16)
    for u in range(units):
        c_o, m_o = cq.quantize_channel_group(k[u], bits)
        np.testing.assert_array_equal(gm[u, 0], m_o)
        np.testing.assert_array_equal(gc[u], oq.pack_codes(c_o, bits))
