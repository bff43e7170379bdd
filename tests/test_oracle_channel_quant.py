"""Pins for the oracle's per-channel key quantisation and its pending-token buffering
(paperlayer summary, "C. Experiments on per-channel quantization of keys": group size 64,
per channel; MiKV reading notes, Appendix C: buffering until a group is full)."""
from pathlib import Path

import numpy as np
import pytest

from oracle import channel_quant as cq
from oracle import quant as oq

GOLDEN = Path(__file__).parent / "golden" / "channel_quant_hand.txt"


def _golden():
    rows = {}
    for line in GOLDEN.read_text().splitlines():
        if not line.strip() or line.startswith("#"):
            continue
        key, val = [p.strip() for p in line.split("|")]
        rows[key] = np.array([float(x) for x in val.split()])
    return rows


def test_hand_derived_group():
    g = _golden()
    k = np.stack([g[f"t{i}"] for i in range(4)]).astype(np.float16)
    codes, meta = cq.quantize_channel_group(k, 2)
    np.testing.assert_array_equal(codes[:, 0], g["c0"])
    np.testing.assert_array_equal(codes[:, 1], g["c1"])
    np.testing.assert_array_equal(meta[:, 0].view(np.float16).astype(np.float64), g["scale"])
    np.testing.assert_array_equal(meta[:, 1].view(np.float16).astype(np.float64), g["zero"])
    np.testing.assert_array_equal(cq.dequantize_channel_group(codes, meta), k.astype(np.float64))


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_error_bound_and_channel_independence(bits):
    rng = np.random.default_rng(bits)
    k = rng.standard_normal((64, 128)).astype(np.float16)
    codes, meta = cq.quantize_channel_group(k, bits)
    s = meta[:, 0].view(np.float16).astype(np.float64)
    err = np.abs(cq.dequantize_channel_group(codes, meta) - k.astype(np.float64))
    # half a step per channel, plus the fp16 rounding of the zero point and of the step
    assert np.all(err <= s / 2 + 2e-3 * (np.abs(k).max(axis=0) + 1) + 1e-9)
    # a huge outlier in channel 5 changes channel 5 only (per token it would move every
    # channel of its token's group)
    k2 = k.copy()
    k2[17, 5] = np.float16(400.0)
    codes2, meta2 = cq.quantize_channel_group(k2, bits)
    others = np.arange(128) != 5
    np.testing.assert_array_equal(codes2[:, others], codes[:, others])
    np.testing.assert_array_equal(meta2[others], meta[others])
    tok_codes, _ = oq.quantize_groups(k.astype(np.float32), bits, 64)
    tok_codes2, _ = oq.quantize_groups(k2.astype(np.float32), bits, 64)
    assert np.any(tok_codes2[17, :64] != tok_codes[17, :64])


def test_constant_channel():
    k = np.zeros((64, 4), dtype=np.float16)
    k[:, 2] = np.float16(1.5)
    codes, meta = cq.quantize_channel_group(k, 2)
    assert np.all(codes == 0)
    assert np.all(meta[:, 0].view(np.float16) == 0)
    assert meta[2, 1].view(np.float16) == np.float16(1.5)


@pytest.mark.parametrize("n", [0, 1, 63, 64, 65, 200])
def test_pending_buffer(n):
    rng = np.random.default_rng(n)
    rows = rng.standard_normal((n, 128)).astype(np.float16)
    r = cq.RetainedKeys(128, 2)
    for x in rows:
        r.append(x)
    assert len(r) == n
    assert len(r.groups) == n // 64 and len(r.pending) == n % 64
    keys = r.keys_f64()
    assert keys.shape == (n, 128)
    # pending keys are exact; every full group equals its own one-shot quantisation
    np.testing.assert_array_equal(keys[64 * (n // 64):], rows[64 * (n // 64):].astype(np.float64))
    for gi in range(n // 64):
        c, m = cq.quantize_channel_group(rows[64 * gi:64 * gi + 64], 2)
        np.testing.assert_array_equal(keys[64 * gi:64 * gi + 64], cq.dequantize_channel_group(c, m))
