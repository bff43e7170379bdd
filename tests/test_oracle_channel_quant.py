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


def _exact(q, k, v):
    l = (q.astype(np.float64) @ k.astype(np.float64).T) / np.sqrt(q.shape[1])
    p = np.exp(l - l.max(axis=1, keepdims=True))
    return (p @ v.astype(np.float64)) / p.sum(axis=1, keepdims=True)


def test_attention_with_only_pending_keys_is_exact():
    """Fewer than 64 retained keys: all pending in FP16, so attention is exact attention."""
    rng = np.random.default_rng(21)
    q = rng.standard_normal((4, 128)).astype(np.float16)
    k = rng.standard_normal((90, 128)).astype(np.float16)
    v = rng.standard_normal((90, 128)).astype(np.float16)
    r = cq.RetainedKeys(128, 2)
    for row in k[30:]:
        r.append(row)
    assert len(r.groups) == 0
    out, _ = cq.decode_attention_channel_keys(q, k[:30], v[:30], r, v[30:])
    np.testing.assert_allclose(out, _exact(q, k, v), rtol=1e-12, atol=1e-12)


def test_attention_error_shrinks_with_bits():
    rng = np.random.default_rng(22)
    q = rng.standard_normal((4, 128)).astype(np.float16)
    k = rng.standard_normal((1000, 128)).astype(np.float16)
    v = rng.standard_normal((1000, 128)).astype(np.float16)
    want = _exact(q, k, v)
    errs = []
    for bits in (2, 4, 8):
        r = cq.RetainedKeys(128, bits)
        for row in k[200:]:
            r.append(row)
        out, _ = cq.decode_attention_channel_keys(q, k[:200], v[:200], r, v[200:])
        errs.append(np.abs(out - want).max())
    assert errs[0] > errs[1] > errs[2] and errs[2] < 1e-2


def test_per_channel_keys_beat_per_token_on_outlier_channels():
    """The pages' observation (Appendix C): with channel-aligned key outliers, per-channel
    INT2 keys reconstruct the keys better than per-token INT2 keys without the balancer."""
    rng = np.random.default_rng(23)
    k = rng.standard_normal((256, 128)).astype(np.float32)
    k[:, [3, 40, 77, 100]] *= 16.0                       # systematic outlier channels
    k = k.astype(np.float16)
    r = cq.RetainedKeys(128, 2)
    for row in k:
        r.append(row)
    err_channel = np.abs(r.keys_f64() - k.astype(np.float64)).mean()
    codes, meta = oq.quantize_groups(k.astype(np.float32), 2, 64)
    err_token = np.abs(oq.dequantize(codes, meta, 64) - k.astype(np.float64)).mean()
    assert err_channel < 0.5 * err_token


@pytest.mark.parametrize("bits", [2, 4])
def test_full_groups_on_an_exact_grid_give_exact_attention(bits):
    """Keys whose every channel, within each group of 64, lies on a grid z_c + j * s_c with
    s_c a power of two and both ends j = 0 and j = qmax present: the quantiser finds
    s = (max - min) / qmax = s_c and z = min exactly, every code is the grid index, and the
    dequantised keys are the keys themselves.  Attention over two full groups and 20 pending
    keys is then exactly softmax attention over the original keys (scipy's softmax here)."""
    from scipy.special import softmax
    rng = np.random.default_rng(40 + bits)
    qmax = 2 ** bits - 1
    D, n_groups, n_pending = 128, 2, 20
    rows = []
    for _ in range(n_groups):
        s_c = 2.0 ** -rng.integers(2, 6, size=D)                 # per channel, exact in fp16
        z_c = rng.integers(-40, 40, size=D) * s_c
        j = rng.integers(0, qmax + 1, size=(64, D))
        j[0], j[1] = 0, qmax                                       # both ends in every channel
        x = z_c + j * s_c
        assert np.array_equal(x.astype(np.float16).astype(np.float64), x)   # exact in fp16
        rows.append(x.astype(np.float16))
    pend = rng.standard_normal((n_pending, D)).astype(np.float16)
    k_lo = np.concatenate(rows + [pend])
    r = cq.RetainedKeys(D, bits)
    for row in k_lo:
        r.append(row)
    assert len(r.groups) == n_groups and len(r.pending) == n_pending
    np.testing.assert_array_equal(r.keys_f64(), k_lo.astype(np.float64))
    q = rng.standard_normal((4, D)).astype(np.float16)
    k_hi = rng.standard_normal((30, D)).astype(np.float16)
    v = rng.standard_normal((30 + len(k_lo), D)).astype(np.float16)
    out, lse = cq.decode_attention_channel_keys(q, k_hi, v[:30], r, v[30:])
    k_all = np.concatenate([k_hi, k_lo]).astype(np.float64)
    w = softmax(q.astype(np.float64) @ k_all.T / np.sqrt(D), axis=1)
    np.testing.assert_allclose(out, w @ v.astype(np.float64), rtol=1e-12, atol=1e-13)
