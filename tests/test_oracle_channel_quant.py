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


# ------------------------------------------------------------------ the composed cache
def _textbook(q, k, v):
    """float64 softmax attention by torch's scaled_dot_product_attention (an independent routine)."""
    import torch
    qt = torch.from_numpy(q.astype(np.float64))[None, :, None, :]
    kt = torch.from_numpy(k.astype(np.float64))[None, None].expand(1, q.shape[0], -1, -1)
    vt = torch.from_numpy(v.astype(np.float64))[None, None].expand(1, q.shape[0], -1, -1)
    return torch.nn.functional.scaled_dot_product_attention(qt, kt, vt)[0, :, 0].numpy()


def _binary_inputs(rng, B, Hkv, L, D, bits):
    """Keys that take two values per (key head, channel), z_c and z_c + qmax s_c, and values
    that take two values per (token, 64-channel group), a and a + qmax sigma, with power-of-two
    steps: any group of them quantises exactly (both ends present, or a constant channel /
    group with scale 0), per channel or per token, so the whole cache reconstructs K and V."""
    qmax = 2 ** bits - 1
    s = 2.0 ** -rng.integers(3, 6, size=(B, Hkv, 1, D))
    z = rng.integers(-8, 8, size=(B, Hkv, 1, D)) * s
    k = (z + qmax * s * rng.integers(0, 2, size=(B, Hkv, L, D))).astype(np.float16)
    sig = 2.0 ** -rng.integers(3, 6, size=(B, Hkv, L, 2, 1))
    a = rng.integers(-8, 8, size=(B, Hkv, L, 2, 1)) * sig
    v = (a + qmax * sig * rng.integers(0, 2, size=(B, Hkv, L, 2, 64))).reshape(B, Hkv, L, D).astype(np.float16)
    assert np.array_equal(k.astype(np.float64), z + qmax * s * (k.astype(np.float64) != z))
    return k, v


@pytest.mark.parametrize("bits", [2, 4])
def test_channel_cache_on_binary_inputs_is_exact_attention(bits):
    """Prefill (H2O selection, 2 full groups + 32 waiting pairs per unit) and 45 decode steps
    (a pair demoted on 4 steps of 5; the third group closes on the way): every step's output
    equals softmax attention over all L tokens' original keys and values, since every pair is
    kept (FP16 or quantised exactly) and none is lost or duplicated.  The positions of both
    tiers partition 0 .. L - 1 at every step."""
    rng = np.random.default_rng(60 + bits)
    B, Hq, Hkv, T, D, steps = 1, 4, 2, 200, 128, 45
    k, v = _binary_inputs(rng, B, Hkv, T + steps, D, bits)
    q = rng.standard_normal((B, Hq, T + steps, D)).astype(np.float16)
    cache, _ = cq.prefill_channel(q[:, :, :T], k[:, :, :T], v[:, :, :T], lo_bits=bits, budget_pct=20,
                                  window=8, extra_steps=steps)
    assert (cache.n_hi, cache.n_lo, cache.n_pending) == (40, 160, 32)
    closed = False
    for s in range(steps):
        L = T + s + 1
        out, _, _ = cq.decode_step_channel(cache, q[:, :, L - 1], k[:, :, L - 1], v[:, :, L - 1], L - 1,
                                           budget_pct=20, window=8)
        for g in range(Hkv):
            pos = sorted(cache.pos_hi[0, g, :cache.n_hi].tolist() + cache.pos_lo[0, g, :cache.n_lo].tolist())
            assert pos == list(range(L))
            hs = slice(g * 2, g * 2 + 2)
            want = _textbook(q[0, hs, L - 1], k[0, g, :L], v[0, g, :L])
            np.testing.assert_allclose(out[0, hs], want, rtol=1e-11, atol=1e-12)
        closed |= cache.n_lo >= 192
    assert closed and cache.n_lo // 64 == 3


def test_the_64th_pair_closes_the_group():
    """Counts and slot order: 160 evicted tokens give two groups and 32 waiting pairs in
    position order; demoted pairs wait in order of arrival; the 32nd demotion closes the third
    group, whose slots 128 .. 191 hold the 32 waiting evicted positions then the 32 victims,
    and whose keys dequantise to the original keys of those tokens (binary inputs)."""
    rng = np.random.default_rng(70)
    B, Hq, Hkv, T, D = 1, 2, 1, 200, 128
    k, v = _binary_inputs(rng, B, Hkv, T, D, 2)
    q = rng.standard_normal((B, Hq, T, D)).astype(np.float16)
    cache, info = cq.prefill_channel(q, k, v, lo_bits=2, budget_pct=40, window=8, extra_steps=0)
    assert (cache.n_hi, cache.n_lo, cache.n_pending) == (80, 120, 56)
    # demote 8 times by hand: important slot 0 each time (swap-remove keeps the tier dense)
    victims = []
    for i in range(8):
        victims.append(int(cache.pos_hi[0, 0, 0]))
        cache.demote(np.zeros((1, 1), np.int32))
        assert cache.n_pending == (57 + i) % 64
    assert cache.n_lo == 128 and cache.n_pending == 0
    np.testing.assert_array_equal(cache.pos_lo[0, 0, 64:128],
                                  np.concatenate([info["evict_pos"][0, 0, 64:120], victims]))
    r, _ = cache.retained(0, 0)
    assert len(r.groups) == 2 and not r.pending
    np.testing.assert_array_equal(r.keys_f64()[64:], k[0, 0, cache.pos_lo[0, 0, 64:128]].astype(np.float64))


def test_channel_cache_with_only_waiting_pairs_is_exact():
    """Fewer than 64 retained tokens: every retained pair waits in FP16, so attention over the
    cache is exact attention over the prompt, whatever the inputs."""
    rng = np.random.default_rng(71)
    q = rng.standard_normal((1, 4, 80, 128)).astype(np.float16)
    k = rng.standard_normal((1, 2, 80, 128)).astype(np.float16)
    v = rng.standard_normal((1, 2, 80, 128)).astype(np.float16)
    cache, _ = cq.prefill_channel(q, k, v, lo_bits=2, budget_pct=40, window=8)
    assert cache.n_lo == 48 and cache.n_pending == 48
    out, _, _ = cache.attend(q[:, :, -1])
    for g in range(2):
        want = _textbook(q[0, 2 * g:2 * g + 2, -1], k[0, g], v[0, g])
        np.testing.assert_allclose(out[0, 2 * g:2 * g + 2], want, rtol=1e-11, atol=1e-12)
