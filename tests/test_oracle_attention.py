"""Pins for the oracle's decode attention and the composed pipeline (no GPU).

Definitions: MiKV notes "2) Outlier-aware handling" (quantised keys hold
I(k*b), queries divided by b) and section 3.4 (permutation invariance, tiers
grouped by precision, Q and the attention map in floating point).
"""
import numpy as np
import pytest
import torch

from oracle import attention, pipeline, quant, select


def _textbook(q, k, v):
    """float64 softmax attention by torch's scaled_dot_product_attention (an independent routine)."""
    qt = torch.from_numpy(q.astype(np.float64))[None, :, None, :]          # [1, H, 1, D]
    kt = torch.from_numpy(k.astype(np.float64))[None, None].expand(1, q.shape[0], -1, -1)
    vt = torch.from_numpy(v.astype(np.float64))[None, None].expand(1, q.shape[0], -1, -1)
    return torch.nn.functional.scaled_dot_product_attention(qt, kt, vt)[0, :, 0].numpy()


def _inputs(rng, B=1, Hq=4, Hkv=2, T=96, D=128, out=16.0):
    gain_q = np.ones((Hq, D)); gain_q[:, rng.choice(D, 4, replace=False)] = out
    gain_k = np.ones((Hkv, D)); gain_k[:, rng.choice(D, 4, replace=False)] = out
    q = (rng.standard_normal((B, Hq, T, D)) * gain_q[None, :, None]).astype(np.float16)
    k = (rng.standard_normal((B, Hkv, T, D)) * gain_k[None, :, None]).astype(np.float16)
    v = rng.standard_normal((B, Hkv, T, D)).astype(np.float16)
    return q, k, v


def test_full_fp16_budget_is_textbook_attention():
    rng = np.random.default_rng(0)
    q, k, v = _inputs(rng)
    cache, _ = pipeline.prefill(q, k, v, hi_bits=16, lo_bits=2, budget_pct=100, window=8)
    assert cache.n_lo == 0 and cache.n_hi == 96
    qd = q[:, :, -1]
    out, lse, _ = cache.attend(qd)
    for h in range(4):
        ref = _textbook(qd[0, h:h + 1], k[0, h // 2], v[0, h // 2])[0]
        np.testing.assert_allclose(out[0, h], ref, rtol=1e-10, atol=1e-12)
        l = (qd[0, h].astype(np.float64) @ k[0, h // 2].astype(np.float64).T) / np.sqrt(128)
        assert abs(lse[0, h] - (l.max() + np.log(np.exp(l - l.max()).sum()))) < 1e-10


def test_quantised_tier_uses_q_over_b():
    """Keys built so that k*b lies exactly on the quantisation grid: the low tier then
    reconstructs k*b exactly and attention must equal textbook attention on the original
    (q, k).  Using q instead of q/b on that tier fails this."""
    D, T = 128, 40
    rng = np.random.default_rng(1)
    b = np.ones(D, np.float32)
    b[:32] = 2.0
    b[32:48] = 0.5
    # k*b = code * 0.25 + (-1): codes 0..15 (INT4 grid), each group spans all 16 levels
    codes = np.tile(np.arange(16), (T, D // 16)).astype(np.float64)
    for t in range(T):
        rng.shuffle(codes[t, :64]); rng.shuffle(codes[t, 64:])
    kb = codes * 0.25 - 1.0
    k = (kb / b.astype(np.float64)).astype(np.float16)
    assert np.array_equal(k.astype(np.float32) * b, kb.astype(np.float32))
    v = (np.tile(np.arange(16), (T, D // 16)) * 0.5 - 2.0).astype(np.float16)
    q = (rng.standard_normal((2, D)) * 2).astype(np.float16)
    xk = quant.balance_keys(k, b)
    kc, km = quant.quantize_groups(xk, 4, 64)
    vc, vm = quant.quantize_groups(v.astype(np.float32), 4, 64)
    np.testing.assert_array_equal(quant.dequantize(kc, km, 64), kb)
    lo = dict(n=T, k=quant.pack_codes(kc, 4), v=quant.pack_codes(vc, 4), k_meta=km, v_meta=vm)
    hi = dict(n=0, k=np.zeros((0, D), np.uint16), v=np.zeros((0, D), np.uint16),
              k_meta=None, v_meta=None)
    out, _, _ = attention.decode_attention_unit(q, hi, lo, b, 16, 4, 64)
    ref = _textbook(q, k, v)
    np.testing.assert_allclose(out, ref, rtol=1e-9, atol=1e-11)


def test_permutation_invariance_of_slots():
    rng = np.random.default_rng(2)
    q, k, v = _inputs(rng, T=80)
    cache, _ = pipeline.prefill(q, k, v, hi_bits=16, lo_bits=4, budget_pct=30, window=8)
    qd = q[:, :, -1]
    out0, lse0, _ = cache.attend(qd)
    perm_hi = rng.permutation(cache.n_hi)
    perm_lo = rng.permutation(cache.n_lo)
    for name, perm, n in (("k_hi", perm_hi, cache.n_hi), ("v_hi", perm_hi, cache.n_hi),
                          ("k_lo", perm_lo, cache.n_lo), ("v_lo", perm_lo, cache.n_lo),
                          ("k_lo_meta", perm_lo, cache.n_lo), ("v_lo_meta", perm_lo, cache.n_lo)):
        arr = getattr(cache, name)
        arr[:, :, :n] = arr[:, :, perm]
    out1, lse1, _ = cache.attend(qd)
    np.testing.assert_allclose(out1, out0, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse1, lse0, rtol=1e-13)


def test_tiers_partition_the_prompt():
    rng = np.random.default_rng(3)
    q, k, v = _inputs(rng, B=2, T=120)
    cache, info = pipeline.prefill(q, k, v, hi_bits=8, lo_bits=2, budget_pct=25, window=16)
    keep = select.n_keep(120, 25, 16)
    assert cache.n_hi == keep and cache.n_lo == 120 - keep
    for b in range(2):
        for g in range(2):
            ph = cache.pos_hi[b, g, :cache.n_hi]
            pl = cache.pos_lo[b, g, :cache.n_lo]
            assert sorted(ph.tolist() + pl.tolist()) == list(range(120))
            assert set(range(104, 120)) <= set(ph.tolist())         # recent window kept
            np.testing.assert_array_equal(cache.scores[b, g, :keep], info["S"][b, g, ph])


def test_decode_loop_invariants():
    """Per step the high tier grows by one, is trimmed back to n_keep(L), the window stays,
    and each score grows by at most rep (one probability per query head)."""
    rng = np.random.default_rng(4)
    B, Hq, Hkv, T, D = 1, 4, 2, 64, 128
    q, k, v = _inputs(rng, B, Hq, Hkv, T + 6, D)
    cache, _ = pipeline.prefill(q[:, :, :T], k[:, :, :T], v[:, :, :T], hi_bits=16, lo_bits=4,
                                budget_pct=20, window=8, extra_steps=6)
    for s in range(6):
        L = T + s + 1
        before = {int(p): float(x) for p, x in zip(cache.pos_hi[0, 0, :cache.n_hi], cache.scores[0, 0, :cache.n_hi])}
        out, lse, victims = pipeline.decode_step(cache, q[:, :, T + s], k[:, :, T + s], v[:, :, T + s],
                                                 L - 1, budget_pct=20, window=8)
        assert cache.n_hi == select.n_keep(L, 20, 8)
        assert cache.n_hi + cache.n_lo == L
        ph = cache.pos_hi[0, 0, :cache.n_hi].tolist()
        assert set(range(L - 8, L)) <= set(ph)
        for p, x in zip(ph, cache.scores[0, 0, :cache.n_hi]):
            if p in before:
                assert before[p] <= x <= before[p] + 2 + 1e-12
        all_pos = sorted(ph + cache.pos_lo[0, 0, :cache.n_lo].tolist())
        assert all_pos == list(range(L))


def test_demoted_int8_token_requantised_from_its_int8_value():
    """INT8 important tier: the demoted token's low-bit codes are those of its float32 INT8
    dequantisation (already balanced), not of the original key."""
    rng = np.random.default_rng(5)
    q, k, v = _inputs(rng, 1, 2, 1, 50, 128)
    cache, _ = pipeline.prefill(q, k, v, hi_bits=8, lo_bits=2, budget_pct=50, window=4, extra_steps=2)
    j = 3
    kc = quant.unpack_codes(cache.k_hi[0, 0, j], 8, 128)
    x = quant.dequantize_f32(kc, cache.k_hi_meta[0, 0, j], 64)
    want, want_m = quant.quantize_groups(x, 2, 64)
    n_lo = cache.n_lo
    cache.demote(np.array([[j]], np.int32))
    np.testing.assert_array_equal(quant.unpack_codes(cache.k_lo[0, 0, n_lo], 2, 128), want)
    np.testing.assert_array_equal(cache.k_lo_meta[0, 0, n_lo], want_m)


def test_budget_zero_is_uniform_rtn():
    """Budget 0 with no window: every token is in the low tier, in position order, each slot
    holding the per-token quantisation of its own (balanced) key and value, and attention is
    softmax attention (torch's) over the dequantised keys s*code + z with q / b."""
    rng = np.random.default_rng(6)
    B, Hq, Hkv, T, D = 1, 4, 2, 80, 128
    q, k, v = _inputs(rng, B, Hq, Hkv, T, D)
    cache, info = pipeline.prefill(q, k, v, hi_bits=16, lo_bits=4, budget_pct=0, window=0)
    assert cache.n_hi == 0 and cache.n_lo == T
    b = info["balancer"]
    qd = q[:, :, -1]
    out, _, _ = cache.attend(qd)
    for g in range(Hkv):
        np.testing.assert_array_equal(cache.pos_lo[0, g, :T], np.arange(T))
        for t in (0, 17, T - 1):
            xk = k[0, g, t].astype(np.float32) * b[0, g]
            kc, km = quant.quantize_groups(xk.astype(np.float32), 4, 64)
            vc, vm = quant.quantize_groups(v[0, g, t].astype(np.float32), 4, 64)
            np.testing.assert_array_equal(cache.k_lo[0, g, t], quant.pack_codes(kc, 4))
            np.testing.assert_array_equal(cache.k_lo_meta[0, g, t], km)
            np.testing.assert_array_equal(cache.v_lo[0, g, t], quant.pack_codes(vc, 4))
            np.testing.assert_array_equal(cache.v_lo_meta[0, g, t], vm)
        # dequantised rows by hand: fp16 scale and zero per 64-channel group
        codes_k = np.unpackbits(cache.k_lo[0, g, :T, :, None], axis=2, bitorder="little")
        codes_k = codes_k.reshape(T, D, 4) @ (1 << np.arange(4))
        codes_v = np.unpackbits(cache.v_lo[0, g, :T, :, None], axis=2, bitorder="little")
        codes_v = codes_v.reshape(T, D, 4) @ (1 << np.arange(4))
        mk = cache.k_lo_meta[0, g, :T].view(np.float16).astype(np.float64)      # [T, 2, 2]
        mv = cache.v_lo_meta[0, g, :T].view(np.float16).astype(np.float64)
        grp = np.arange(D) // 64
        kt = mk[:, grp, 0] * codes_k + mk[:, grp, 1]
        vt = mv[:, grp, 0] * codes_v + mv[:, grp, 1]
        for h in range(g * 2, g * 2 + 2):
            qb = qd[0, h].astype(np.float64) / b[0, g].astype(np.float64)
            ref = _textbook(qb[None], kt, vt)[0]
            np.testing.assert_allclose(out[0, h], ref, rtol=1e-10, atol=1e-12)


def test_two_demotions_traced_by_hand():
    """Two decode steps with a zero query (every logit 0, so each step adds 1/L to every
    important score and leaves their order alone), traced by hand.

    Prompt of 10 tokens; important slots hold positions [0, 3, 5, 7, 9] with scores
    [2, 0.5, 0.5, 1, 0.25]; budget 48 %, window 2.
    Step 1 (L = 11): token 10 joins at slot 5 with score 0, every score gains a = 1/11;
      n_keep(11) = 5 < 6, so one demotion.  Candidates are positions < 9: slots 0-3.  The
      lowest score, 0.5 + a, is shared by positions 3 and 5; the later one, 5 (slot 2), is
      the victim.  Slot 5 (position 10, score a) moves into slot 2: positions
      [0, 3, 10, 7, 9]; the low tier's slot 5 takes position 5.
    Step 2 (L = 12): token 11 joins at slot 5 with score 0, every score gains b = 1/12;
      n_keep(12) = 5 < 6.  Candidates are positions < 10: slots 0, 1, 3, 4 (position 10 in
      slot 2 is in the window).  Lowest: slot 4 (position 9, 0.25 + a + b).  Slot 5
      (position 11, score b) moves into slot 4: positions [0, 3, 10, 7, 11], scores
      [2+a+b, 0.5+a+b, a+b, 1+a+b, b]; the low tier's slot 6 takes position 9.
    With a zero query the output is the plain mean of the attended values."""
    rng = np.random.default_rng(9)
    D = 128
    k = rng.standard_normal((1, 1, 12, D)).astype(np.float16)
    v = rng.standard_normal((1, 1, 12, D)).astype(np.float16)
    cache = pipeline.OracleCache(1, 1, 1, D, 64, 16, 4, 8, 8, None)
    hi_pos = np.array([[[0, 3, 5, 7, 9]]], np.int32)
    cache.append("hi", k, v, hi_pos, 0, np.array([[[2.0, 0.5, 0.5, 1.0, 0.25]]]))
    cache.append("lo", k, v, np.array([[[1, 2, 4, 6, 8]]], np.int32), 0)
    q0 = np.zeros((1, 1, D), np.float16)
    a, b_ = 1.0 / 11, 1.0 / 12
    row = lambda t: k[0, 0, t].view(np.uint16)

    out, _, vic = pipeline.decode_step(cache, q0, k[:, :, 10], v[:, :, 10], 10, budget_pct=48, window=2)
    assert vic[0, 0] == 2
    np.testing.assert_array_equal(cache.pos_hi[0, 0, :5], [0, 3, 10, 7, 9])
    np.testing.assert_allclose(cache.scores[0, 0, :5], [2 + a, 0.5 + a, a, 1 + a, 0.25 + a], rtol=1e-15)
    np.testing.assert_array_equal(cache.k_hi[0, 0, 2], row(10))
    np.testing.assert_array_equal(cache.pos_lo[0, 0, :6], [1, 2, 4, 6, 8, 5])
    kc, km = quant.quantize_groups(k[0, 0, 5].astype(np.float32), 4, 64)
    np.testing.assert_array_equal(cache.k_lo[0, 0, 5], quant.pack_codes(kc, 4))
    np.testing.assert_array_equal(cache.k_lo_meta[0, 0, 5], km)

    out, _, vic = pipeline.decode_step(cache, q0, k[:, :, 11], v[:, :, 11], 11, budget_pct=48, window=2)
    assert vic[0, 0] == 4
    np.testing.assert_array_equal(cache.pos_hi[0, 0, :5], [0, 3, 10, 7, 11])
    np.testing.assert_allclose(cache.scores[0, 0, :5], [2 + a + b_, 0.5 + a + b_, a + b_, 1 + a + b_, b_],
                               rtol=1e-15)
    np.testing.assert_array_equal(cache.k_hi[0, 0, 4], row(11))
    np.testing.assert_array_equal(cache.pos_lo[0, 0, :7], [1, 2, 4, 6, 8, 5, 9])
    assert (cache.n_hi, cache.n_lo) == (5, 7)
    # the second step attended 6 important rows (FP16) and 6 low rows (dequantised), weight 1/12 each
    hi_v = v[0, 0, [0, 3, 10, 7, 9, 11]].astype(np.float64)
    lo_v = [quant.dequantize(*quant.quantize_groups(v[0, 0, t].astype(np.float32), 4, 64), 64)
            for t in (1, 2, 4, 6, 8, 5)]
    want = (hi_v.sum(axis=0) + np.sum(lo_v, axis=0)) / 12
    np.testing.assert_allclose(out[0, 0], want, rtol=1e-12, atol=1e-14)
