"""GPU parity of the per-channel key cache (MIKV_KEYS_PER_CHANNEL) against the oracle's
ChannelKeyCache (paperlayer summary, "C. Experiments on per-channel quantization of keys";
MiKV reading notes, Appendix C remarks).

Bars: bit-exact for codes, key meta per (group, channel), value meta per token, positions and
the waiting FP16 pairs; H2O scores normwise 1e-5; attention within 2e-3 and 1e-4.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import ATTN_TOL, SCORE_RTOL, dev, to_np, u16
from mixed_precision_kv_balancer_gb300 import _lib, inputs
from mixed_precision_kv_balancer_gb300.cache import MikvCache
from oracle import channel_quant as cq
from oracle import select as osel

pytestmark = pytest.mark.gpu

CH = _lib.MIKV_KEYS_PER_CHANNEL


def _np(x):
    return {k: v.numpy() for k, v in x.items()}


def compare_unit(gc, oc, b, g, bo=None, go=None):
    """Bit-exact comparison of unit (b, g) of the library cache with unit (bo, go) of the oracle's."""
    bo = b if bo is None else bo
    go = g if go is None else go
    assert (gc.n_hi, gc.n_lo) == (oc.n_hi, oc.n_lo)
    nh, nl = oc.n_hi, oc.n_lo
    nfull = nl - nl % 64
    np.testing.assert_array_equal(u16(gc.k_hi[b, g, :nh]), oc.k_hi[bo, go, :nh])
    np.testing.assert_array_equal(u16(gc.v_hi[b, g, :nh]), oc.v_hi[bo, go, :nh])
    np.testing.assert_array_equal(to_np(gc.pos_hi[b, g, :nh]), oc.pos_hi[bo, go, :nh])
    np.testing.assert_array_equal(to_np(gc.k_lo[b, g, :nfull]), oc.k_lo[bo, go, :nfull])
    np.testing.assert_array_equal(u16(gc.k_lo_meta[b, g, :nfull // 64]), oc.k_lo_meta[bo, go, :nfull // 64])
    np.testing.assert_array_equal(to_np(gc.v_lo[b, g, :nfull]), oc.v_lo[bo, go, :nfull])
    np.testing.assert_array_equal(u16(gc.v_lo_meta[b, g, :nfull]), oc.v_lo_meta[bo, go, :nfull])
    np.testing.assert_array_equal(to_np(gc.pos_lo[b, g, :nl]), oc.pos_lo[bo, go, :nl])
    np.testing.assert_array_equal(u16(gc.k_pend[b, g, :nl % 64]), oc.k_pend[bo, go, :nl % 64])
    np.testing.assert_array_equal(u16(gc.v_pend[b, g, :nl % 64]), oc.v_pend[bo, go, :nl % 64])


def compare_all(gc, oc):
    for b in range(gc.B):
        for g in range(gc.Hkv):
            compare_unit(gc, oc, b, g)


CASES = [
    # lo, B, Hq, Hkv, T, p, W
    (2, 1, 4, 4, 512, 20, 32),     # the tiny workload's shape: 6 closed groups + 26 waiting
    (4, 2, 8, 2, 300, 25, 16),     # GQA 4, INT4
    (2, 1, 10, 2, 200, 40, 8),     # GQA 5 (two n-tiles)
    (2, 2, 8, 8, 100, 50, 8),      # fewer than 64 retained: all waiting
    (4, 1, 8, 2, 64 + 16, 20, 16), # exactly one closed group, nothing waiting
]


@pytest.mark.parametrize("lo,B,Hq,Hkv,T,p,W", CASES)
def test_channel_prefill_and_attention(lo, B, Hq, Hkv, T, p, W):
    wl = inputs.WORKLOADS["tiny"].scaled(B=B, Hq=Hq, Hkv=Hkv, T=T + 1, lo_bits=lo, n_outlier=8)
    x = inputs.make_prefill(wl, 5, "cpu")
    xn = _np(x)
    qT = {k: v[:, :, :T] for k, v in xn.items()}
    oc, info = cq.prefill_channel(qT["q"], qT["k"], qT["v"], lo_bits=lo, budget_pct=p, window=W)
    keep = osel.n_keep(T, p, W)
    gc = MikvCache(B, Hq, Hkv, 128, 16, lo, keep + 1, T - keep + 1, dev(), key_mode=CH)
    d = {k: torch.from_numpy(np.ascontiguousarray(v)).to(dev()) for k, v in qT.items()}
    ginfo = gc.prefill(d["q"], d["k"], d["v"], p, W, keep_intermediates=True)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_np(ginfo["keep_pos"]), info["keep_pos"])
    compare_all(gc, oc)
    q_dec = xn["q"][:, :, -1]
    want, lse_o, _ = oc.attend(q_dec)
    _lib.mikv_decode_attention(torch.from_numpy(q_dec).to(dev()), gc, gc.out, gc.lse)
    torch.cuda.synchronize()
    err = np.abs(to_np(gc.out) - want).max()
    assert err <= ATTN_TOL, err
    assert err <= 1e-4, err
    np.testing.assert_allclose(to_np(gc.lse), lse_o, rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("lo,Hq,Hkv,T,steps", [(2, 8, 2, 300, 40), (4, 4, 4, 220, 30)])
def test_channel_decode_steps_match_oracle(lo, Hq, Hkv, T, steps):
    """Decode steps through mikv_decode_step: demoted pairs wait in FP16 and a group closes
    on the way; every buffer bit-exact and the output within the bar at every step."""
    B, p, W = 2, 20, 16
    wl = inputs.WORKLOADS["tiny"].scaled(B=B, Hq=Hq, Hkv=Hkv, T=T, lo_bits=lo, n_outlier=8)
    xn = _np(inputs.make_prefill(wl, 6, "cpu"))
    oc, info = cq.prefill_channel(xn["q"], xn["k"], xn["v"], lo_bits=lo, budget_pct=p, window=W,
                                  extra_steps=steps)
    keep = osel.n_keep(T, p, W)
    gc = MikvCache(B, Hq, Hkv, 128, 16, lo, keep + steps + 1, T - keep + steps + 1, dev(), key_mode=CH)
    d = {k: torch.from_numpy(v).to(dev()) for k, v in xn.items()}
    gc.prefill(d["q"], d["k"], d["v"], p, W)
    torch.cuda.synchronize()
    compare_all(gc, oc)
    closed = False
    worst = 0.0
    for s in range(steps):
        t = inputs.make_decode_token(wl, 6, s, "cpu")
        out_o, _, _ = cq.decode_step_channel(oc, t["q"].numpy(), t["k"].numpy(), t["v"].numpy(), T + s,
                                             budget_pct=p, window=W)
        n_lo = gc.n_lo
        out, _ = gc.decode_step(t["q"].to(dev()), t["k"].to(dev()), t["v"].to(dev()), T + s, p, W)
        torch.cuda.synchronize()
        closed |= gc.n_lo // 64 > n_lo // 64
        err = np.abs(to_np(out) - out_o).max()
        worst = max(worst, err)
        assert err <= ATTN_TOL, (s, err)
        compare_all(gc, oc)
        got = to_np(gc.scores[:, :, :gc.n_hi]).astype(np.float64)
        want = oc.scores[:, :, :oc.n_hi]
        assert np.abs(got - want).max() <= SCORE_RTOL * np.abs(want).max()
    assert closed
    assert worst <= 1e-4, worst


def test_channel_fused_step_equals_separate_calls():
    """The four-launch step and the five separate calls leave identical buffers, also when
    the demoted pair closes a group."""
    lo, B, Hq, Hkv, T, p, W, steps = 2, 2, 8, 2, 300, 20, 16, 40
    wl = inputs.WORKLOADS["tiny"].scaled(B=B, Hq=Hq, Hkv=Hkv, T=T, lo_bits=lo, n_outlier=8)
    d = {k: v.to(dev()) for k, v in inputs.make_prefill(wl, 7, "cpu").items()}
    keep = osel.n_keep(T, p, W)
    caches = []
    for _ in range(2):
        gc = MikvCache(B, Hq, Hkv, 128, 16, lo, keep + steps + 1, T - keep + steps + 1, dev(), key_mode=CH)
        gc.prefill(d["q"], d["k"], d["v"], p, W)
        caches.append(gc)
    fused, calls = caches
    closed = False
    for s in range(steps):
        t = {k: v.to(dev()) for k, v in inputs.make_decode_token(wl, 7, s, "cpu").items()}
        n_lo = fused.n_lo
        o1, l1 = fused.decode_step(t["q"], t["k"], t["v"], T + s, p, W)
        o1, l1 = o1.clone(), l1.clone()
        o2, l2 = calls.decode_step_calls(t["q"], t["k"], t["v"], T + s, p, W)
        torch.cuda.synchronize()
        closed |= fused.n_lo // 64 > n_lo // 64
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
        assert (fused.n_hi, fused.n_lo) == (calls.n_hi, calls.n_lo)
        nf = fused.n_lo - fused.n_lo % 64
        for nm, n in (("k_hi", fused.n_hi), ("v_hi", fused.n_hi), ("pos_hi", fused.n_hi), ("k_lo", nf),
                      ("v_lo", nf), ("v_lo_meta", nf), ("k_lo_meta", nf // 64), ("pos_lo", fused.n_lo),
                      ("k_pend", fused.n_lo % 64), ("v_pend", fused.n_lo % 64)):
            assert torch.equal(getattr(fused, nm)[:, :, :n], getattr(calls, nm)[:, :, :n]), nm
        assert torch.equal(fused.scores[:, :, :fused.n_hi], calls.scores[:, :, :calls.n_hi])
    assert closed


class ChannelUnitMirror:
    """Oracle per-channel cache of one (batch, key head) unit following the library's steps
    (the library's victims; the oracle's float64 scores must rank each one first unless the two
    lowest candidates are within the score bar of each other)."""

    def __init__(self, wl, gc, x, info, b, g, steps):
        self.wl, self.b, self.g = wl, b, g
        kp = to_np(info["keep_pos"][b, g]).astype(np.int32)
        ep = to_np(info["evict_pos"][b, g]).astype(np.int32)
        cap_lo = -(-(len(ep) + steps + 1) // 64) * 64
        self.oc = cq.ChannelKeyCache(1, 1, wl.Hq // wl.Hkv, 128, wl.lo_bits, len(kp) + steps + 1, cap_lo)
        src_k, src_v = to_np(x["k"][b, g])[None, None], to_np(x["v"][b, g])[None, None]
        ks = to_np(info["keep_scores"][b, g]).astype(np.float64)[None, None]
        self.oc.append("hi", src_k, src_v, kp[None, None], 0, ks)
        self.oc.append("lo", src_k, src_v, ep[None, None], 0)
        self.near_ties = 0

    def step(self, gc, tok, out, L_before, n_lo_before):
        wl, oc, b, g = self.wl, self.oc, self.b, self.g
        rep, L, W = wl.Hq // wl.Hkv, L_before + 1, wl.window
        oc.append("hi", to_np(tok["k"][b, g])[None, None, None], to_np(tok["v"][b, g])[None, None, None],
                  np.zeros((1, 1, 1), np.int32), L - 1)
        q = to_np(tok["q"][b, g * rep:(g + 1) * rep])[None]
        want, lse, logits = oc.attend(q)
        from oracle import scores as osc
        oc.scores[0, 0, :oc.n_hi] = osc.decode_score_update(oc.scores[0, 0, :oc.n_hi], logits[0], lse[0])
        err = np.abs(to_np(out[b, g * rep:(g + 1) * rep]) - want[0]).max()
        if gc.n_lo > n_lo_before:   # the library demoted: follow its victim
            vpos = int(to_np(gc.pos_lo[b, g, n_lo_before]))
            pos = oc.pos_hi[0, 0, :oc.n_hi]
            j_lib = int(np.nonzero(pos == vpos)[0][0])
            s = oc.scores[0, 0, :oc.n_hi]
            j_or = osel.demote_victim(s.astype(np.float32), pos, L, W)
            if j_lib != j_or:
                assert abs(s[j_lib] - s[j_or]) <= 2 * SCORE_RTOL * np.abs(s).max()
                self.near_ties += 1
            oc.demote(np.array([[j_lib]], np.int32))
        compare_unit(gc, oc, b, g, 0, 0)
        got = to_np(gc.scores[b, g, :gc.n_hi]).astype(np.float64)
        assert np.abs(got - oc.scores[0, 0, :oc.n_hi]).max() <= SCORE_RTOL * np.abs(oc.scores[0, 0, :oc.n_hi]).max()
        return err


@pytest.mark.parametrize("lo", [2, 4])
def test_channel_fullsize_lockstep(lo):
    """The full-depth workload's layer shape (B 4 here, T 8192, 20 % FP16, window 32) with
    per-channel keys: 26 waiting pairs after prefill, a group closes at the 38th demotion;
    sampled units follow an oracle cache step by step for 48 steps."""
    wl = inputs.WORKLOADS["llama31_8b_full"].scaled(B=4, layers=1, lo_bits=lo)
    d = dev()
    steps = 48
    x = inputs.make_prefill(wl, 0, d)
    T, W = wl.T, wl.window
    keep = osel.n_keep(T, wl.budget_pct, W)
    gc = MikvCache(wl.B, wl.Hq, wl.Hkv, 128, 16, lo, keep + steps + 1, T - keep + steps + 1, d, key_mode=CH)
    info = gc.prefill(x["q"], x["k"], x["v"], wl.budget_pct, W, keep_intermediates=True)
    torch.cuda.synchronize()
    assert gc.n_lo % 64 == 26
    mirrors = [ChannelUnitMirror(wl, gc, x, info, b, g, steps) for b, g in ((0, 3), (3, 6))]
    for m in mirrors:
        compare_unit(gc, m.oc, m.b, m.g, 0, 0)
    del x, info
    worst, closed = 0.0, False
    for s in range(steps):
        tok = inputs.make_decode_token(wl, 0, s, d)
        n_lo = gc.n_lo
        out, _ = gc.decode_step(tok["q"], tok["k"], tok["v"], T + s, wl.budget_pct, W)
        torch.cuda.synchronize()
        closed |= gc.n_lo // 64 > n_lo // 64
        for m in mirrors:
            err = m.step(gc, tok, out, T + s, n_lo)
            worst = max(worst, err)
            assert err <= ATTN_TOL, (s, err)
    assert closed
    assert worst <= 1e-4, worst
    assert sum(m.near_ties for m in mirrors) <= 1
