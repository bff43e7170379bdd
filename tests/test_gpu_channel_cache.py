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
