"""Full-size parity: each workload at its stated sizes, through the same calls and launch
configuration the bench uses, checked on what the oracle can compute one by one.

- balancer: bit-exact for every (batch, key head);
- H2O prefill scores: sampled columns of sampled query heads within the score bar, and
  mass conservation (every causal row sums to one, so sum_i S_i = rep * T) everywhere;
- selection: valid (window kept, sizes, no evicted older token outranks a kept one);
- codes and meta: bit-exact against the oracle's quantisation of the token each slot holds;
- V.W_O norms (CriticalKV workload): sampled tokens;
- attention of the first decode step for sampled (batch, key head) units, against the
  oracle's attention over a cache the oracle builds itself from the inputs (the important
  set is the library's selection, whose validity is checked above).
Inputs are drawn on the device (large) and the sampled slices copied to the host.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import ATTN_TOL, SCORE_RTOL, dev, to_np, u16
from mixed_precision_kv_balancer_gb300 import inputs
from mixed_precision_kv_balancer_gb300.cache import MikvCache
from oracle import balance as obal
from oracle import pipeline as opipe
from oracle import quant as oquant
from oracle import scores as oscores
from oracle import select as osel

pytestmark = pytest.mark.gpu

WORKLOADS = ["llama2_7b", "llama31_8b", "qwen25_32b", "llama31_8b_full"]


def _units(wl, n, seed):
    rng = np.random.default_rng(seed)
    return [(int(rng.integers(wl.B)), int(rng.integers(wl.Hkv))) for _ in range(n)]


@pytest.mark.parametrize("name", WORKLOADS)
def test_fullsize_workload(name):
    wl = inputs.WORKLOADS[name]
    d = dev()
    torch.manual_seed(0)
    x = inputs.make_prefill(wl, 0, d)
    T, rep, W = wl.T, wl.rep, wl.window
    keep = osel.n_keep(T, wl.budget_pct, W)
    w_o = inputs.make_w_o(wl, 0, d) if wl.policy == "criticalkv" else None
    gc = MikvCache(wl.B, wl.Hq, wl.Hkv, 128, wl.hi_bits, wl.lo_bits, keep + 2, T - keep + 2, d)
    info = gc.prefill(x["q"], x["k"], x["v"], wl.budget_pct, W, policy=wl.policy, alpha=wl.alpha,
                      w_o=w_o, keep_intermediates=True)
    tok = inputs.make_decode_token(wl, 0, 0, d)
    out, _ = gc.decode_step(tok["q"], tok["k"], tok["v"], T, wl.budget_pct, W, policy=wl.policy)
    torch.cuda.synchronize()

    # balancer: every unit, bit-exact (computed per batch row to bound host memory)
    for b in range(wl.B):
        want = obal.channel_balancer(to_np(x["q"][b:b + 1]), to_np(x["k"][b:b + 1]))
        np.testing.assert_array_equal(to_np(gc.balancer[b:b + 1]).view(np.uint32), want.view(np.uint32))

    # scores: mass conservation everywhere; sampled columns of sampled heads
    S = to_np(info["S"]).astype(np.float64)
    np.testing.assert_allclose(S.sum(axis=2), rep * T, rtol=1e-5)
    S_head = to_np(info["S_head"])
    units = _units(wl, 2, 1)
    cols = sorted(set(range(T - 48, T)) | {T - 300, T - 257, T - 129})  # oracle cost ~ rows below
    for b, g in units:
        for h in (g * rep, g * rep + rep - 1):
            want = oscores.column_scores_at(to_np(x["q"][b, h]), to_np(x["k"][b, g]), cols)
            got = S_head[b, h, cols].astype(np.float64)
            # the normwise bar, relative to the head's largest score
            assert np.abs(got - want).max() <= SCORE_RTOL * S_head[b, h].max()

    # selection validity (every unit)
    kp, ep = to_np(info["keep_pos"]), to_np(info["evict_pos"])
    assert kp.shape[2] == keep and ep.shape[2] == T - keep
    for b in range(wl.B):
        for g in range(wl.Hkv):
            k_, e_ = kp[b, g], ep[b, g]
            assert (np.diff(k_) > 0).all() and (np.diff(e_) > 0).all()
            assert np.array_equal(np.sort(np.concatenate([k_, e_])), np.arange(T))
            assert set(range(T - W, T)) <= set(k_.tolist())
            if wl.policy == "h2o":
                older_k = k_[k_ < T - W]
                s = S[b, g].astype(np.float32)
                if len(older_k) and len(e_):
                    # ranking key (score desc, position asc): the weakest kept older token
                    # outranks the strongest evicted one
                    weakest = min(older_k, key=lambda i: (s[i], -i))
                    strongest = max(e_, key=lambda i: (s[i], -i))
                    assert (s[weakest], -weakest) > (s[strongest], -strongest)

    # codes: each sampled slot holds the oracle's quantisation of its token
    bal = to_np(gc.balancer)
    for b, g in units:
        kv_k, kv_v = to_np(x["k"][b, g]), to_np(x["v"][b, g])
        slots = np.random.default_rng(2).choice(gc.n_lo, 64, replace=False)
        pos = to_np(gc.pos_lo[b, g])[slots]
        kc, km = oquant.quantize_groups(oquant.balance_keys(kv_k[pos], bal[b, g]), wl.lo_bits, 64)
        vc, vm = oquant.quantize_groups(kv_v[pos].astype(np.float32), wl.lo_bits, 64)
        np.testing.assert_array_equal(to_np(gc.k_lo[b, g])[slots], oquant.pack_codes(kc, wl.lo_bits))
        np.testing.assert_array_equal(to_np(gc.v_lo[b, g])[slots], oquant.pack_codes(vc, wl.lo_bits))
        np.testing.assert_array_equal(u16(gc.k_lo_meta[b, g])[slots], km)
        np.testing.assert_array_equal(u16(gc.v_lo_meta[b, g])[slots], vm)

    # V.W_O norms (CriticalKV)
    if wl.policy == "criticalkv":
        N = to_np(info["N"])
        rows = np.random.default_rng(3).choice(T, 40, replace=False)
        for b, g in units:
            h = g * rep
            want = osel.vwo_l1(to_np(x["v"][b, g])[rows], to_np(w_o)[h * 128:(h + 1) * 128])
            np.testing.assert_allclose(N[b, h, rows], want, rtol=SCORE_RTOL)

    # first decode step's attention for sampled units: a step attends before it demotes, so the
    # reference cache is the prefill selection plus the new token
    for b, g in units:
        src_k = np.concatenate([to_np(x["k"][b, g]), to_np(tok["k"][b, g])[None]], axis=0)[None, None]
        src_v = np.concatenate([to_np(x["v"][b, g]), to_np(tok["v"][b, g])[None]], axis=0)[None, None]
        oc = opipe.OracleCache(1, 1, rep, 128, 64, wl.hi_bits, wl.lo_bits, keep + 1, T - keep,
                               bal[b:b + 1, g:g + 1])
        hi_pos = np.concatenate([kp[b, g], [T]]).astype(np.int32)[None, None]
        oc.append("hi", src_k, src_v, hi_pos, 0)
        oc.append("lo", src_k, src_v, ep[b, g].astype(np.int32)[None, None], 0)
        qd = to_np(tok["q"][b, g * rep:(g + 1) * rep])[None]
        want, _, _ = oc.attend(qd)
        err = np.abs(to_np(out[b, g * rep:(g + 1) * rep]) - want[0]).max()
        assert err <= ATTN_TOL, err
        assert err <= 1e-4, err
