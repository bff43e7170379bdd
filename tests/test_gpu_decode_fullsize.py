"""Full-size decode: mikv_decode_step run for the workloads' stated step counts, at their
stated sizes, checked step by step against the oracle.

At these sizes the important tier holds more than one chunk of the fused step's score and
demotion kernel (1024 slots per CTA), so the per-chunk victim candidates, the ticket and the
last CTA's reduction, victim move and swap-remove all run as they do in the bench.

Two checks:

* ``test_decode_lockstep``: for sampled (batch, key head) units an oracle cache of that unit
  follows the library step by step.  Every step compares the attention output (2e-3 bar, and
  1e-4, the fp32 level it reaches), the H2O scores (normwise 1e-5 per unit) and the unit's
  whole state bit for bit: important tier (rows or codes and meta, positions) and low tier
  (codes, meta, positions).  The victim is the integer decision the library takes on its
  fp32 scores; the oracle's float64 scores must put it at the minimum of (score ascending,
  position descending) among tokens older than the window, exactly, unless the two lowest
  candidates are within the score bar of each other (a near-tie, counted and bounded).
* ``test_fused_step_equals_calls_fullsize``: the fused step and the five separate calls on
  two copies of the same cache stay bit-identical, and at every step the separate path's own
  fp32 scores, read back before its demotion, are given to the oracle's victim rule: the
  library's victim must equal the oracle's for every unit (identical score tensors), its new
  low-tier slot must be the oracle's quantisation of the victim's row, and the victim's
  important slot must hold the former last slot.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import ATTN_TOL, SCORE_RTOL, dev, to_np, u16
from mixed_precision_kv_balancer_gb300 import _lib, inputs
from mixed_precision_kv_balancer_gb300.cache import MikvCache
from oracle import pipeline as opipe
from oracle import quant as oquant
from oracle import scores as oscores
from oracle import select as osel

pytestmark = pytest.mark.gpu

CHUNK = 1024  # important-tier slots per CTA of the fused score + demotion kernel


def _sample_units(wl, n, seed):
    rng = np.random.default_rng(seed)
    units = {(int(rng.integers(wl.B)), int(rng.integers(wl.Hkv))) for _ in range(4 * n)}
    return sorted(units)[:n]


class UnitMirror:
    """Oracle cache of one (batch, key head) unit that follows the library's steps."""

    def __init__(self, wl, gc, x, info, b, g, steps):
        self.wl, self.b, self.g = wl, b, g
        kp = to_np(info["keep_pos"][b, g]).astype(np.int32)
        ep = to_np(info["evict_pos"][b, g]).astype(np.int32)
        bal = None if gc.balancer is None else to_np(gc.balancer[b:b + 1, g:g + 1])
        self.oc = opipe.OracleCache(1, 1, wl.rep, 128, 64, wl.hi_bits, wl.lo_bits,
                                    len(kp) + steps + 1, len(ep) + steps + 1, bal)
        src_k = to_np(x["k"][b, g])[None, None]
        src_v = to_np(x["v"][b, g])[None, None]
        ks = to_np(info["keep_scores"][b, g]).astype(np.float64)[None, None]
        self.oc.append("hi", src_k, src_v, kp[None, None], 0, ks)
        self.oc.append("lo", src_k, src_v, ep[None, None], 0)
        self.near_ties = 0

    def compare_state(self, gc):
        """Bit-exact comparison of the unit's occupied slots; scores within the score bar."""
        oc, b, g = self.oc, self.b, self.g
        assert (gc.n_hi, gc.n_lo) == (oc.n_hi, oc.n_lo)
        nh, nl = oc.n_hi, oc.n_lo
        if gc.hi_bits == 16:
            np.testing.assert_array_equal(u16(gc.k_hi[b, g, :nh]), oc.k_hi[0, 0, :nh])
            np.testing.assert_array_equal(u16(gc.v_hi[b, g, :nh]), oc.v_hi[0, 0, :nh])
        else:
            np.testing.assert_array_equal(to_np(gc.k_hi[b, g, :nh]), oc.k_hi[0, 0, :nh])
            np.testing.assert_array_equal(to_np(gc.v_hi[b, g, :nh]), oc.v_hi[0, 0, :nh])
            np.testing.assert_array_equal(u16(gc.k_hi_meta[b, g, :nh]), oc.k_hi_meta[0, 0, :nh])
            np.testing.assert_array_equal(u16(gc.v_hi_meta[b, g, :nh]), oc.v_hi_meta[0, 0, :nh])
        np.testing.assert_array_equal(to_np(gc.pos_hi[b, g, :nh]), oc.pos_hi[0, 0, :nh])
        np.testing.assert_array_equal(to_np(gc.k_lo[b, g, :nl]), oc.k_lo[0, 0, :nl])
        np.testing.assert_array_equal(to_np(gc.v_lo[b, g, :nl]), oc.v_lo[0, 0, :nl])
        np.testing.assert_array_equal(u16(gc.k_lo_meta[b, g, :nl]), oc.k_lo_meta[0, 0, :nl])
        np.testing.assert_array_equal(u16(gc.v_lo_meta[b, g, :nl]), oc.v_lo_meta[0, 0, :nl])
        np.testing.assert_array_equal(to_np(gc.pos_lo[b, g, :nl]), oc.pos_lo[0, 0, :nl])
        got = to_np(gc.scores[b, g, :nh]).astype(np.float64)
        want = oc.scores[0, 0, :nh]
        assert np.abs(got - want).max() <= SCORE_RTOL * np.abs(want).max()

    def attend(self, tok, L_before):
        """The oracle's half of one step: append the new token, attend, add the scores.
        Returns (out [rep, D], demotion expected)."""
        oc, b, g, wl = self.oc, self.b, self.g, self.wl
        L = L_before + 1
        k_new = to_np(tok["k"][b, g])[None, None, None]
        v_new = to_np(tok["v"][b, g])[None, None, None]
        oc.append("hi", k_new, v_new, np.zeros((1, 1, 1), np.int32), pos_base=L - 1)
        q = to_np(tok["q"][b, g * wl.rep:(g + 1) * wl.rep])[None]
        out, lse, logits = oc.attend(q)
        oc.scores[0, 0, :oc.n_hi] = oscores.decode_score_update(oc.scores[0, 0, :oc.n_hi],
                                                                 logits[0], lse[0])
        demote = wl.policy == "h2o" and oc.n_hi > osel.n_keep(L, wl.budget_pct, wl.window)
        return out[0], demote

    def follow_demotion(self, gc, L):
        """Find the library's victim (the position its new low-tier slot holds), check it
        against the oracle's scores and apply it to the oracle cache."""
        oc, b, g, W = self.oc, self.b, self.g, self.wl.window
        nh = oc.n_hi
        vpos = int(to_np(gc.pos_lo[b, g, oc.n_lo]))
        pos = oc.pos_hi[0, 0, :nh]
        hit = np.nonzero(pos == vpos)[0]
        assert len(hit) == 1, (vpos, hit)
        j_lib = int(hit[0])
        assert vpos < L - W
        s = oc.scores[0, 0, :nh]
        j_or = osel.demote_victim(s.astype(np.float32), pos, L, W)
        if j_lib != j_or:
            # only a near-tie may decide differently in fp32 than in float64
            assert abs(s[j_lib] - s[j_or]) <= 2 * SCORE_RTOL * np.abs(s).max(), \
                (j_lib, j_or, s[j_lib], s[j_or])
            self.near_ties += 1
        oc.demote(np.array([[j_lib]], np.int32))


# (workload, changes, steps, units): the five workloads at their stated sizes and step
# counts (the full-depth one layer at a time), and the full-depth shape's sweep of the
# low-tier width and the budget.
LOCKSTEP = [
    ("tiny", {}, 32, 4),
    ("llama2_7b", {}, 128, 2),
    ("llama31_8b", {}, 64, 2),
    ("qwen25_32b", {}, 32, 2),
    ("llama31_8b_full", dict(layers=1), 16, 3),
    ("llama31_8b_full", dict(layers=1, lo_bits=4), 8, 2),
    ("llama31_8b_full", dict(layers=1, budget_pct=10), 8, 2),
    ("llama31_8b_full", dict(layers=1, budget_pct=40), 8, 2),
    ("llama31_8b_full", dict(layers=1, lo_bits=4, budget_pct=10), 8, 2),
    ("llama31_8b_full", dict(layers=1, lo_bits=4, budget_pct=40), 8, 2),
    ("llama31_8b_full", dict(layers=1, B=1, T=32768), 6, 3),   # important tier of 7 chunks
]


@pytest.mark.parametrize("name,changes,steps,nunits", LOCKSTEP,
                         ids=[f"{n}-{'-'.join(f'{k}{v}' for k, v in c.items()) or 'stated'}-{s}steps"
                              for n, c, s, _ in LOCKSTEP])
def test_decode_lockstep(name, changes, steps, nunits):
    wl = inputs.WORKLOADS[name].scaled(**changes)
    d = dev()
    x = inputs.make_prefill(wl, 0, d)
    T, W = wl.T, wl.window
    keep = osel.n_keep(T, wl.budget_pct, W)
    w_o = inputs.make_w_o(wl, 0, d) if wl.policy == "criticalkv" else None
    gc = MikvCache(wl.B, wl.Hq, wl.Hkv, 128, wl.hi_bits, wl.lo_bits, keep + steps + 1,
                   T - keep + steps + 1, d)
    info = gc.prefill(x["q"], x["k"], x["v"], wl.budget_pct, W, policy=wl.policy, alpha=wl.alpha,
                      w_o=w_o, keep_intermediates=True)
    torch.cuda.synchronize()
    units = _sample_units(wl, nunits, 5)
    mirrors = [UnitMirror(wl, gc, x, info, b, g, steps) for b, g in units]
    for m in mirrors:
        m.compare_state(gc)
    del x, info
    max_chunks = 0
    demotions = 0
    worst = 0.0
    for s in range(steps):
        tok = inputs.make_decode_token(wl, 0, s, d)
        want = [m.attend(tok, T + s) for m in mirrors]
        n_lo_before = gc.n_lo
        max_chunks = max(max_chunks, (gc.n_hi + 1 + CHUNK - 1) // CHUNK)
        out, _ = gc.decode_step(tok["q"], tok["k"], tok["v"], T + s, wl.budget_pct, W,
                                policy=wl.policy)
        torch.cuda.synchronize()
        for m, (o_want, demote) in zip(mirrors, want):
            b, g = m.b, m.g
            err = np.abs(to_np(out[b, g * wl.rep:(g + 1) * wl.rep]) - o_want).max()
            worst = max(worst, err)
            assert err <= ATTN_TOL, (s, b, g, err)
            assert (gc.n_lo == n_lo_before + 1) == demote
            if demote:
                m.follow_demotion(gc, T + s + 1)
            m.compare_state(gc)
        demotions += int(gc.n_lo > n_lo_before)
    assert worst <= 1e-4, worst
    if wl.policy == "h2o" and wl.budget_pct > 0:
        assert demotions > 0
    assert sum(m.near_ties for m in mirrors) <= 1
    if name != "tiny" and changes.get("budget_pct", wl.budget_pct) >= 20:
        assert max_chunks >= 2, max_chunks   # the multi-chunk reduction ran


def _snapshot(gc, nh):
    """Host copies of the important tier (rows, positions) before a demotion."""
    return dict(k=u16(gc.k_hi[:, :, :nh]).copy(), v=u16(gc.v_hi[:, :, :nh]).copy(),
                pos=to_np(gc.pos_hi[:, :, :nh]).copy())


@pytest.mark.parametrize("changes,steps", [(dict(B=4), 6), (dict(B=1, T=32768), 4),
                                           (dict(B=2, lo_bits=4, budget_pct=40), 4)])
def test_fused_step_equals_calls_fullsize(changes, steps):
    wl = inputs.WORKLOADS["llama31_8b_full"].scaled(layers=1, **changes)
    d = dev()
    x = inputs.make_prefill(wl, 0, d)
    T, W = wl.T, wl.window
    keep = osel.n_keep(T, wl.budget_pct, W)
    caches = []
    for _ in range(2):
        gc = MikvCache(wl.B, wl.Hq, wl.Hkv, 128, wl.hi_bits, wl.lo_bits, keep + steps + 1,
                       T - keep + steps + 1, d)
        gc.prefill(x["q"], x["k"], x["v"], wl.budget_pct, W)
        caches.append(gc)
    fused, calls = caches
    assert fused.n_hi > CHUNK
    bal = to_np(calls.balancer)
    demoted = 0
    for s in range(steps):
        L = T + s + 1
        t = inputs.make_decode_token(wl, 0, s, d)
        o1, l1 = fused.decode_step(t["q"], t["k"], t["v"], T + s, wl.budget_pct, W)
        o1, l1 = o1.clone(), l1.clone()
        # the five calls, stopping before the demotion to read the fp32 scores it ranks
        _lib.mikv_quantize_append(_lib.MIKV_TIER_HI, calls, t["k"][:, :, None, :],
                                  t["v"][:, :, None, :], calls.zero_pos, 1, L - 1)
        _lib.mikv_decode_attention(t["q"], calls, calls.out, calls.lse, calls.hi_logits,
                                   ws=calls.ws_decode)
        _lib.mikv_score_update(_lib.MIKV_DECODE, calls, hi_logits=calls.hi_logits, lse=calls.lse)
        torch.cuda.synchronize()
        nh, nl = calls.n_hi, calls.n_lo
        over = nh > osel.n_keep(L, wl.budget_pct, W)
        demoted += int(over)
        if over:
            S = to_np(calls.scores[:, :, :nh]).copy()
            snap = _snapshot(calls, nh)
            sc_last = S[:, :, nh - 1].copy()
            _lib.mikv_select(_lib.MIKV_DEMOTE, calls, L, wl.budget_pct, W, evict_pos=calls.victim)
            _lib.mikv_quantize_append(_lib.MIKV_TIER_DEMOTE, calls, None, None, calls.victim, 1)
            torch.cuda.synchronize()
            victim = to_np(calls.victim)
            for b in range(wl.B):
                for g in range(wl.Hkv):
                    j = osel.demote_victim(S[b, g], snap["pos"][b, g], L, W)
                    assert victim[b, g] == j, (s, b, g, victim[b, g], j)
            # the new low-tier slot: the oracle's quantisation of the victim's FP16 row
            vk = np.take_along_axis(snap["k"], victim[:, :, None, None].astype(np.int64), axis=2)[:, :, 0]
            vv = np.take_along_axis(snap["v"], victim[:, :, None, None].astype(np.int64), axis=2)[:, :, 0]
            xk = oquant.balance_keys(vk.view(np.float16), bal)
            kc, km = oquant.quantize_groups(xk, wl.lo_bits, 64)
            vc, vm = oquant.quantize_groups(vv.view(np.float16).astype(np.float32), wl.lo_bits, 64)
            np.testing.assert_array_equal(to_np(calls.k_lo[:, :, nl]), oquant.pack_codes(kc, wl.lo_bits))
            np.testing.assert_array_equal(to_np(calls.v_lo[:, :, nl]), oquant.pack_codes(vc, wl.lo_bits))
            np.testing.assert_array_equal(u16(calls.k_lo_meta[:, :, nl]), km)
            np.testing.assert_array_equal(u16(calls.v_lo_meta[:, :, nl]), vm)
            vpos = np.take_along_axis(snap["pos"], victim[:, :, None].astype(np.int64), axis=2)[:, :, 0]
            np.testing.assert_array_equal(to_np(calls.pos_lo[:, :, nl]), vpos)
            # the victim's important slot now holds the former last slot (swap-remove)
            for b in range(wl.B):
                for g in range(wl.Hkv):
                    j = int(victim[b, g])
                    if j != nh - 1:
                        np.testing.assert_array_equal(u16(calls.k_hi[b, g, j]), snap["k"][b, g, nh - 1])
                        np.testing.assert_array_equal(u16(calls.v_hi[b, g, j]), snap["v"][b, g, nh - 1])
                        assert int(to_np(calls.pos_hi[b, g, j])) == snap["pos"][b, g, nh - 1]
                        assert to_np(calls.scores[b, g, j]) == sc_last[b, g]
        # the fused step left every buffer bit-identical
        assert torch.equal(o1, calls.out) and torch.equal(l1, calls.lse)
        assert (fused.n_hi, fused.n_lo) == (calls.n_hi, calls.n_lo)
        for nm in ("k_hi", "v_hi", "k_lo", "v_lo", "k_lo_meta", "v_lo_meta", "pos_hi", "pos_lo"):
            n = fused.n_hi if "hi" in nm else fused.n_lo
            assert torch.equal(getattr(fused, nm)[:, :, :n], getattr(calls, nm)[:, :, :n]), nm
        assert torch.equal(fused.scores[:, :, :fused.n_hi], calls.scores[:, :, :calls.n_hi])
    assert demoted >= 2
