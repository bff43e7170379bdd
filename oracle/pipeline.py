"""The whole hot path composed on one two-tier cache (oracle).

Sources: MiKV reading notes (velog), "Key contributions" 1)-3) and section 3.4;
paperlayer summary of arXiv 2402.18096v1, sections 3.1-3.4; CriticalKV summary
(gist.science), "Algorithm".  The MiKV framework keeps the tokens an eviction
policy would drop, in low precision, next to the important tokens kept in high
precision (FP16, or INT8 per section 3.3).

Per layer:
  prefill  balancer -> H2O scores -> selection (H2O or CriticalKV) ->
           important tokens appended to the high tier, the rest quantised to
           the low tier, both in ascending position order;
  decode   new token appended to the high tier (score 0) -> attention over both
           tiers -> score update -> if the high tier is over budget (H2O only),
           the victim is re-quantised into the low tier and the last high slot
           moves into its place.

Readings where the pages are silent (step order, slot order, demotion):
* per decode step: append, attend, update, demote (H2O evicts after the
  step's attention); at most one demotion per step because the budget grows
  by at most one token per step;
* a demoted token is re-quantised from what the high tier holds: the original
  fp16 key/value (balanced key fl(k*b)), or for an INT8 tier its float32
  dequantisation, which is already balanced;
* CriticalKV selects once at the end of prefill (it plugs into pipelines that
  do so); during decode its new tokens join the high tier, with no demotion.
"""
from __future__ import annotations

import numpy as np

from . import attention, balance, quant, scores, select


class OracleCache:
    """Slot-ordered two-tier cache of one layer, same contents as the library's buffers."""

    def __init__(self, B, Hkv, Hq, D, gs, hi_bits, lo_bits, cap_hi, cap_lo, balancer):
        self.B, self.Hkv, self.Hq, self.D, self.gs = B, Hkv, Hq, D, gs
        self.rep = Hq // Hkv
        self.hi_bits, self.lo_bits = hi_bits, lo_bits
        self.cap_hi, self.cap_lo = cap_hi, cap_lo
        self.n_hi = self.n_lo = 0
        self.balancer = balancer                     # [B,Hkv,D] float32 or None
        ng = D // gs
        if hi_bits == 16:
            self.k_hi = np.zeros((B, Hkv, cap_hi, D), np.uint16)
            self.v_hi = np.zeros((B, Hkv, cap_hi, D), np.uint16)
        else:
            self.k_hi = np.zeros((B, Hkv, cap_hi, D * hi_bits // 8), np.uint8)
            self.v_hi = np.zeros((B, Hkv, cap_hi, D * hi_bits // 8), np.uint8)
        self.k_hi_meta = np.zeros((B, Hkv, cap_hi, ng, 2), np.uint16)
        self.v_hi_meta = np.zeros((B, Hkv, cap_hi, ng, 2), np.uint16)
        self.k_lo = np.zeros((B, Hkv, cap_lo, D * lo_bits // 8), np.uint8)
        self.v_lo = np.zeros((B, Hkv, cap_lo, D * lo_bits // 8), np.uint8)
        self.k_lo_meta = np.zeros((B, Hkv, cap_lo, ng, 2), np.uint16)
        self.v_lo_meta = np.zeros((B, Hkv, cap_lo, ng, 2), np.uint16)
        self.pos_hi = np.zeros((B, Hkv, cap_hi), np.int32)
        self.pos_lo = np.zeros((B, Hkv, cap_lo), np.int32)
        self.scores = np.zeros((B, Hkv, cap_hi), np.float64)

    # -- quantisation of one token row ------------------------------------------------
    def _bal(self, b, g):
        return None if self.balancer is None else self.balancer[b, g]

    def _encode(self, xk: np.ndarray, xv: np.ndarray, bits: int):
        """float32 (balanced key, value) rows -> packed (k, k_meta, v, v_meta)."""
        kc, km = quant.quantize_groups(xk, bits, self.gs)
        vc, vm = quant.quantize_groups(xv, bits, self.gs)
        return quant.pack_codes(kc, bits), km, quant.pack_codes(vc, bits), vm

    # -- append ------------------------------------------------------------------------
    def append(self, tier: str, k, v, src_pos, pos_base=0, src_scores=None):
        """k, v [B,Hkv,S,D] fp16 sources; src_pos [B,Hkv,n] int -> slots n_tier..n_tier+n-1."""
        n = src_pos.shape[2]
        if tier == "hi":
            base = self.n_hi
            assert base + n <= self.cap_hi
        else:
            base = self.n_lo
            assert base + n <= self.cap_lo
        for b in range(self.B):
            for g in range(self.Hkv):
                idx = src_pos[b, g].astype(np.int64)
                kr, vr = k[b, g, idx], v[b, g, idx]
                sl = slice(base, base + n)
                if tier == "hi":
                    if self.hi_bits == 16:
                        self.k_hi[b, g, sl] = kr.view(np.uint16)
                        self.v_hi[b, g, sl] = vr.view(np.uint16)
                    else:
                        xk = quant.balance_keys(kr, self._bal(b, g))
                        pk, km, pv, vm = self._encode(xk, vr.astype(np.float32), self.hi_bits)
                        self.k_hi[b, g, sl], self.k_hi_meta[b, g, sl] = pk, km
                        self.v_hi[b, g, sl], self.v_hi_meta[b, g, sl] = pv, vm
                    self.pos_hi[b, g, sl] = idx + pos_base
                    self.scores[b, g, sl] = 0.0 if src_scores is None else src_scores[b, g]
                else:
                    xk = quant.balance_keys(kr, self._bal(b, g))
                    pk, km, pv, vm = self._encode(xk, vr.astype(np.float32), self.lo_bits)
                    self.k_lo[b, g, sl], self.k_lo_meta[b, g, sl] = pk, km
                    self.v_lo[b, g, sl], self.v_lo_meta[b, g, sl] = pv, vm
                    self.pos_lo[b, g, sl] = idx + pos_base
        if tier == "hi":
            self.n_hi += n
        else:
            self.n_lo += n

    # -- demotion ----------------------------------------------------------------------
    def demote(self, victims: np.ndarray):
        """victims [B,Hkv] high-tier slots: re-quantise into the low tier, swap-remove."""
        assert self.n_lo + 1 <= self.cap_lo and self.n_hi >= 1
        last = self.n_hi - 1
        D = self.D
        for b in range(self.B):
            for g in range(self.Hkv):
                j = int(victims[b, g])
                if self.hi_bits == 16:
                    kr = self.k_hi[b, g, j].view(np.float16)
                    xk = quant.balance_keys(kr, self._bal(b, g))
                    xv = self.v_hi[b, g, j].view(np.float16).astype(np.float32)
                else:
                    kc = quant.unpack_codes(self.k_hi[b, g, j], self.hi_bits, D)
                    vc = quant.unpack_codes(self.v_hi[b, g, j], self.hi_bits, D)
                    xk = quant.dequantize_f32(kc, self.k_hi_meta[b, g, j], self.gs)
                    xv = quant.dequantize_f32(vc, self.v_hi_meta[b, g, j], self.gs)
                pk, km, pv, vm = self._encode(xk, xv, self.lo_bits)
                s = self.n_lo
                self.k_lo[b, g, s], self.k_lo_meta[b, g, s] = pk, km
                self.v_lo[b, g, s], self.v_lo_meta[b, g, s] = pv, vm
                self.pos_lo[b, g, s] = self.pos_hi[b, g, j]
                for arr in (self.k_hi, self.v_hi, self.k_hi_meta, self.v_hi_meta, self.pos_hi,
                            self.scores):
                    arr[b, g, j] = arr[b, g, last]
        self.n_hi -= 1
        self.n_lo += 1

    # -- views ---------------------------------------------------------------------------
    def unit(self, b: int, g: int):
        hi = dict(n=self.n_hi, k=self.k_hi[b, g, :self.n_hi], v=self.v_hi[b, g, :self.n_hi],
                  k_meta=self.k_hi_meta[b, g, :self.n_hi], v_meta=self.v_hi_meta[b, g, :self.n_hi])
        lo = dict(n=self.n_lo, k=self.k_lo[b, g, :self.n_lo], v=self.v_lo[b, g, :self.n_lo],
                  k_meta=self.k_lo_meta[b, g, :self.n_lo], v_meta=self.v_lo_meta[b, g, :self.n_lo])
        return hi, lo

    def attend(self, q: np.ndarray):
        """q [B,Hq,D] fp16 -> out [B,Hq,D], lse [B,Hq], hi_logits [B,Hq,n_hi] (float64)."""
        B, Hq, D = q.shape
        rep = self.rep
        out = np.zeros((B, Hq, D))
        lse = np.zeros((B, Hq))
        logits = np.zeros((B, Hq, self.n_hi))
        for b in range(B):
            for g in range(self.Hkv):
                hi, lo = self.unit(b, g)
                hs = slice(g * rep, (g + 1) * rep)
                o, l, lh = attention.decode_attention_unit(
                    q[b, hs], hi, lo, self._bal(b, g), self.hi_bits, self.lo_bits, self.gs)
                out[b, hs], lse[b, hs], logits[b, hs] = o, l, lh
        return out, lse, logits


def prefill(q, k, v, *, hi_bits, lo_bits, budget_pct, window, gs=None, policy="h2o",
            alpha=0.5, w_o=None, use_balancer=True, extra_steps=0):
    """Build one layer's cache from prompt activations q [B,Hq,T,D], k/v [B,Hkv,T,D] (fp16).

    Returns (cache, info) with the intermediate results the tests compare:
    balancer, S_head, S, N (CriticalKV), keep/evict positions.
    """
    B, Hq, T, D = q.shape
    Hkv = k.shape[1]
    rep = Hq // Hkv
    gs = gs or D // 2
    b = balance.channel_balancer(q, k) if use_balancer else None
    s_head, s_grp = scores.prefill_scores(q, k)
    s_grp32 = s_grp.astype(np.float32)
    s_head32 = s_head.astype(np.float32)
    keep = select.n_keep(T, budget_pct, window)
    n_vwo = None
    if policy == "criticalkv":
        n_vwo = select.vwo_norms(v, w_o, rep)
        n_vwo32 = n_vwo.astype(np.float32)
    keep_pos = np.zeros((B, Hkv, keep), np.int32)
    evict_pos = np.zeros((B, Hkv, T - keep), np.int32)
    for bi in range(B):
        for g in range(Hkv):
            if policy == "h2o":
                kp, ep = select.h2o_select(s_grp32[bi, g], T, keep, window)
            else:
                hs = slice(g * rep, (g + 1) * rep)
                kp, ep = select.criticalkv_select(s_grp32[bi, g], s_head32[bi, hs], n_vwo32[bi, hs],
                                                  T, keep, window, alpha)
            keep_pos[bi, g], evict_pos[bi, g] = kp, ep
    cap_hi = keep + extra_steps + 1
    cap_lo = (T - keep) + extra_steps + 1
    cache = OracleCache(B, Hkv, Hq, D, gs, hi_bits, lo_bits, cap_hi, cap_lo, b)
    kept_scores = np.take_along_axis(s_grp, keep_pos.astype(np.int64), axis=2)
    cache.append("hi", k, v, keep_pos, 0, kept_scores)
    cache.append("lo", k, v, evict_pos, 0)
    info = dict(balancer=b, S_head=s_head, S=s_grp, N=n_vwo, keep_pos=keep_pos, evict_pos=evict_pos)
    return cache, info


def decode_step(cache: OracleCache, q_new, k_new, v_new, L_before: int, *, budget_pct, window,
                policy="h2o"):
    """One decode step on one layer; q_new [B,Hq,D], k_new/v_new [B,Hkv,D] fp16.

    Returns (out, lse, victims or None).
    """
    L = L_before + 1
    B, Hkv = cache.B, cache.Hkv
    src = np.zeros((B, Hkv, 1), np.int32)
    cache.append("hi", k_new[:, :, None, :], v_new[:, :, None, :], src, pos_base=L - 1)
    out, lse, logits = cache.attend(q_new)
    rep = cache.rep
    for b in range(B):
        for g in range(Hkv):
            hs = slice(g * rep, (g + 1) * rep)
            cache.scores[b, g, :cache.n_hi] = scores.decode_score_update(
                cache.scores[b, g, :cache.n_hi], logits[b, hs], lse[b, hs])
    victims = None
    if policy == "h2o" and cache.n_hi > select.n_keep(L, budget_pct, window):
        victims = np.zeros((B, Hkv), np.int32)
        for b in range(B):
            for g in range(Hkv):
                victims[b, g] = select.demote_victim(
                    cache.scores[b, g, :cache.n_hi].astype(np.float32),
                    cache.pos_hi[b, g, :cache.n_hi], L, window)
        cache.demote(victims)
    return out, lse, victims
