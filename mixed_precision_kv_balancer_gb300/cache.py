"""Device-resident two-tier cache of one layer and the per-layer step sequencing.

The buffers are torch tensors (device memory comes from torch's allocator); every
operation on them is one of the library's C ABI calls.  This module only decides
which call comes next, with which counts:

  prefill  mikv_balance_prefill -> mikv_score_update(PREFILL) -> mikv_select(H2O |
           CRITICALKV) -> mikv_quantize_append(HI, kept) -> mikv_quantize_append(LO, evicted)
  decode   mikv_quantize_append(HI, new token) -> mikv_decode_attention ->
           mikv_score_update(DECODE) -> [H2O, over budget] mikv_select(DEMOTE) ->
           mikv_quantize_append(DEMOTE); mikv_decode_step runs the same step in four
           launches (append, split-K attention, merge, score update + demotion)

(MiKV reading notes, "Key contributions 1)-3)" and section 3.4; CriticalKV
summary, "Algorithm".)  The budget is n_keep(L) = min(L, max(W, floor(p*L/100)))
and at most one token is demoted per step, after the step's attention.
"""
from __future__ import annotations

import torch

from . import _lib


def n_keep(L: int, budget_pct: int, window: int) -> int:
    return min(L, max(window, (budget_pct * L) // 100))


class MikvCache:
    """One layer's cache: tiers, metadata, positions, scores, balancer, plus reusable workspaces."""

    def __init__(self, B, Hq, Hkv, D, hi_bits, lo_bits, cap_hi, cap_lo, device="cuda",
                 use_balancer=True, key_mode=_lib.MIKV_KEYS_PER_TOKEN):
        """key_mode MIKV_KEYS_PER_CHANNEL: the low tier keeps per-channel keys in closed groups of
        64 slots and the last n_lo % 64 retained pairs in FP16 (cap_lo is rounded up to a
        multiple of 64; no balancer)."""
        assert D == 128 and Hq % Hkv == 0
        self.B, self.Hq, self.Hkv, self.D = B, Hq, Hkv, D
        self.hi_bits, self.lo_bits = hi_bits, lo_bits
        self.key_mode = key_mode
        per_channel = key_mode == _lib.MIKV_KEYS_PER_CHANNEL
        if per_channel:
            cap_lo = -(-cap_lo // 64) * 64
            use_balancer = False
        self.device = torch.device(device)
        dev = self.device
        ng = D // 64
        if hi_bits == 16:
            self.k_hi = torch.zeros(B, Hkv, cap_hi, D, dtype=torch.float16, device=dev)
            self.v_hi = torch.zeros_like(self.k_hi)
            self.k_hi_meta = self.v_hi_meta = None
        else:
            self.k_hi = torch.zeros(B, Hkv, cap_hi, D * hi_bits // 8, dtype=torch.uint8, device=dev)
            self.v_hi = torch.zeros_like(self.k_hi)
            self.k_hi_meta = torch.zeros(B, Hkv, cap_hi, ng, 2, dtype=torch.float16, device=dev)
            self.v_hi_meta = torch.zeros_like(self.k_hi_meta)
        rb = D * lo_bits // 8
        self.k_lo = torch.zeros(B, Hkv, cap_lo, rb, dtype=torch.uint8, device=dev)
        self.v_lo = torch.zeros_like(self.k_lo)
        self.v_lo_meta = torch.zeros(B, Hkv, cap_lo, ng, 2, dtype=torch.float16, device=dev)
        if per_channel:
            self.k_lo_meta = torch.zeros(B, Hkv, cap_lo // 64, D, 2, dtype=torch.float16, device=dev)
            self.k_pend = torch.zeros(B, Hkv, 64, D, dtype=torch.float16, device=dev)
            self.v_pend = torch.zeros_like(self.k_pend)
        else:
            self.k_lo_meta = torch.zeros_like(self.v_lo_meta)
            self.k_pend = self.v_pend = None
        self.pos_hi = torch.zeros(B, Hkv, cap_hi, dtype=torch.int32, device=dev)
        self.pos_lo = torch.zeros(B, Hkv, cap_lo, dtype=torch.int32, device=dev)
        self.scores = torch.zeros(B, Hkv, cap_hi, dtype=torch.float32, device=dev)
        self.balancer = torch.ones(B, Hkv, D, dtype=torch.float32, device=dev) if use_balancer else None
        s = _lib.mikv_cache()
        s.B, s.Hkv, s.Hq, s.D = B, Hkv, Hq, D
        s.hi_bits, s.lo_bits, s.cap_hi, s.cap_lo = hi_bits, lo_bits, cap_hi, cap_lo
        s.n_hi = s.n_lo = 0
        p = lambda t: None if t is None else t.data_ptr()
        s.k_hi, s.v_hi, s.k_hi_meta, s.v_hi_meta = p(self.k_hi), p(self.v_hi), p(self.k_hi_meta), p(self.v_hi_meta)
        s.k_lo, s.v_lo, s.k_lo_meta, s.v_lo_meta = p(self.k_lo), p(self.v_lo), p(self.k_lo_meta), p(self.v_lo_meta)
        s.pos_hi, s.pos_lo, s.balancer, s.scores = p(self.pos_hi), p(self.pos_lo), p(self.balancer), p(self.scores)
        s.key_mode, s.k_pend, s.v_pend = key_mode, p(self.k_pend), p(self.v_pend)
        self.struct = s
        lib = _lib.load()
        import ctypes
        self.ws_decode = torch.empty(max(256, lib.mikv_decode_step_workspace_bytes(ctypes.byref(s))),
                                     dtype=torch.uint8, device=dev)
        self.out = torch.empty(B, Hq, D, dtype=torch.float32, device=dev)
        self.lse = torch.empty(B, Hq, dtype=torch.float32, device=dev)
        self.hi_logits = torch.empty(B, Hq, cap_hi, dtype=torch.float32, device=dev)
        self.victim = torch.empty(B, Hkv, dtype=torch.int32, device=dev)
        self.zero_pos = torch.zeros(B, Hkv, 1, dtype=torch.int32, device=dev)

    @property
    def n_hi(self) -> int:
        return self.struct.n_hi

    @property
    def n_lo(self) -> int:
        return self.struct.n_lo

    # --- prefill -------------------------------------------------------------------
    def prefill(self, q, k, v, budget_pct, window, policy="h2o", alpha=0.5, w_o=None,
                keep_intermediates=False):
        """q [B,Hq,T,D], k/v [B,Hkv,T,D] fp16 on the device."""
        B, Hq, T, D = q.shape
        dev = self.device
        info = {}
        if self.balancer is not None:
            _lib.mikv_balance_prefill(q, k, self.balancer)
        s_full = torch.empty(B, self.Hkv, T, dtype=torch.float32, device=dev)
        s_head = torch.empty(B, Hq, T, dtype=torch.float32, device=dev) if (
            policy == "criticalkv" or keep_intermediates) else None
        _lib.mikv_score_update(_lib.MIKV_PREFILL, self, q=q, k=k, T=T, scores_full=s_full,
                               scores_head=s_head)
        keep = n_keep(T, budget_pct, window)
        keep_pos = torch.empty(B, self.Hkv, keep, dtype=torch.int32, device=dev)
        evict_pos = torch.empty(B, self.Hkv, T - keep, dtype=torch.int32, device=dev)
        keep_scores = torch.empty(B, self.Hkv, keep, dtype=torch.float32, device=dev)
        vwo = None
        if policy == "criticalkv":
            vwo = torch.empty(B, Hq, T, dtype=torch.float32, device=dev)
            _lib.mikv_select(_lib.MIKV_CRITICALKV, self, T, budget_pct, window, alpha,
                             scores=s_full, scores_head=s_head, v=v, w_o=w_o,
                             hidden=w_o.shape[1], vwo_norm=vwo, keep_pos=keep_pos,
                             evict_pos=evict_pos, keep_scores=keep_scores)
        else:
            _lib.mikv_select(_lib.MIKV_H2O, self, T, budget_pct, window, alpha, scores=s_full,
                             keep_pos=keep_pos, evict_pos=evict_pos, keep_scores=keep_scores)
        _lib.mikv_quantize_append(_lib.MIKV_TIER_HI, self, k, v, keep_pos, keep, 0, keep_scores)
        _lib.mikv_quantize_append(_lib.MIKV_TIER_LO, self, k, v, evict_pos, T - keep, 0)
        if keep_intermediates:
            info = dict(balancer=self.balancer, S=s_full, S_head=s_head, N=vwo,
                        keep_pos=keep_pos, evict_pos=evict_pos, keep_scores=keep_scores)
        return info

    def append_positions(self, k, v, keep_pos, evict_pos, keep_scores=None):
        """Fill the tiers from given positions (no scoring/selection)."""
        _lib.mikv_quantize_append(_lib.MIKV_TIER_HI, self, k, v, keep_pos, keep_pos.shape[2], 0,
                                  keep_scores)
        _lib.mikv_quantize_append(_lib.MIKV_TIER_LO, self, k, v, evict_pos, evict_pos.shape[2], 0)

    # --- decode --------------------------------------------------------------------
    def decode_step(self, q, k, v, L_before, budget_pct, window, policy="h2o", out=None, lse=None):
        """One decode step through mikv_decode_step (append, attention, merge, score update +
        demotion); q [B,Hq,D], k/v [B,Hkv,D] fp16.  Writes out fp32 [B,Hq,D] and lse fp32 [B,Hq]
        (the cache's own buffers unless given) and returns them."""
        pol = _lib.MIKV_H2O if policy == "h2o" else _lib.MIKV_CRITICALKV
        out = self.out if out is None else out
        lse = self.lse if lse is None else lse
        _lib.mikv_decode_step(q, k, v, L_before, budget_pct, window, pol, self, out, lse,
                              ws=self.ws_decode)
        return out, lse

    def decode_step_calls(self, q, k, v, L_before, budget_pct, window, policy="h2o"):
        """The same step as the sequence of the five separate calls."""
        L = L_before + 1
        _lib.mikv_quantize_append(_lib.MIKV_TIER_HI, self, k[:, :, None, :], v[:, :, None, :],
                                  self.zero_pos, 1, L - 1)
        _lib.mikv_decode_attention(q, self, self.out, self.lse, self.hi_logits, ws=self.ws_decode)
        _lib.mikv_score_update(_lib.MIKV_DECODE, self, hi_logits=self.hi_logits, lse=self.lse)
        if policy == "h2o" and self.n_hi > n_keep(L, budget_pct, window):
            _lib.mikv_select(_lib.MIKV_DEMOTE, self, L, budget_pct, window, evict_pos=self.victim)
            _lib.mikv_quantize_append(_lib.MIKV_TIER_DEMOTE, self, None, None, self.victim, 1)
        return self.out, self.lse
