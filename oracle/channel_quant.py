"""Per-channel key quantisation with pending-token buffering (oracle; the pages' Appendix C
alternative).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources:
* MiKV reading notes (velog), "Alternative approach: per-channel quantization" and the
  Appendix C summary: per-channel quantisation isolates outlier channels; applying it to a
  cache means holding KV pairs in a temporary buffer until enough of them have accumulated,
  keeping important and unimportant pairs apart, and evicting from group-wise tiles whose
  sizes become uneven.
* paperlayer summary of arXiv 2402.18096v1, "C. Experiments on per-channel quantization of
  keys": the simulated scheme uses group size 64 and quantises the keys per channel, with 20 %
  of the pairs in FP16 (importance cache) and 80 % in INTx (retained cache).

Readings (the pages give no formula):
* A group is 64 consecutive keys of the retained (low-precision) tier of one (batch, key
  head), in slot order.  Per channel c the group's 64 values are quantised with the per-token
  quantizer's arithmetic (oracle/quant.py: fp32, fp16 scale and zero, round half to even),
  along the token axis instead of the channel axis: scale and zero per (group, channel).
* Per-channel scales already isolate the outlier channels, so the channel balancer is not
  applied to these keys (b = 1); the query attends them as it is.
* Values keep the per-token quantizer (their outliers are not channel-aligned).
* Buffering: a retained key waits in FP16 until 64 pending keys fill a group, which is then
  quantised at once; at prefill the evicted keys in position order fill floor(n / 64) groups
  and the rest waits.  Attention reads the quantised groups and the pending keys.
"""
import numpy as np

from .quant import dequantize, pack_codes, quantize_groups, unpack_codes

GROUP = 64


def quantize_channel_group(k: np.ndarray, bits: int):
    """One group: k [G][D] (fp16 or float32 keys) -> (codes uint8 [G][D], meta uint16 [D][2] =
    fp16 bits of (scale, zero) per channel).  The per-token quantizer on the transpose: each
    channel's G values form one quantisation group."""
    x = k.astype(np.float32)
    G = x.shape[0]
    codes_t, meta = quantize_groups(np.ascontiguousarray(x.T), bits, G)   # [D][G], [D][1][2]
    return np.ascontiguousarray(codes_t.T), meta[:, 0, :]


def dequantize_channel_group(codes: np.ndarray, meta: np.ndarray) -> np.ndarray:
    """Exact s_c * code + z_c in float64: codes [G][D], meta [D][2] -> [G][D]."""
    G = codes.shape[0]
    return np.ascontiguousarray(dequantize(np.ascontiguousarray(codes.T), meta[:, None, :], G).T)


class RetainedKeys:
    """The retained tier's keys of one (batch, key head): quantised groups plus the pending
    FP16 keys, in slot order."""

    def __init__(self, D: int, bits: int, group: int = GROUP):
        self.D, self.bits, self.group = D, bits, group
        self.groups = []          # (codes [group][D], meta [D][2])
        self.pending = []         # fp16 rows

    def append(self, k_row: np.ndarray):
        self.pending.append(np.asarray(k_row, dtype=np.float16))
        if len(self.pending) == self.group:
            self.groups.append(quantize_channel_group(np.stack(self.pending), self.bits))
            self.pending = []

    def __len__(self):
        return len(self.groups) * self.group + len(self.pending)

    def keys_f64(self) -> np.ndarray:
        """Every retained key as attended, float64, slot order: dequantised groups, then the
        pending keys exactly."""
        parts = [dequantize_channel_group(c, m) for c, m in self.groups]
        if self.pending:
            parts.append(np.stack(self.pending).astype(np.float64))
        return np.concatenate(parts, axis=0) if parts else np.zeros((0, self.D))


def decode_attention_channel_keys(q: np.ndarray, k_hi: np.ndarray, v_hi: np.ndarray, retained: RetainedKeys,
                                  v_lo: np.ndarray):
    """Decode attention of one key head's query heads over an FP16 important tier and a
    retained tier with per-channel keys, float64.

    q [rep][D] (fp16); k_hi, v_hi [n_hi][D] fp16 (the important tier, attended as stored);
    retained: the retained tier's keys (groups and pending, slot order); v_lo [n_lo][D] the
    retained values as attended (float, e.g. dequantised per token).  Softmax over the union
    of both tiers, logits q.k / sqrt(D).  Returns out [rep][D], lse [rep]."""
    D = q.shape[1]
    qf = q.astype(np.float64)
    k = np.concatenate([k_hi.astype(np.float64), retained.keys_f64()], axis=0)
    v = np.concatenate([v_hi.astype(np.float64), np.asarray(v_lo, dtype=np.float64)], axis=0)
    assert k.shape[0] == v.shape[0]
    logits = (qf @ k.T) / np.sqrt(D)
    m = logits.max(axis=1, keepdims=True)
    p = np.exp(logits - m)
    s = p.sum(axis=1, keepdims=True)
    return (p @ v) / s, (m + np.log(s))[:, 0]


# ----------------------------------------------------------------------------------------
# The per-channel alternative composed into one layer's cache.
#
# Readings, in addition to those above (the pages name the buffering and the uneven
# group-wise tiles but give no procedure):
# * the important tier is FP16 (the pages' Appendix C setup: 20 % FP16 importance cache,
#   80 % INTx retained cache) and is handled exactly as in the per-token cache (oracle/
#   pipeline.py): selection, H2O scores, demotion victim, swap-remove;
# * a retained pair (key and value) waits in FP16 until 64 pairs fill a group; only then are
#   its keys quantised per channel and its values per token (the MiKV notes speak of holding
#   KV pairs in a temporary buffer until enough of them have accumulated).  Attention reads
#   the quantised groups and the waiting pairs as they are;
# * at prefill the evicted tokens, in position order, fill floor(n / 64) groups and the rest
#   waits; a demoted pair joins the waiting ones (slot order = order of arrival), and the pair
#   that brings them to 64 closes the group at once;
# * the layout follows the per-token cache: per-token code rows (keys and values), value meta
#   per (token, 64-channel group), key meta per (group of 64 slots, channel), positions per
#   slot; waiting pairs sit in an FP16 buffer of 64 rows, the slot's position already in
#   pos_lo.
class ChannelKeyCache:
    """One layer: FP16 important tier + retained tier with per-channel keys (slot order)."""

    def __init__(self, B, Hkv, Hq, D, lo_bits, cap_hi, cap_lo):
        assert cap_lo % GROUP == 0
        self.B, self.Hkv, self.Hq, self.D, self.bits = B, Hkv, Hq, D, lo_bits
        self.rep = Hq // Hkv
        self.cap_hi, self.cap_lo = cap_hi, cap_lo
        self.n_hi = self.n_lo = 0
        rb = D * lo_bits // 8
        self.k_hi = np.zeros((B, Hkv, cap_hi, D), np.uint16)
        self.v_hi = np.zeros((B, Hkv, cap_hi, D), np.uint16)
        self.pos_hi = np.zeros((B, Hkv, cap_hi), np.int32)
        self.scores = np.zeros((B, Hkv, cap_hi), np.float64)
        self.k_lo = np.zeros((B, Hkv, cap_lo, rb), np.uint8)
        self.k_lo_meta = np.zeros((B, Hkv, cap_lo // GROUP, D, 2), np.uint16)
        self.v_lo = np.zeros((B, Hkv, cap_lo, rb), np.uint8)
        self.v_lo_meta = np.zeros((B, Hkv, cap_lo, D // GROUP, 2), np.uint16)
        self.pos_lo = np.zeros((B, Hkv, cap_lo), np.int32)
        self.k_pend = np.zeros((B, Hkv, GROUP, D), np.uint16)
        self.v_pend = np.zeros((B, Hkv, GROUP, D), np.uint16)

    @property
    def n_pending(self) -> int:
        return self.n_lo % GROUP

    # -- the retained tier ------------------------------------------------------------
    def _close_group(self, b, g, first):
        """Quantise the 64 waiting pairs into slots first .. first + 63."""
        k = self.k_pend[b, g].view(np.float16)
        v = self.v_pend[b, g].view(np.float16).astype(np.float32)
        kc, km = quantize_channel_group(k, self.bits)
        vc, vm = quantize_groups(v, self.bits, GROUP)
        sl = slice(first, first + GROUP)
        self.k_lo[b, g, sl] = pack_codes(kc, self.bits)
        self.k_lo_meta[b, g, first // GROUP] = km
        self.v_lo[b, g, sl] = pack_codes(vc, self.bits)
        self.v_lo_meta[b, g, sl] = vm

    def _retain(self, b, g, slot, k_row, v_row, pos):
        """Pair (k_row, v_row) fp16 bits enters retained slot `slot` (waiting)."""
        p = slot % GROUP
        self.k_pend[b, g, p] = k_row
        self.v_pend[b, g, p] = v_row
        self.pos_lo[b, g, slot] = pos
        if p == GROUP - 1:
            self._close_group(b, g, slot - (GROUP - 1))

    # -- appends ------------------------------------------------------------------------
    def append(self, tier, k, v, src_pos, pos_base=0, src_scores=None):
        """k, v [B,Hkv,S,D] fp16; src_pos [B,Hkv,n] -> slots n_tier .. n_tier + n - 1."""
        n = src_pos.shape[2]
        base = self.n_hi if tier == "hi" else self.n_lo
        assert base + n <= (self.cap_hi if tier == "hi" else self.cap_lo)
        for b in range(self.B):
            for g in range(self.Hkv):
                idx = src_pos[b, g].astype(np.int64)
                for j in range(n):
                    kr, vr = k[b, g, idx[j]].view(np.uint16), v[b, g, idx[j]].view(np.uint16)
                    if tier == "hi":
                        self.k_hi[b, g, base + j], self.v_hi[b, g, base + j] = kr, vr
                        self.pos_hi[b, g, base + j] = idx[j] + pos_base
                        self.scores[b, g, base + j] = 0.0 if src_scores is None else src_scores[b, g, j]
                    else:
                        self._retain(b, g, base + j, kr, vr, idx[j] + pos_base)
        if tier == "hi":
            self.n_hi += n
        else:
            self.n_lo += n

    def demote(self, victims):
        """victims [B,Hkv] important slots: the pair joins the waiting ones, swap-remove."""
        last = self.n_hi - 1
        for b in range(self.B):
            for g in range(self.Hkv):
                j = int(victims[b, g])
                self._retain(b, g, self.n_lo, self.k_hi[b, g, j].copy(), self.v_hi[b, g, j].copy(),
                             self.pos_hi[b, g, j])
                for arr in (self.k_hi, self.v_hi, self.pos_hi, self.scores):
                    arr[b, g, j] = arr[b, g, last]
        self.n_hi -= 1
        self.n_lo += 1

    # -- attention ----------------------------------------------------------------------
    def retained(self, b, g):
        """(RetainedKeys of the unit, retained values as attended [n_lo][D] float64)."""
        D, bits = self.D, self.bits
        r = RetainedKeys(D, bits)
        full = self.n_lo - self.n_pending
        vals = []
        for gi in range(full // GROUP):
            sl = slice(gi * GROUP, (gi + 1) * GROUP)
            r.groups.append((unpack_codes(self.k_lo[b, g, sl], bits, D), self.k_lo_meta[b, g, gi]))
            vals.append(dequantize(unpack_codes(self.v_lo[b, g, sl], bits, D), self.v_lo_meta[b, g, sl], GROUP))
        r.pending = [row.view(np.float16) for row in self.k_pend[b, g, :self.n_pending]]
        vals.append(self.v_pend[b, g, :self.n_pending].view(np.float16).astype(np.float64))
        return r, np.concatenate(vals, axis=0)

    def attend(self, q):
        """q [B,Hq,D] fp16 -> out [B,Hq,D], lse [B,Hq], hi_logits [B,Hq,n_hi] (float64)."""
        B, Hq, D = q.shape
        rep = self.rep
        out, lse = np.zeros((B, Hq, D)), np.zeros((B, Hq))
        logits = np.zeros((B, Hq, self.n_hi))
        for b in range(B):
            for g in range(self.Hkv):
                hs = slice(g * rep, (g + 1) * rep)
                k_hi = self.k_hi[b, g, :self.n_hi].view(np.float16)
                v_hi = self.v_hi[b, g, :self.n_hi].view(np.float16)
                r, v_lo = self.retained(b, g)
                out[b, hs], lse[b, hs] = decode_attention_channel_keys(q[b, hs], k_hi, v_hi, r, v_lo)
                logits[b, hs] = (q[b, hs].astype(np.float64) @ k_hi.astype(np.float64).T) / np.sqrt(D)
        return out, lse, logits


def prefill_channel(q, k, v, *, lo_bits, budget_pct, window, extra_steps=0):
    """One layer's per-channel-key cache from prompt activations q [B,Hq,T,D], k/v [B,Hkv,T,D]
    fp16: H2O scores and selection as in the per-token pipeline (no balancer: per-channel
    scales already isolate the outlier channels), important tokens FP16, the rest retained."""
    from . import scores as osc
    from . import select as osel
    B, Hq, T, D = q.shape
    Hkv = k.shape[1]
    _, s_grp = osc.prefill_scores(q, k)
    keep = osel.n_keep(T, budget_pct, window)
    keep_pos = np.zeros((B, Hkv, keep), np.int32)
    evict_pos = np.zeros((B, Hkv, T - keep), np.int32)
    for b in range(B):
        for g in range(Hkv):
            keep_pos[b, g], evict_pos[b, g] = osel.h2o_select(s_grp[b, g].astype(np.float32), T, keep, window)
    cap_lo = -(-(T - keep + extra_steps + 1) // GROUP) * GROUP
    cache = ChannelKeyCache(B, Hkv, Hq, D, lo_bits, keep + extra_steps + 1, cap_lo)
    cache.append("hi", k, v, keep_pos, 0, np.take_along_axis(s_grp, keep_pos.astype(np.int64), axis=2))
    cache.append("lo", k, v, evict_pos, 0)
    return cache, dict(S=s_grp, keep_pos=keep_pos, evict_pos=evict_pos)


def decode_step_channel(cache, q_new, k_new, v_new, L_before, *, budget_pct, window):
    """One decode step (per-token pipeline order): append the new token to the important tier,
    attend, add the step's attention to the H2O scores, demote at most one pair into the
    retained tier's waiting buffer.  Returns (out, lse, victims or None)."""
    from . import scores as osc
    from . import select as osel
    L = L_before + 1
    B, Hkv = cache.B, cache.Hkv
    cache.append("hi", k_new[:, :, None, :], v_new[:, :, None, :], np.zeros((B, Hkv, 1), np.int32), L - 1)
    out, lse, logits = cache.attend(q_new)
    rep = cache.rep
    for b in range(B):
        for g in range(Hkv):
            hs = slice(g * rep, (g + 1) * rep)
            cache.scores[b, g, :cache.n_hi] = osc.decode_score_update(cache.scores[b, g, :cache.n_hi],
                                                                     logits[b, hs], lse[b, hs])
    victims = None
    if cache.n_hi > osel.n_keep(L, budget_pct, window):
        victims = np.zeros((B, Hkv), np.int32)
        for b in range(B):
            for g in range(Hkv):
                victims[b, g] = osel.demote_victim(cache.scores[b, g, :cache.n_hi].astype(np.float32),
                                                   cache.pos_hi[b, g, :cache.n_hi], L, window)
        cache.demote(victims)
    return out, lse, victims
