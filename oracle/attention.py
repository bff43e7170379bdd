"""Decode attention over the two-tier mixed-precision cache (oracle, float64).

Sources:
* MiKV reading notes (velog), "2) Outlier-aware handling": quantised keys hold
  I(k * b) and the query is divided by b (q / b), so (q/b).(k b) = q.k; the
  query stays in floating point and absorbs the balancer exactly.
* Same notes, section 3.4 "Accelerating the mixed-precision KV cache", and the
  paperlayer summary, section 3.4: self-attention is permutation invariant
  after positional embedding, so KV pairs can be grouped by precision into
  contiguous tiers; Q and the attention map stay in floating point while K and
  V are low precision.

Definition used (one batch row, one query head h of key head g):
  logit_i = q_h . k_i / sqrt(D)    for a full-precision (FP16) important token,
  logit_i = (q_h / b_g) . k~_i / sqrt(D)  for a quantised token (INT8 important
            tier or the low-bit tier; k~ is the dequantised balanced key),
  p = softmax over the union of both tiers,  o_h = sum_i p_i v~_i,
  lse_h = log sum_i exp(logit_i).
Reading: the FP16 tier stores the original key, so it is attended with the
original query; then a 100% FP16 budget is exactly full attention.
"""
import numpy as np

from .quant import dequantize, unpack_codes


def _tier_kv(tier: dict, bits: int, gs: int, D: int):
    """float64 (K, V) rows of one tier of one (batch, key head)."""
    if tier["n"] == 0:
        return np.zeros((0, D)), np.zeros((0, D))
    if bits == 16:
        k = tier["k"].view(np.float16).astype(np.float64)
        v = tier["v"].view(np.float16).astype(np.float64)
        return k, v
    kc = unpack_codes(tier["k"], bits, D)
    vc = unpack_codes(tier["v"], bits, D)
    return dequantize(kc, tier["k_meta"], gs), dequantize(vc, tier["v_meta"], gs)


def decode_attention_unit(q: np.ndarray, hi: dict, lo: dict, b: np.ndarray | None,
                          hi_bits: int, lo_bits: int, gs: int):
    """q [rep, D] fp16 for the query heads of one key head.

    hi/lo: dict(n, k, v, k_meta, v_meta) holding that key head's tier rows in slot order
    (fp16 bits for a 16-bit tier, packed codes otherwise).
    Returns out [rep, D], lse [rep], hi_logits [rep, n_hi] (float64).
    """
    D = q.shape[1]
    qf = q.astype(np.float64)
    qb = qf / b.astype(np.float64) if b is not None else qf
    k_hi, v_hi = _tier_kv(hi, hi_bits, gs, D)
    k_lo, v_lo = _tier_kv(lo, lo_bits, gs, D)
    q_for_hi = qf if hi_bits == 16 else qb
    l_hi = (q_for_hi @ k_hi.T) / np.sqrt(D)
    l_lo = (qb @ k_lo.T) / np.sqrt(D)
    logits = np.concatenate([l_hi, l_lo], axis=1)
    m = logits.max(axis=1, keepdims=True)
    p = np.exp(logits - m)
    s = p.sum(axis=1, keepdims=True)
    out = (p @ np.concatenate([v_hi, v_lo], axis=0)) / s
    lse = (m + np.log(s))[:, 0]
    return out, lse, l_hi


def topk_count(L: int, budget_pct: int) -> int:
    """Tokens kept per query head by the post-attention top-k: max(1, floor(p * L / 100))."""
    return max(1, budget_pct * L // 100)


def topk_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, keep: int, select_logits=None):
    """Post-attention top-k over a full-precision cache, one query head.

    Source: MiKV reading notes (velog), "1-4) Quantitative analysis": the oracle-eviction
    simulation computes the attention map over the full cache first and applies top-k
    sparsity after the attention, an upper-bound proxy for knowing which past KV pairs
    matter for the token being generated.
    Reading: the kept tokens are the `keep` largest attention weights of this query head
    (equivalently the largest logits), ties to the lower index; the output is attention
    over the kept tokens alone (softmax renormalised over them, as if the rest had been
    evicted).  `select_logits` (default: this function's own float64 logits) is what the
    selection ranks, so a test can take the decision in the kernel's precision.

    q [D], k [L][D], v [L][D] (fp16 or float) -> (out [D], lse, kept indices ascending), float64.
    """
    D = q.shape[0]
    logits = (k.astype(np.float64) @ q.astype(np.float64)) / np.sqrt(D)
    key = logits if select_logits is None else np.asarray(select_logits)
    order = sorted(range(len(key)), key=lambda i: (-float(key[i]), i))
    kept = np.array(sorted(order[:keep]), dtype=np.int64)
    lk = logits[kept]
    m = lk.max()
    w = np.exp(lk - m)
    out = (w @ v.astype(np.float64)[kept]) / w.sum()
    return out, m + np.log(w.sum()), kept
