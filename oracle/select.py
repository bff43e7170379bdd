"""Token selection (oracle): H2O top-k with a recent window, CriticalKV two-stage
selection, the per-step demotion victim and the V.W_O norms it needs.

Sources:
* MiKV reading notes (velog), "Key contributions, 1)" and "Observation": an
  importance-based eviction policy (H2O) decides which KV pairs are important;
  the evicted ones are kept in low precision instead of being dropped.
  paperlayer summary, section 5: eviction policies keep local (recent) tokens
  and heavy hitters.
* CriticalKV summary (gist.science, arXiv 2502.03805), "Algorithm: perturbation-
  constrained selection": stage 1 spends b' = b * alpha (alpha = 0.5) of the
  budget on the highest attention weights; stage 2 spends the remaining b'' on
  the entries with the largest product of attention weight and the L1 norm of
  the projected value state; "Theoretical framework": the projected value is
  V W_O, W_O the output projection.

Readings (the pages are silent on these):
* budget n_keep(L) = min(L, max(W, floor(p * L / 100))) tokens per
  (batch, key head); the W most recent positions count inside the budget and
  are always kept; the rest of the budget goes to the best-ranked older tokens.
* ranking key (score descending, position ascending): equal scores keep the
  lower position; the demotion victim is the opposite end of the same order
  (score ascending, position descending) among important tokens older than
  the window.  Scores are compared as given (float32 in the library).
* CriticalKV: bud = n_keep - W, b' = floor(alpha * bud), b'' = bud - b';
  stage 2 ranks the tokens not taken by stage 1 by
  C_i = sum over the group's query heads h of S^h_i * N_{h,i},
  N_{h,i} = || v_i W_O[h*D:(h+1)*D, :] ||_1, with the product and the sum
  taken in float32 (h ascending, no fused multiply-add) because they decide
  the selection; A is the accumulated prefill attention (stage 1 ranks by the
  group score, stage 2 uses the per-head scores).  With one query head per
  key head and W_O = I this is the page's A_i * ||V_i||_1.
* The stage-1 claim that the kept attention mass exceeds 50% is reported by
  the page, not enforced.
"""
import math

import numpy as np


def n_keep(L: int, budget_pct: int, window: int) -> int:
    """Important-tier size for a sequence of L tokens (integer arithmetic)."""
    return min(L, max(window, (budget_pct * L) // 100))


def _order_desc(key: np.ndarray, pos: np.ndarray) -> np.ndarray:
    """Indices sorted by (key descending, pos ascending)."""
    return np.lexsort((pos, -key.astype(np.float64)))


def h2o_select(S: np.ndarray, L: int, keep: int, window: int):
    """S [L] scores of one (batch, key head) -> (keep_pos ascending, evict_pos ascending), int32."""
    w = min(window, L)
    recent = np.arange(L - w, L)
    older = np.arange(0, L - w)
    take = keep - w
    assert 0 <= take <= len(older)
    top = older[_order_desc(S[older], older)[:take]]
    kept = np.sort(np.concatenate([top, recent]))
    mask = np.ones(L, dtype=bool)
    mask[kept] = False
    return kept.astype(np.int32), np.nonzero(mask)[0].astype(np.int32)


def criticalkv_budget(keep: int, window: int, L: int, alpha: float):
    """(b', b'') split of the non-window budget."""
    bud = keep - min(window, L)
    b1 = int(math.floor(alpha * bud))
    return b1, bud - b1


def criticalkv_key(S_head: np.ndarray, N: np.ndarray) -> np.ndarray:
    """C_i = sum_h fl32(S^h_i * N_{h,i}), float32, h ascending.  S_head, N: [rep, L] float32."""
    c = np.zeros(S_head.shape[1], dtype=np.float32)
    for h in range(S_head.shape[0]):
        prod = (S_head[h].astype(np.float32) * N[h].astype(np.float32)).astype(np.float32)
        c = (c + prod).astype(np.float32)
    return c


def criticalkv_select(S: np.ndarray, S_head: np.ndarray, N: np.ndarray, L: int, keep: int,
                      window: int, alpha: float):
    """Two-stage selection for one (batch, key head).  S [L] group score, S_head/N [rep, L]."""
    w = min(window, L)
    recent = np.arange(L - w, L)
    older = np.arange(0, L - w)
    b1, b2 = criticalkv_budget(keep, window, L, alpha)
    stage1 = older[_order_desc(S[older], older)[:b1]]
    rest = np.setdiff1d(older, stage1)
    c = criticalkv_key(S_head, N)
    stage2 = rest[_order_desc(c[rest], rest)[:b2]]
    kept = np.sort(np.concatenate([stage1, stage2, recent]))
    mask = np.ones(L, dtype=bool)
    mask[kept] = False
    return kept.astype(np.int32), np.nonzero(mask)[0].astype(np.int32)


def vwo_l1(v: np.ndarray, w_o_h: np.ndarray) -> np.ndarray:
    """N_i = || v_i @ W_O^(h) ||_1 in float64; v [L,D] fp16, w_o_h [D, hidden] fp16 (rows of head h)."""
    return np.abs(v.astype(np.float64) @ w_o_h.astype(np.float64)).sum(axis=1)


def vwo_norms(v: np.ndarray, w_o: np.ndarray, rep: int) -> np.ndarray:
    """All heads: v [B,Hkv,L,D], w_o [Hq*D, hidden] -> N [B,Hq,L] float64."""
    B, Hkv, L, D = v.shape
    Hq = Hkv * rep
    out = np.zeros((B, Hq, L))
    for b in range(B):
        for h in range(Hq):
            out[b, h] = vwo_l1(v[b, h // rep], w_o[h * D:(h + 1) * D])
    return out


def demote_victim(S: np.ndarray, pos: np.ndarray, L: int, window: int) -> int:
    """Important-tier slot to demote: among slots with pos < L - window, the minimum of
    (score ascending, position descending).  S float32 [n_hi], pos [n_hi]."""
    cand = np.nonzero(pos < L - window)[0]
    assert len(cand) > 0
    order = np.lexsort((-pos[cand].astype(np.int64), S[cand].astype(np.float64)))
    return int(cand[order[0]])
