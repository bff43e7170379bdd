"""H2O accumulated attention importance (oracle, float64).

Sources: MiKV reading notes (velog), "Observation 1-4" and "Key contributions,
1)": the eviction policy is H2O (Zhang et al., 2023), which ranks cached tokens
by accumulated attention; paperlayer summary of arXiv 2402.18096v1, section 5
(heavy hitters and local tokens).  The pages name H2O but do not print its
formula; the plainest reading is used:

* prefill: for every prompt token i, the sum over all query rows t >= i of
  the causal softmax probability softmax_t(q_t . k / sqrt(D))_i;
* decode: every step adds that step's attention probability of each cached
  important-tier token;
* GQA: a key head's score is the sum over the query heads of its group.  With
  one query head per key head this is H2O itself; summing instead of averaging
  does not change any ranking.
* Only important-tier (high-precision) tokens accumulate during decode: the
  pages never promote a retained low-bit token back, so its score is unused.
"""
import numpy as np


def prefill_column_scores(qh: np.ndarray, k: np.ndarray) -> np.ndarray:
    """One query head: qh [T,D], k [T,D] (fp16) -> S [T] float64, S_i = sum_{t>=i} softmax_t(...)_i."""
    T, D = qh.shape
    logits = (qh.astype(np.float64) @ k.astype(np.float64).T) / np.sqrt(D)   # [t, i]
    causal = np.tril(np.ones((T, T), dtype=bool))                            # key i <= query t
    logits = np.where(causal, logits, -np.inf)
    m = logits.max(axis=1, keepdims=True)
    p = np.exp(logits - m)
    p = p / p.sum(axis=1, keepdims=True)
    return p.sum(axis=0)


def prefill_scores(q: np.ndarray, k: np.ndarray):
    """q [B,Hq,T,D], k [B,Hkv,T,D] -> (S_head [B,Hq,T], S [B,Hkv,T]) float64."""
    B, Hq, T, D = q.shape
    Hkv = k.shape[1]
    rep = Hq // Hkv
    s_head = np.zeros((B, Hq, T))
    for b in range(B):
        for h in range(Hq):
            s_head[b, h] = prefill_column_scores(q[b, h], k[b, h // rep])
    s_grp = s_head.reshape(B, Hkv, rep, T).sum(axis=2)
    return s_head, s_grp


def row_lse(qh: np.ndarray, k: np.ndarray, rows) -> np.ndarray:
    """Natural log-sum-exp of causal row t (keys 0..t) for each t in rows, float64."""
    D = qh.shape[1]
    kf = k.astype(np.float64)
    out = np.empty(len(rows))
    for j, t in enumerate(rows):
        l = (kf[: t + 1] @ qh[t].astype(np.float64)) / np.sqrt(D)
        m = l.max()
        out[j] = m + np.log(np.exp(l - m).sum())
    return out


def column_scores_at(qh: np.ndarray, k: np.ndarray, cols) -> np.ndarray:
    """S_i for the listed key columns only (same definition as prefill_column_scores)."""
    T, D = qh.shape
    lo = int(min(cols))
    rows = list(range(lo, T))
    lse = row_lse(qh, k, rows)
    qf = qh[lo:].astype(np.float64)
    out = np.empty(len(cols))
    for j, i in enumerate(cols):
        l = (qf[i - lo:] @ k[i].astype(np.float64)) / np.sqrt(D)      # rows t >= i
        out[j] = np.exp(l - lse[i - lo:]).sum()
    return out


def decode_score_update(s: np.ndarray, logits: np.ndarray, lse: np.ndarray) -> np.ndarray:
    """One (batch, key head): s [n_hi] += sum_h exp(logits[h, j] - lse[h]); logits [rep, n_hi], lse [rep]."""
    return s + np.exp(logits - lse[:, None]).sum(axis=0)
