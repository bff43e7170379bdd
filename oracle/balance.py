"""Channel balancer (oracle).

Source: "No Token Left Behind" reading notes (velog), section "Key contributions,
2) Outlier-aware handling", balancer equation: during prefill, for layer l,
head h and channel c, b_lhc is the square root of the ratio between the largest
|q| and the largest |k| of that channel over the prompt tokens 0..t-1; keys are
multiplied by b before quantisation and queries are divided by it.  The
paperlayer summary of arXiv 2402.18096v1, section 3.2, states the same
(prefill-computed balancer applied to keys and queries).

Readings where the pages are silent:
* GQA: one b per key head (keys are shared).  The query maximum runs over all
  query heads of the key head's group, so that q/b uses the b its key was
  scaled with.  With one query per key head this is the page's formula.
* Batch: b is per sequence, indexed [batch, key head, channel].
* q and k are the post-RoPE tensors, the ones that are cached and attended.
* A channel whose query or key maximum is zero gets b = 1.
* The notes claim b <= 1 in one place; the formula gives b > 1 wherever the
  query maximum is larger.  The formula is used as written, with no clamp.
* Arithmetic: maxima are exact (|fp16| widened to float32); the ratio and the
  square root are float32, round-to-nearest-even, in that order.
"""
import numpy as np


def channel_balancer(q: np.ndarray, k: np.ndarray) -> np.ndarray:
    """q [B,Hq,T,D] fp16, k [B,Hkv,T,D] fp16 -> b [B,Hkv,D] float32."""
    B, Hq, T, D = q.shape
    Hkv = k.shape[1]
    assert Hq % Hkv == 0 and k.shape == (B, Hkv, T, D)
    rep = Hq // Hkv
    qa = np.abs(q.astype(np.float32)).reshape(B, Hkv, rep, T, D)
    m_q = qa.max(axis=(2, 3))                              # [B,Hkv,D]
    m_k = np.abs(k.astype(np.float32)).max(axis=2)         # [B,Hkv,D]
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = (m_q / m_k).astype(np.float32)             # float32 RN division
        b = np.sqrt(ratio).astype(np.float32)              # float32 RN square root
    b = np.where((m_q == 0) | (m_k == 0), np.float32(1.0), b)
    return b.astype(np.float32)
