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

from .quant import dequantize, quantize_groups

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
