"""Seeded synthetic inputs shared by the CUDA path, the oracle tests and the bench.

This module only draws numbers.  It holds none of the cache method's arithmetic
(no balancer, no quantizer, no attention, no selection): it produces fp16
query/key/value tensors shaped like the activations the MiKV pages study, and
nothing else.  Both sides of every parity test receive the very same tensors
from here.

Recipe (stand-in for model activations on MMLU/GSM8k/HumanEval/Line-Retrieval/
Ruler/LongBench, which this build does not have):

* q, k, v ~ N(0, 1) drawn by a torch generator seeded per
  (seed, layer, tensor, step) sub-stream.
* Systematic outlier channels in Q and K ("Outlier-aware" section of the MiKV
  notes; Figure 5 there: a few channels per head carry large magnitudes, and
  their positions are stable along the sequence).  Per head, ``n_outlier``
  channels are drawn once (independently for every query head and every key
  head) and multiplied by ``outlier_scale`` at every position.
* Rotary position embedding, rotate-half convention, pairs (j, j + D/2),
  frequency theta**(-2j/D), positions 0..T-1 for the prompt and T+s for decode
  step s.  It is applied after the outlier scaling, so RoPE spreads each
  outlier into its rotation partner (the notes observe RoPE duplicating the
  outliers).
* V gets neither outliers nor RoPE.
* W_O (CriticalKV workload) ~ N(0, 1/hidden), fp16, shape [Hq*D, hidden]:
  row block [h*D, (h+1)*D) is the slice that multiplies head h's output.
"""
from __future__ import annotations

import dataclasses
import hashlib
import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: shapes, cache policy and input recipe."""

    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    T: int
    steps: int
    budget_pct: int
    window: int
    hi_bits: int
    lo_bits: int
    n_outlier: int
    outlier_scale: float
    rope_theta: float
    policy: str = "h2o"          # "h2o" or "criticalkv"
    alpha: float = 0.5
    layers: int = 1
    hidden: int = 0              # W_O output width (criticalkv only)
    seed: int = 0

    @property
    def rep(self) -> int:
        return self.Hq // self.Hkv

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads.  Values marked "(chosen)" are not stated for that
# workload and take the plainest neighbouring value.
WORKLOADS = {
    # batch 1, 4 heads MHA, prompt 512 + 32 decode steps, 20% FP16 (window 32), INT4.
    "tiny": Workload("tiny", B=1, Hq=4, Hkv=4, D=128, T=512, steps=32,
                     budget_pct=20, window=32, hi_bits=16, lo_bits=4,
                     n_outlier=4, outlier_scale=16.0, rope_theta=1e4),
    # Llama-2-7B layer: 32 heads MHA, batch 8, 4096 + 128 steps, 25% FP16, INT2.
    "llama2_7b": Workload("llama2_7b", B=8, Hq=32, Hkv=32, D=128, T=4096, steps=128,
                          budget_pct=25, window=32, hi_bits=16, lo_bits=2,   # window (chosen)
                          n_outlier=6, outlier_scale=20.0, rope_theta=1e4),
    # Llama-3.1-8B GQA layer: 32/8 heads, batch 16, 16384 + 64 steps, 20% INT8 (window 64), INT4.
    "llama31_8b": Workload("llama31_8b", B=16, Hq=32, Hkv=8, D=128, T=16384, steps=64,
                           budget_pct=20, window=64, hi_bits=8, lo_bits=4,
                           n_outlier=8, outlier_scale=16.0, rope_theta=5e5),
    # Qwen2.5-32B GQA layer: 40/8 heads, batch 1, 32768, CriticalKV 40% alpha 0.5, FP16 / INT2.
    "qwen25_32b": Workload("qwen25_32b", B=1, Hq=40, Hkv=8, D=128, T=32768, steps=32,  # steps (chosen)
                           budget_pct=40, window=32, hi_bits=16, lo_bits=2,            # window (chosen)
                           n_outlier=8, outlier_scale=16.0, rope_theta=5e5,            # theta (chosen)
                           policy="criticalkv", alpha=0.5, hidden=5120),
    # Full depth: 32 layers of Llama-3.1-8B KV shape, batch 64, 8192 + 16 steps, 20% FP16, INT2.
    "llama31_8b_full": Workload("llama31_8b_full", B=64, Hq=32, Hkv=8, D=128, T=8192, steps=16,
                                budget_pct=20, window=32, hi_bits=16, lo_bits=2,    # window (chosen)
                                n_outlier=8, outlier_scale=16.0, rope_theta=5e5,    # theta (chosen)
                                layers=32),
}

_TENSOR_IDS = {"q": 1, "k": 2, "v": 3, "w_o": 4, "q_out": 5, "k_out": 6}


def substream_seed(seed: int, layer: int, tensor: str, step: int) -> int:
    """Derive an independent 63-bit seed for one (layer, tensor, step) stream."""
    tag = f"mikv/{seed}/{layer}/{_TENSOR_IDS[tensor]}/{step}".encode()
    return int.from_bytes(hashlib.sha256(tag).digest()[:8], "little") & ((1 << 63) - 1)


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def outlier_channels(wl: Workload, layer: int, which: str) -> torch.Tensor:
    """[H, n_outlier] channel indices (int64, CPU) for 'q' (per query head) or 'k' (per key head)."""
    H = wl.Hq if which == "q" else wl.Hkv
    g = _gen("cpu", substream_seed(wl.seed, layer, which + "_out", 0))
    rows = [torch.randperm(wl.D, generator=g)[: wl.n_outlier] for _ in range(H)]
    return torch.stack(rows) if rows else torch.zeros(0, wl.n_outlier, dtype=torch.int64)


def _channel_gain(wl: Workload, layer: int, which: str, device) -> torch.Tensor:
    """[H, D] float32 multiplier: outlier_scale on the head's outlier channels, 1 elsewhere."""
    idx = outlier_channels(wl, layer, which)
    gain = torch.ones(idx.shape[0], wl.D, dtype=torch.float32)
    if wl.n_outlier > 0:
        gain.scatter_(1, idx, wl.outlier_scale)
    return gain.to(device)


def _rope(x: torch.Tensor, pos: torch.Tensor, theta: float) -> torch.Tensor:
    """Rotate-half rotary embedding on the last dim of x (float32) at integer positions pos."""
    D = x.shape[-1]
    half = D // 2
    j = torch.arange(half, dtype=torch.float64, device=x.device)
    inv = torch.pow(torch.tensor(theta, dtype=torch.float64, device=x.device), -2.0 * j / D)
    ang = (pos.to(torch.float64)[:, None] * inv[None, :])
    cos = torch.cos(ang).to(torch.float32)
    sin = torch.sin(ang).to(torch.float32)
    x1, x2 = x[..., :half], x[..., half:]
    return torch.cat([x1 * cos - x2 * sin, x2 * cos + x1 * sin], dim=-1)


def _draw(shape, device, seed) -> torch.Tensor:
    return torch.randn(shape, generator=_gen(device, seed), device=device, dtype=torch.float32)


def make_prefill(wl: Workload, layer: int = 0, device="cpu", b_chunk: int | None = None):
    """Prompt activations of one layer: dict(q=[B,Hq,T,D], k=[B,Hkv,T,D], v=[B,Hkv,T,D]) fp16.

    ``b_chunk`` bounds the float32 working set on large workloads; the values
    do not depend on it (every batch row has its own sub-stream).
    """
    B, T, D = wl.B, wl.T, wl.D
    pos = torch.arange(T, device=device)
    out = {}
    for name, H in (("q", wl.Hq), ("k", wl.Hkv), ("v", wl.Hkv)):
        t = torch.empty(B, H, T, D, dtype=torch.float16, device=device)
        gain = None if name == "v" else _channel_gain(wl, layer, name, device)
        for b in range(B):
            x = _draw((H, T, D), device, substream_seed(wl.seed, layer, name, b))
            if gain is not None:
                x = x * gain[:, None, :]
                x = _rope(x, pos, wl.rope_theta)
            t[b] = x.to(torch.float16)
        out[name] = t
    return out


def make_decode_token(wl: Workload, layer: int, step: int, device="cpu"):
    """New token of decode step ``step`` (position T+step): q [B,Hq,D], k [B,Hkv,D], v [B,Hkv,D] fp16."""
    B, D = wl.B, wl.D
    pos = torch.full((1,), wl.T + step, device=device, dtype=torch.int64)
    out = {}
    for name, H in (("q", wl.Hq), ("k", wl.Hkv), ("v", wl.Hkv)):
        # decode sub-streams are keyed by step; prompt sub-streams by batch row.
        x = _draw((B, H, 1, D), device, substream_seed(wl.seed, layer, name, 1_000_000 + step))
        if name != "v":
            x = x * _channel_gain(wl, layer, name, device)[None, :, None, :]
            x = _rope(x, pos, wl.rope_theta)
        out[name] = x[:, :, 0, :].to(torch.float16).contiguous()
    return out


def make_w_o(wl: Workload, layer: int = 0, device="cpu") -> torch.Tensor:
    """Output projection [Hq*D, hidden] fp16 ~ N(0, 1/hidden)."""
    hidden = wl.hidden or wl.Hq * wl.D
    x = _draw((wl.Hq * wl.D, hidden), device, substream_seed(wl.seed, layer, "w_o", 0))
    return (x / math.sqrt(hidden)).to(torch.float16)
