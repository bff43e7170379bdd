"""GPU parity of the post-attention top-k over the full cache (MiKV reading notes, "1-4)
Quantitative analysis": the oracle-eviction simulation) through the C ABI, against the
float64 oracle on the same seeded inputs.

The selection is an integer decision taken on fp32 logits by the kernel and on float64
logits by the oracle: the kept sets must agree except at near-ties, where every differing
slot's logit must lie within 1e-4 of the k-th largest.  The output and lse are compared with
the oracle evaluated on the kernel's kept set, within 1e-4 max-abs (the fp32 level of the
decode attention bar).
"""
import numpy as np
import pytest
import torch

from gpu_helpers import dev, to_np
from mixed_precision_kv_balancer_gb300 import _lib, inputs
from mixed_precision_kv_balancer_gb300.cache import MikvCache
from oracle import attention as oatt

pytestmark = pytest.mark.gpu


def _full_cache(wl):
    x = inputs.make_prefill(wl, 0, "cpu")
    c = MikvCache(wl.B, wl.Hq, wl.Hkv, wl.D, 16, 2, wl.T + 1, 1, dev())
    g = {n: t.to(dev()) for n, t in x.items()}
    c.prefill(g["q"], g["k"], g["v"], 100, 0)          # every token in the FP16 tier, slot = position
    torch.cuda.synchronize()
    assert c.n_hi == wl.T and c.n_lo == 0
    return c, x


def _check(wl, p, heads=None):
    c, x = _full_cache(wl)
    q = inputs.make_decode_token(wl, 0, 0, "cpu")["q"]
    k_keep = oatt.topk_count(wl.T, p)
    out = torch.empty(wl.B, wl.Hq, 128, device=dev())
    lse = torch.empty(wl.B, wl.Hq, device=dev())
    keep = torch.empty(wl.B, wl.Hq, k_keep, dtype=torch.int32, device=dev())
    _lib.mikv_topk_attention(q.to(dev()), c, p, out, lse=lse, keep_idx=keep)
    torch.cuda.synchronize()
    out, lse, keep = to_np(out), to_np(lse), to_np(keep)
    rep = wl.Hq // wl.Hkv
    kn, vn = x["k"].numpy(), x["v"].numpy()
    heads = heads or [(b, h) for b in range(wl.B) for h in range(wl.Hq)]
    for b, h in heads:
        K, V, qh = kn[b, h // rep], vn[b, h // rep], q[b, h].numpy()
        kg = keep[b, h]
        assert np.all(np.diff(kg) > 0), "kept slots must be ascending and distinct"
        _, _, ko = oatt.topk_attention(qh, K, V, k_keep)
        diff = np.setdiff1d(kg, ko).tolist() + np.setdiff1d(ko, kg).tolist()
        if diff:
            l = (K.astype(np.float64) @ qh.astype(np.float64)) / np.sqrt(128)
            kth = np.sort(l)[::-1][k_keep - 1]
            assert max(abs(l[i] - kth) for i in diff) <= 1e-4, f"({b},{h}): selection differs beyond a near-tie"
        ind = np.zeros(wl.T)
        ind[kg] = 1.0
        oo, lo, _ = oatt.topk_attention(qh, K, V, k_keep, select_logits=ind)
        assert np.abs(out[b, h] - oo).max() <= 1e-4, (b, h, np.abs(out[b, h] - oo).max())
        assert abs(lse[b, h] - lo) <= 1e-4, (b, h, lse[b, h], lo)


@pytest.mark.parametrize("p", [0, 20, 100])
def test_topk_attention_small(p):
    _check(inputs.WORKLOADS["tiny"].scaled(B=2, Hq=8, Hkv=2, T=300), p)


def test_topk_attention_chunked_and_ragged():
    """k = 1500 kept tokens (more than one 1024-token chunk), L not a multiple of anything."""
    _check(inputs.WORKLOADS["tiny"].scaled(B=1, Hq=4, Hkv=4, T=3001), 50)


def test_topk_attention_llama_shape_sampled():
    """Llama-3.1-8B heads (GQA 32 / 8) at T = 8192, 20 %: sampled heads against the oracle."""
    wl = inputs.WORKLOADS["llama31_8b"].scaled(B=2, T=8192)
    rng = np.random.default_rng(0)
    heads = [(int(b), int(h)) for b, h in zip(rng.integers(0, wl.B, 12), rng.integers(0, wl.Hq, 12))]
    _check(wl, 20, heads)
