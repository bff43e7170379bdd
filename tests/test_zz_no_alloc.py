"""The allocation-free balancer entry point, for callers that cannot allocate device memory
(a plugin handed only its input and output buffers, or a serving loop that must not enter
the allocator).  It must return exactly what mikv_balance_prefill returns, call after call,
although every call reuses the same static scratch array.

This file is collected last, so a run that stops at the first failure has already run
every other test; it also passes when run alone in a fresh process."""
import numpy as np
import pytest
import torch

from mixed_precision_kv_balancer_gb300 import _lib, inputs

pytestmark = pytest.mark.gpu


def _balancer_pair(wl, layer):
    dev = torch.device("cuda:0")
    x = inputs.make_prefill(wl, layer, "cpu")
    q, k = x["q"].to(dev), x["k"].to(dev)
    ref = torch.empty(wl.B, wl.Hkv, wl.D, dtype=torch.float32, device=dev)
    got = torch.full_like(ref, float("nan"))
    _lib.mikv_balance_prefill(q, k, ref)
    _lib.mikv_balance_prefill_noalloc(q, k, got)
    torch.cuda.synchronize()
    return ref.cpu().numpy(), got.cpu().numpy()


def test_noalloc_matches_workspace_version_twice():
    base = inputs.WORKLOADS["tiny"]
    # two calls in a row with different shapes and values: the second must not see the
    # first one's maxima left in the shared array
    for wl, layer in ((base.scaled(B=4, Hq=32, Hkv=8, T=300, n_outlier=8), 11),
                      (base.scaled(B=2, Hq=8, Hkv=2, T=97, outlier_scale=2.0), 12)):
        ref, got = _balancer_pair(wl, layer)
        np.testing.assert_array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_noalloc_rejects_shapes_above_its_limit():
    dev = torch.device("cuda:0")
    q = torch.zeros(2, 1024, 1, 128, dtype=torch.float16, device=dev)   # B*Hkv = 2048 > 1024
    k = torch.zeros(2, 1024, 1, 128, dtype=torch.float16, device=dev)
    b = torch.empty(2, 1024, 128, dtype=torch.float32, device=dev)
    with pytest.raises(_lib.MikvError) as ei:
        _lib.mikv_balance_prefill_noalloc(q, k, b)
    assert ei.value.code == -2 and "static scratch limit" in str(ei.value)
