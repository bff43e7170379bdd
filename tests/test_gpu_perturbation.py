"""GPU parity of the step after attention: y = o . W_O and the per-head output perturbation
||(o - o^) . W_O^(h)||_1 (CriticalKV summary, gist.science, "Theoretical framework"), through
the C ABI, against the float64 oracle on the same seeded inputs.

Bars, from the arithmetic: the kernel multiplies fp16 (hi, lo) splits of o and o - o^
(~2^-22 relative) by the fp16 W_O exactly and accumulates in fp32.  y is a sum of Hq*D
signed terms, so it is checked normwise per batch row (max error <= 1e-5 * max |y|);
the perturbations are sums of absolute values and are checked with the score bar
(normwise 1e-5 per row, componentwise 1e-4 for entries >= 1e-3 of the row maximum).
"""
import numpy as np
import pytest
import torch

from gpu_helpers import assert_scores_close, dev, to_np
from mixed_precision_kv_balancer_gb300 import _lib, inputs
from oracle import perturbation as opt

pytestmark = pytest.mark.gpu


def _case(B, Hq, hidden, seed, eps=1e-2):
    """o like an attention output (|o| ~ 0.3), o^ = o plus a small perturbation, and the
    workload's W_O recipe (N(0, 1/hidden), fp16)."""
    wl = inputs.WORKLOADS["tiny"].scaled(B=B, Hq=Hq, Hkv=1, hidden=hidden)
    g = torch.Generator().manual_seed(seed)
    o = 0.3 * torch.randn(B, Hq, 128, generator=g)
    oh = o + eps * torch.randn(B, Hq, 128, generator=g)
    w = inputs.make_w_o(wl, seed, "cpu")                     # [Hq*D][hidden]
    return o, oh, w


def _run(o, oh, w, want_y=True, want_pert=True):
    B, Hq, _ = o.shape
    hidden = w.shape[1]
    y = torch.full((B, hidden), float("nan"), device=dev()) if want_y else None
    pert = torch.full((B, Hq), float("nan"), device=dev()) if want_pert else None
    _lib.mikv_output_perturbation(o.to(dev()), None if oh is None else oh.to(dev()),
                                  w.t().contiguous().to(dev()), y=y, pert=pert)
    torch.cuda.synchronize()
    return (None if y is None else to_np(y)), (None if pert is None else to_np(pert))


def _assert_y(got, want):
    err = np.abs(got.astype(np.float64) - want).max(axis=1) / np.abs(want).max(axis=1)
    assert err.max() <= 1e-5, f"y normwise error {err.max():.3e}"


@pytest.mark.parametrize("B,Hq,hidden", [(1, 4, 128), (3, 5, 640), (33, 8, 128), (2, 10, 256), (7, 28, 3584),
                                         (70, 6, 384), (5, 2, 256)])
def test_output_perturbation_matches_oracle(B, Hq, hidden):
    o, oh, w = _case(B, Hq, hidden, seed=B * 100 + Hq)
    y, pert = _run(o, oh, w)
    _assert_y(y, opt.output_projection(o.numpy(), w.numpy()))
    assert_scores_close(pert, opt.head_perturbation(o.numpy(), oh.numpy(), w.numpy()))


@pytest.mark.parametrize("B,Hq,hidden", [(64, 32, 4096), (1, 40, 5120)])
def test_output_perturbation_full_size(B, Hq, hidden):
    """The bench's shapes: Llama-3.1-8B (batch 64) and Qwen2.5-32B (batch 1)."""
    o, oh, w = _case(B, Hq, hidden, seed=7)
    y, pert = _run(o, oh, w)
    _assert_y(y, opt.output_projection(o.numpy(), w.numpy()))
    assert_scores_close(pert, opt.head_perturbation(o.numpy(), oh.numpy(), w.numpy()))


def test_identical_outputs_give_exactly_zero():
    o, _, w = _case(5, 8, 512, seed=3)
    _, pert = _run(o, o.clone(), w, want_y=False)
    assert np.all(pert == 0.0)


def test_projection_only_and_raw_distance():
    o, oh, w = _case(4, 6, 384, seed=4)
    y, _ = _run(o, None, w, want_pert=False)                 # y alone needs no o^
    _assert_y(y, opt.output_projection(o.numpy(), w.numpy()))
    pert = torch.empty(4, 6, device=dev())                   # no W_O: ||o - o^||_1 over D
    _lib.mikv_output_perturbation(o.to(dev()), oh.to(dev()), None, pert=pert)
    torch.cuda.synchronize()
    assert_scores_close(to_np(pert), opt.head_perturbation(o.numpy(), oh.numpy()))


def test_large_and_tiny_differences():
    """Relative accuracy does not depend on the size of o - o^ (the difference is split
    into its own hi / lo parts, not formed from the split o)."""
    for eps in (1e-5, 3.0):
        o, oh, w = _case(3, 4, 256, seed=11, eps=eps)
        _, pert = _run(o, oh, w, want_y=False)
        assert_scores_close(pert, opt.head_perturbation(o.numpy(), oh.numpy(), w.numpy()))
