"""Shared helpers of the GPU parity tests (compare library buffers with the oracle's)."""
import numpy as np
import torch

ATTN_TOL = 2e-3        # max-abs on attention outputs
SCORE_RTOL = 1e-5      # relative, on H2O scores and V.W_O norms


def dev():
    return torch.device("cuda:0")


def to_np(t):
    return t.detach().cpu().numpy()


def u16(t):
    """fp16 tensor -> its raw bits as uint16 numpy."""
    return to_np(t.contiguous().view(torch.int16)).view(np.uint16)


def compare_tiers(gc, oc, what=("hi", "lo")):
    """Bit-exact comparison of every occupied slot of the two caches."""
    assert gc.n_hi == oc.n_hi and gc.n_lo == oc.n_lo, (gc.n_hi, oc.n_hi, gc.n_lo, oc.n_lo)
    nh, nl = gc.n_hi, gc.n_lo
    if "hi" in what:
        if gc.hi_bits == 16:
            np.testing.assert_array_equal(u16(gc.k_hi[:, :, :nh]), oc.k_hi[:, :, :nh])
            np.testing.assert_array_equal(u16(gc.v_hi[:, :, :nh]), oc.v_hi[:, :, :nh])
        else:
            np.testing.assert_array_equal(to_np(gc.k_hi[:, :, :nh]), oc.k_hi[:, :, :nh])
            np.testing.assert_array_equal(to_np(gc.v_hi[:, :, :nh]), oc.v_hi[:, :, :nh])
            np.testing.assert_array_equal(u16(gc.k_hi_meta[:, :, :nh]), oc.k_hi_meta[:, :, :nh])
            np.testing.assert_array_equal(u16(gc.v_hi_meta[:, :, :nh]), oc.v_hi_meta[:, :, :nh])
        np.testing.assert_array_equal(to_np(gc.pos_hi[:, :, :nh]), oc.pos_hi[:, :, :nh])
    if "lo" in what:
        np.testing.assert_array_equal(to_np(gc.k_lo[:, :, :nl]), oc.k_lo[:, :, :nl])
        np.testing.assert_array_equal(to_np(gc.v_lo[:, :, :nl]), oc.v_lo[:, :, :nl])
        np.testing.assert_array_equal(u16(gc.k_lo_meta[:, :, :nl]), oc.k_lo_meta[:, :, :nl])
        np.testing.assert_array_equal(u16(gc.v_lo_meta[:, :, :nl]), oc.v_lo_meta[:, :, :nl])
        np.testing.assert_array_equal(to_np(gc.pos_lo[:, :, :nl]), oc.pos_lo[:, :, :nl])


def assert_scores_close(got, want, rtol=SCORE_RTOL, comp_rtol=1e-4):
    """Scores/norms bar.  Normwise, per (batch, head) row: max_i |got_i - want_i| <= rtol *
    max_i |want_i| (the reading of "within 1e-5 relative" for an accumulated vector).
    Componentwise diagnostic for entries >= 1e-3 * row max: |d_i| / |want_i| <= comp_rtol,
    the bound fp32 logits allow when |q.k| reaches ~2^12 (one fp32 ulp there is 2.4e-4, i.e.
    ~3e-5 of a probability, doubled for the row log-sum-exp).  Returns the measured
    (normwise, componentwise) maxima."""
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    if want.size == 0:  # e.g. an empty important tier
        return 0.0, 0.0
    mx = np.abs(want).max(axis=-1, keepdims=True)
    d = np.abs(got - want)
    norm = (d / np.maximum(mx, 1e-30)).max()
    assert norm <= rtol, f"normwise relative error {norm:.3e} > {rtol}"
    big = np.abs(want) >= 1e-3 * mx
    rel = np.where(big, d / np.maximum(np.abs(want), 1e-30), 0)
    if rel.max() > comp_rtol:
        idx = np.unravel_index(rel.argmax(), rel.shape)
        raise AssertionError(f"componentwise relative error {rel.max():.3e} at {idx}: got "
                             f"{got[idx]!r} want {want[idx]!r} row max {mx[idx[:-1]][0]!r}")
    return float(norm), float(rel.max())
