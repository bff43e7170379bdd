"""Pins for the oracle's post-attention top-k ("oracle eviction", MiKV reading notes, "1-4)
Quantitative analysis": attention map over the full cache first, top-k sparsity after it)."""
import numpy as np
import pytest

from oracle import attention as oatt


def _full(q, k, v):
    l = (k.astype(np.float64) @ q.astype(np.float64)) / np.sqrt(q.shape[0])
    p = np.exp(l - l.max())
    return (p @ v.astype(np.float64)) / p.sum(), l.max() + np.log(p.sum())


def test_topk_count():
    assert oatt.topk_count(8192, 20) == 1638
    assert oatt.topk_count(10, 0) == 1          # at least the strongest token
    assert oatt.topk_count(7, 100) == 7
    assert oatt.topk_count(32768, 40) == 13107


@pytest.mark.parametrize("seed", range(3))
def test_keeping_everything_is_full_attention(seed):
    rng = np.random.default_rng(seed)
    L, D = 37, 16
    q, k, v = rng.standard_normal(D), rng.standard_normal((L, D)), rng.standard_normal((L, D))
    out, lse, kept = oatt.topk_attention(q, k, v, L)
    fo, fl = _full(q, k, v)
    np.testing.assert_allclose(out, fo, rtol=1e-13, atol=1e-13)
    assert lse == pytest.approx(fl, rel=1e-14)
    assert list(kept) == list(range(L))


def test_keeping_one_returns_the_strongest_value_row():
    rng = np.random.default_rng(7)
    L, D = 20, 8
    q, k, v = rng.standard_normal(D), rng.standard_normal((L, D)), rng.standard_normal((L, D))
    out, lse, kept = oatt.topk_attention(q, k, v, 1)
    i = int(np.argmax(k @ q))
    assert list(kept) == [i]
    np.testing.assert_array_equal(out, v[i])
    assert lse == pytest.approx(float(k[i] @ q) / np.sqrt(D), rel=1e-14)


def test_hand_case_with_a_tie():
    # D = 4 (sqrt 2): logits = k.q / 2; rows 1 and 3 tie at the top-2 boundary -> the lower (1) is kept
    q = np.array([2.0, 0.0, 0.0, 0.0])
    k = np.array([[4.0, 0, 0, 0], [1.0, 0, 0, 0], [0.0, 0, 0, 0], [1.0, 0, 0, 0]])
    v = np.array([[1.0, 0, 0, 0], [0.0, 1, 0, 0], [0.0, 0, 1, 0], [0.0, 0, 0, 1]])
    out, lse, kept = oatt.topk_attention(q, k, v, 2)        # logits 4, 1, 0, 1
    assert list(kept) == [0, 1]
    w = np.array([1.0, np.exp(-3.0)])
    np.testing.assert_allclose(out, np.array([w[0], w[1], 0, 0]) / w.sum(), rtol=1e-15)
    assert lse == pytest.approx(4.0 + np.log(1.0 + np.exp(-3.0)), rel=1e-15)


@pytest.mark.parametrize("seed", range(4))
def test_brute_force_and_mass_bound(seed):
    rng = np.random.default_rng(10 + seed)
    L, D = int(rng.integers(3, 30)), 8
    q, k, v = rng.standard_normal(D), rng.standard_normal((L, D)), rng.standard_normal((L, D))
    keep = int(rng.integers(1, L + 1))
    out, lse, kept = oatt.topk_attention(q, k, v, keep)
    l = (k @ q) / np.sqrt(D)
    # every kept logit >= every dropped one
    dropped = np.setdiff1d(np.arange(L), kept)
    if len(dropped):
        assert l[kept].min() >= l[dropped].max()
    # the kept softmax mass is at least keep / L (the top-k hold at least the average share)
    p = np.exp(l - l.max()) / np.exp(l - l.max()).sum()
    assert p[kept].sum() >= keep / L - 1e-12
    # brute force: renormalised weighted sum over the kept set
    w = np.exp(l[kept] - l[kept].max())
    np.testing.assert_allclose(out, (w @ v[kept]) / w.sum(), rtol=1e-12, atol=1e-14)
    # selecting on supplied logits follows them, not the oracle's own
    out2, _, kept2 = oatt.topk_attention(q, k, v, keep, select_logits=-l)
    assert set(kept2) == set(np.argsort(l, kind="stable")[:keep]) or keep == L
