"""Pins for the oracle's selection rules (no GPU).

Definitions: H2O top-k with recent window (MiKV notes, "Key contributions, 1)";
paperlayer section 5: local tokens and heavy hitters); CriticalKV two-stage
selection (gist.science CriticalKV summary, "Algorithm"): b' = b*alpha by
attention weight, the remaining b'' by A_i * ||V_i W_O||_1.
"""
import math

import numpy as np
import pytest

from oracle import select


def _brute_h2o(S, L, keep, W):
    w = min(W, L)
    older = sorted(range(L - w), key=lambda i: (-float(S[i]), i))
    kept = sorted(older[: keep - w] + list(range(L - w, L)))
    return kept


def test_n_keep():
    assert select.n_keep(512, 20, 32) == 102
    assert select.n_keep(4096, 25, 32) == 1024
    assert select.n_keep(16384, 20, 64) == 3276
    assert select.n_keep(32768, 40, 32) == 13107
    assert select.n_keep(8192, 20, 32) == 1638
    assert select.n_keep(100, 20, 32) == 32      # window floor
    assert select.n_keep(10, 20, 32) == 10       # shorter than the window: keep all
    assert select.n_keep(50, 100, 0) == 50
    assert select.n_keep(50, 0, 0) == 0


@pytest.mark.parametrize("seed", range(6))
def test_h2o_matches_sorted_brute_force_with_ties(seed):
    rng = np.random.default_rng(seed)
    L = int(rng.integers(1, 60))
    W = int(rng.integers(0, 12))
    S = rng.integers(0, 5, size=L).astype(np.float32)     # many exact ties
    keep = select.n_keep(L, int(rng.integers(0, 101)), W)
    kp, ep = select.h2o_select(S, L, keep, W)
    assert kp.tolist() == _brute_h2o(S, L, keep, W)
    assert sorted(kp.tolist() + ep.tolist()) == list(range(L))
    assert ep.tolist() == sorted(ep.tolist())


def test_h2o_tie_keeps_lower_position():
    S = np.array([1, 3, 3, 3, 0, 0], np.float32)
    kp, _ = select.h2o_select(S, 6, 4, 2)     # window {4,5}; two of the 3-ties: positions 1, 2
    assert kp.tolist() == [1, 2, 4, 5]


def test_criticalkv_budget_split():
    assert select.criticalkv_budget(13107, 32, 32768, 0.5) == (6537, 6538)
    assert select.criticalkv_budget(102, 32, 512, 0.5) == (35, 35)
    assert select.criticalkv_budget(101, 32, 512, 0.5) == (34, 35)
    assert select.criticalkv_budget(50, 0, 100, 1.0) == (50, 0)
    assert select.criticalkv_budget(50, 0, 100, 0.0) == (0, 50)


def _brute_vwo(v, w):
    """Python loops: sum_n | sum_c v[i,c] * w[c,n] |."""
    L, D = v.shape
    out = []
    for i in range(L):
        tot = 0.0
        for n in range(w.shape[1]):
            tot += abs(sum(float(v[i, c]) * float(w[c, n]) for c in range(D)))
        out.append(tot)
    return np.array(out)


def test_vwo_norm_brute_and_head_slices():
    rng = np.random.default_rng(7)
    B, Hkv, rep, L, D, hidden = 1, 2, 2, 5, 4, 6
    v = rng.standard_normal((B, Hkv, L, D)).astype(np.float16)
    w = rng.standard_normal((Hkv * rep * D, hidden)).astype(np.float16)
    N = select.vwo_norms(v, w, rep)
    for h in range(Hkv * rep):
        want = _brute_vwo(v[0, h // rep], w[h * D:(h + 1) * D])
        np.testing.assert_allclose(N[0, h], want, rtol=1e-12)


def test_criticalkv_reduces_to_attention_times_value_norm():
    """rep = 1, W_O = I: the stage-2 key is the page's A_i * ||V_i||_1."""
    rng = np.random.default_rng(8)
    L, D = 40, 8
    v = rng.standard_normal((1, 1, L, D)).astype(np.float16)
    N = select.vwo_norms(v, np.eye(D, dtype=np.float16), 1)[0].astype(np.float32)   # [1, L]
    np.testing.assert_allclose(N[0], np.abs(v[0, 0].astype(np.float64)).sum(axis=1), rtol=1e-7)
    S = rng.random(L).astype(np.float32)
    key = select.criticalkv_key(S[None], N)
    np.testing.assert_array_equal(key, np.float32(S * N[0]))
    keep, W, alpha = 20, 4, 0.5
    kp, _ = select.criticalkv_select(S, S[None], N, L, keep, W, alpha)
    b1, b2 = select.criticalkv_budget(keep, W, L, alpha)
    older = list(range(L - W))
    st1 = sorted(older, key=lambda i: (-float(S[i]), i))[:b1]
    rest = [i for i in older if i not in st1]
    st2 = sorted(rest, key=lambda i: (-float(key[i]), i))[:b2]
    assert kp.tolist() == sorted(st1 + st2 + list(range(L - W, L)))


def test_criticalkv_alpha_one_is_h2o():
    rng = np.random.default_rng(9)
    L = 50
    S = rng.random(L).astype(np.float32)
    Sh = rng.random((3, L)).astype(np.float32)
    N = rng.random((3, L)).astype(np.float32)
    a, _ = select.criticalkv_select(S, Sh, N, L, 20, 5, 1.0)
    b, _ = select.h2o_select(S, L, 20, 5)
    np.testing.assert_array_equal(a, b)


def test_criticalkv_key_order_is_float32_sum():
    Sh = np.array([[1e8], [1.0], [-1e8]], np.float32)
    N = np.ones((3, 1), np.float32)
    # ((0 + 1e8) + 1) + -1e8 = 0 in float32 (1e8 + 1 rounds to 1e8); the exact sum is 1
    assert select.criticalkv_key(Sh, N)[0] == 0.0


def test_demote_victim_brute():
    rng = np.random.default_rng(10)
    for _ in range(20):
        n = int(rng.integers(2, 30))
        S = rng.integers(0, 4, size=n).astype(np.float32)
        pos = rng.permutation(100)[:n].astype(np.int32)
        L, W = 100, int(rng.integers(0, 20))
        cand = [j for j in range(n) if pos[j] < L - W]
        if not cand:
            continue
        want = min(cand, key=lambda j: (float(S[j]), -int(pos[j])))
        assert select.demote_victim(S, pos, L, W) == want
