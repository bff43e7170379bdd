"""Pins for the oracle's H2O importance scores (no GPU).

Definition (plainest reading of H2O, named by the MiKV notes "Observation 1-4"
and "Key contributions, 1)"): prompt token i's score is the sum over query rows
t >= i of the causal softmax probability of i in row t, summed over the query
heads of the key head; each decode step adds that step's probabilities.
"""
import math

import numpy as np

from oracle import scores


def _brute(qh, k):
    """Python loops and math.exp, independent of the numpy formulation."""
    T, D = qh.shape
    S = [0.0] * T
    for t in range(T):
        logits = [sum(float(qh[t, c]) * float(k[i, c]) for c in range(D)) / math.sqrt(D)
                  for i in range(t + 1)]
        m = max(logits)
        e = [math.exp(l - m) for l in logits]
        z = sum(e)
        for i in range(t + 1):
            S[i] += e[i] / z
    return np.array(S)


def test_matches_brute_force_tiny():
    rng = np.random.default_rng(0)
    for T, D in [(1, 4), (5, 4), (9, 8), (13, 16)]:
        q = (rng.standard_normal((T, D)) * 3).astype(np.float16)
        k = (rng.standard_normal((T, D)) * 3).astype(np.float16)
        np.testing.assert_allclose(scores.prefill_column_scores(q, k), _brute(q, k), rtol=1e-12, atol=1e-12)


def test_mass_conservation_and_causality():
    """Each causal row sums to 1: sum_i S_i = rep*T.  Row 0 sees only key 0, so a
    change of the last key moves only the last column's score and the totals."""
    rng = np.random.default_rng(1)
    B, Hq, Hkv, T, D = 2, 4, 2, 64, 32
    q = rng.standard_normal((B, Hq, T, D)).astype(np.float16)
    k = rng.standard_normal((B, Hkv, T, D)).astype(np.float16)
    s_head, s = scores.prefill_scores(q, k)
    np.testing.assert_allclose(s_head.sum(axis=2), T, rtol=1e-12)
    np.testing.assert_allclose(s.sum(axis=2), 2 * T, rtol=1e-12)
    np.testing.assert_allclose(s, s_head.reshape(B, Hkv, 2, T).sum(axis=2), rtol=1e-14)
    # S_0 >= P(row 0) = 1 for every head; the last token only gets row T-1's mass
    assert (s_head[:, :, 0] >= 1 - 1e-12).all()
    assert (s_head[:, :, -1] <= 1 + 1e-12).all()


def test_uniform_logits():
    """q = 0: every row is uniform over its prefix, S_i = sum_{t>=i} 1/(t+1) (harmonic tail)."""
    T = 10
    q = np.zeros((T, 8), np.float16)
    k = np.random.default_rng(2).standard_normal((T, 8)).astype(np.float16)
    want = np.array([sum(1.0 / (t + 1) for t in range(i, T)) for i in range(T)])
    np.testing.assert_allclose(scores.prefill_column_scores(q, k), want, rtol=1e-13)


def test_sampled_columns_match_full():
    rng = np.random.default_rng(3)
    T, D = 200, 64
    q = (rng.standard_normal((T, D)) * 2).astype(np.float16)
    k = (rng.standard_normal((T, D)) * 2).astype(np.float16)
    full = scores.prefill_column_scores(q, k)
    cols = [0, 17, 150, 199]
    np.testing.assert_allclose(scores.column_scores_at(q, k, cols), full[cols], rtol=1e-11)
    rows = [0, 5, 199]
    lse = scores.row_lse(q, k, rows)
    for j, t in enumerate(rows):
        l = np.array([float(q[t].astype(np.float64) @ k[i].astype(np.float64)) for i in range(t + 1)]) / np.sqrt(D)
        assert abs(lse[j] - math.log(sum(math.exp(x) for x in l))) < 1e-10


def test_decode_update_brute():
    rng = np.random.default_rng(4)
    s = rng.random(7)
    logits = rng.standard_normal((3, 7))
    lse = rng.standard_normal(3)
    got = scores.decode_score_update(s, logits, lse)
    for j in range(7):
        want = s[j] + sum(math.exp(logits[h, j] - lse[h]) for h in range(3))
        assert abs(got[j] - want) < 1e-12
