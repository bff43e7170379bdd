"""Pins for the oracle's step after attention (no GPU): the output projection o . W_O and
the per-head perturbation ||(o - o^) W_O^(h)||_1 (CriticalKV summary, gist.science,
"Theoretical framework": L = ||o - o^||_1 with value states projected by W_O)."""
from pathlib import Path

import numpy as np
import pytest

from oracle import perturbation as pt

GOLDEN = Path(__file__).parent / "golden" / "perturbation_hand.txt"


def _golden():
    rows = {}
    for line in GOLDEN.read_text().splitlines():
        if not line.strip() or line.startswith("#"):
            continue
        key, *parts = [p.strip() for p in line.split("|")]
        rows[key] = [np.array([float(x) for x in p.split()]) for p in parts]
    return rows


def test_hand_derived_case():
    g = _golden()
    o = np.stack(g["o"])[None]            # [1][2][2]
    oh = np.stack(g["o_hat"])[None]
    w = np.stack([g[f"w{i}"][0] for i in range(4)])
    np.testing.assert_array_equal(pt.head_perturbation(o, oh, w)[0], g["L"][0])
    np.testing.assert_array_equal(pt.head_perturbation(o, oh)[0], g["L_raw"][0])
    np.testing.assert_array_equal(pt.output_projection(o, w)[0], g["y"][0])


@pytest.mark.parametrize("seed", range(3))
def test_identical_outputs_have_zero_perturbation(seed):
    rng = np.random.default_rng(seed)
    o = rng.standard_normal((3, 4, 8))
    w = rng.standard_normal((32, 24))
    assert np.all(pt.head_perturbation(o, o.copy(), w) == 0.0)
    assert np.all(pt.head_perturbation(o, o.copy()) == 0.0)


def test_identity_projection_reduces_to_the_unprojected_distance():
    rng = np.random.default_rng(4)
    B, Hq, D = 2, 3, 5
    o, oh = rng.standard_normal((B, Hq, D)), rng.standard_normal((B, Hq, D))
    eye = np.eye(Hq * D)
    np.testing.assert_allclose(pt.head_perturbation(o, oh, eye), np.abs(o - oh).sum(axis=2), rtol=1e-15)
    np.testing.assert_allclose(pt.output_projection(o, eye), o.reshape(B, Hq * D), rtol=1e-15)


def test_brute_force_sums():
    rng = np.random.default_rng(5)
    B, Hq, D, hidden = 2, 3, 4, 5
    o, oh = rng.standard_normal((B, Hq, D)), rng.standard_normal((B, Hq, D))
    w = rng.standard_normal((Hq * D, hidden))
    L = pt.head_perturbation(o, oh, w)
    y = pt.output_projection(o, w)
    for b in range(B):
        for c in range(hidden):
            assert y[b, c] == pytest.approx(sum(o[b, h, k] * w[h * D + k, c] for h in range(Hq) for k in range(D)),
                                            rel=1e-12)
        for h in range(Hq):
            want = sum(abs(sum((o[b, h, k] - oh[b, h, k]) * w[h * D + k, c] for k in range(D)))
                       for c in range(hidden))
            assert L[b, h] == pytest.approx(want, rel=1e-12)


def test_properties():
    rng = np.random.default_rng(6)
    B, Hq, D, hidden = 2, 4, 6, 7
    o, oh = rng.standard_normal((B, Hq, D)), rng.standard_normal((B, Hq, D))
    w = rng.standard_normal((Hq * D, hidden))
    L = pt.head_perturbation(o, oh, w)
    # symmetric, absolutely homogeneous in the difference
    np.testing.assert_allclose(pt.head_perturbation(oh, o, w), L, rtol=1e-14)
    np.testing.assert_allclose(pt.head_perturbation(o, o + (-2.5) * (oh - o), w), 2.5 * L, rtol=1e-12)
    # the hidden-state perturbation is bounded by the sum of the per-head ones (triangle inequality)
    dy = np.abs(pt.output_projection(o, w) - pt.output_projection(oh, w)).sum(axis=1)
    assert np.all(dy <= L.sum(axis=1) * (1 + 1e-12))
    # the projection is linear
    np.testing.assert_allclose(pt.output_projection(o + oh, w), pt.output_projection(o, w) + pt.output_projection(oh, w),
                               rtol=1e-12, atol=1e-12)
