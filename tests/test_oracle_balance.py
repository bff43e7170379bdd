"""Pins for the oracle's channel balancer (no GPU).

Definition: MiKV reading notes (velog), "Key contributions, 2) Outlier-aware
handling" - b_c = sqrt(max|q_c| / max|k_c|) over the prompt; keys are scaled
by b before quantisation and queries divided by b.
"""
import os

import numpy as np
import pytest
import sympy

from conftest import GOLDEN
from oracle import balance


def _nearest_f32(expr: str) -> np.float32:
    """float32 nearest to a real expression like 'sqrt(0.75)', chosen by exact comparison."""
    if expr.startswith("sqrt("):
        val = sympy.sqrt(sympy.Rational(expr[5:-1]))
    else:
        val = sympy.Rational(expr)
    f = np.float32(float(val.evalf(60)))
    cands = [np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))]
    return min(cands, key=lambda c: abs(sympy.Rational(float(c)) - val))


def _load_cases():
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "balancer_hand.txt")) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("case"):
                cur = dict(q={}, k={}, b=None)
                cases.append(cur)
            elif line.startswith("q "):
                head, rest = line[2:].split(":")
                h, t = map(int, head.split())
                cur["q"][(h, t)] = [float(x) for x in rest.split()]
            elif line.startswith("k "):
                t, rest = line[2:].split(":")
                cur["k"][int(t)] = [float(x) for x in rest.split()]
            elif line.startswith("b:"):
                cur["b"] = [_nearest_f32(x) for x in line[2:].split()]
    return cases


@pytest.mark.parametrize("case", _load_cases())
def test_hand_cases(case):
    heads = 1 + max(h for h, _ in case["q"])
    T = 1 + max(t for _, t in case["q"])
    D = len(case["b"])
    q = np.zeros((1, heads, T, D), np.float16)
    for (h, t), vals in case["q"].items():
        q[0, h, t] = vals
    k = np.zeros((1, 1, T, D), np.float16)
    for t, vals in case["k"].items():
        k[0, 0, t] = vals
    b = balance.channel_balancer(q, k)
    assert b.dtype == np.float32
    np.testing.assert_array_equal(b[0, 0], np.array(case["b"], np.float32))


def test_balanced_dot_product_identity():
    """(q/b).(k*b) == q.k in exact arithmetic; float64 check to 1e-12 relative."""
    rng = np.random.default_rng(1)
    B, Hq, Hkv, T, D = 2, 4, 2, 16, 128
    q = (rng.standard_normal((B, Hq, T, D)) * rng.choice([1, 16], size=(1, Hq, 1, D))).astype(np.float16)
    k = (rng.standard_normal((B, Hkv, T, D)) * rng.choice([1, 16], size=(1, Hkv, 1, D))).astype(np.float16)
    b = balance.channel_balancer(q, k).astype(np.float64)
    rep = Hq // Hkv
    for bi in range(B):
        for h in range(Hq):
            g = h // rep
            qf, kf = q[bi, h].astype(np.float64), k[bi, g].astype(np.float64)
            lhs = (qf / b[bi, g]) @ (kf * b[bi, g]).T
            rhs = qf @ kf.T
            np.testing.assert_allclose(lhs, rhs, rtol=1e-12, atol=1e-12 * np.abs(rhs).max())


def test_balanced_maxima_are_equal():
    """After balancing, max|q/b| == max|k*b| per channel (both equal sqrt(Mq*Mk))."""
    rng = np.random.default_rng(2)
    q = (rng.standard_normal((1, 2, 64, 128)) * 8).astype(np.float16)
    k = rng.standard_normal((1, 1, 64, 128)).astype(np.float16)
    b = balance.channel_balancer(q, k)[0, 0].astype(np.float64)
    mq = np.abs(q[0].astype(np.float64)).max(axis=(0, 1))
    mk = np.abs(k[0, 0].astype(np.float64)).max(axis=0)
    np.testing.assert_allclose(mq / b, mk * b, rtol=1e-6)


def test_per_batch_and_per_key_head():
    """b is indexed by batch row and key head: changing one sequence leaves the others alone."""
    rng = np.random.default_rng(3)
    q = rng.standard_normal((2, 4, 8, 128)).astype(np.float16)
    k = rng.standard_normal((2, 2, 8, 128)).astype(np.float16)
    b0 = balance.channel_balancer(q, k)
    q2 = q.copy()
    q2[1, 3, 0, 5] = 100.0          # batch row 1, query head 3 -> key head 1
    b1 = balance.channel_balancer(q2, k)
    changed = np.argwhere(b0 != b1)
    assert changed.tolist() == [[1, 1, 5]]
