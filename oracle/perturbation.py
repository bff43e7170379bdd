"""The step after attention (oracle, float64): the output projection o . W_O and the
CriticalKV output-perturbation diagnostic.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources:
* CriticalKV summary (gist.science, arXiv 2502.03805), "Theoretical framework": replacing
  the full KV cache by a subset perturbs the attention output; the perturbation is the L1
  distance between the output over the full cache, o, and the output over the subset, o^:
  L = ||o - o^||_1.  The bound derived for it depends on the attention weights and on the
  value states projected by the output projection W_O (V W_O).
* Same page, "Experimental results", perturbation analysis: the perturbation is reported
  per attention head and for the last layer's hidden state.

Readings (the page gives no formula beyond L = ||o - o^||_1):
* Head h reaches the hidden state through its block of the output projection,
  W_O^(h) = W_O[h*D:(h+1)*D, :] (W_O is [Hq*D][hidden], y = o_flat . W_O), so the head's
  perturbation is L_h = || (o_h - o^_h) . W_O^(h) ||_1 over the hidden dimension; with no
  W_O it is || o_h - o^_h ||_1 over the head dimension D.
* The attention block's output is y = sum_h o_h . W_O^(h) = o_flat . W_O.
* o^ is the output of whatever replaces the full cache (the mixed-precision cache, or the
  kept subset of an eviction policy); both outputs are inputs here.
"""
import numpy as np


def output_projection(o: np.ndarray, w_o: np.ndarray) -> np.ndarray:
    """y[b] = sum_h o[b, h] . W_O[h*D:(h+1)*D, :] = o[b] flattened . W_O.

    o [B][Hq][D], w_o [Hq*D][hidden] -> y [B][hidden], float64."""
    B, Hq, D = o.shape
    assert w_o.shape[0] == Hq * D
    return o.reshape(B, Hq * D).astype(np.float64) @ w_o.astype(np.float64)


def head_perturbation(o: np.ndarray, o_hat: np.ndarray, w_o: np.ndarray | None = None) -> np.ndarray:
    """L[b, h] = || (o[b, h] - o_hat[b, h]) . W_O[h*D:(h+1)*D, :] ||_1, or || o - o_hat ||_1
    over D when w_o is None.  o, o_hat [B][Hq][D] -> L [B][Hq], float64."""
    d = o.astype(np.float64) - o_hat.astype(np.float64)
    B, Hq, D = d.shape
    if w_o is None:
        return np.abs(d).sum(axis=2)
    assert w_o.shape[0] == Hq * D
    w = w_o.astype(np.float64)
    out = np.empty((B, Hq))
    for h in range(Hq):
        z = d[:, h, :] @ w[h * D:(h + 1) * D, :]      # [B][hidden]
        out[:, h] = np.abs(z).sum(axis=1)
    return out
