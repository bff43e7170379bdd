"""Plain CPU oracle of the MiKV mixed-precision KV-cache hot path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product (the CUDA library and its
Python binding) imports, links or executes this package; only the tests, the
package's ``smoke()`` check and the bench's CPU-baseline leg do.  It shares no
code, header, table or helper with the CUDA path: both sides only receive the
same seeded inputs.

Every function restates a definition from the pages it cites and is written to
be checked by eye, not to be fast:

* floating-point results that are compared with a tolerance (attention,
  importance scores, V.W_O norms) are computed in float64;
* where a float decides an integer (quantisation codes, top-k selection) the
  decision is taken in float32 with the operation order stated in the
  function, the precision the kernels use;
* a library routine (numpy matmul, sort, sqrt) may serve as one step; there is
  no blocking, fusion or reordering beyond the definition.

Modules
-------
balance    channel balancer b = sqrt(max|q| / max|k|) (MiKV notes, "Outlier-aware")
quant      per-token asymmetric group quantizer, bit packing
scores     H2O accumulated attention (prefill column sums, decode update)
select     H2O top-k with recent window, CriticalKV two-stage, demotion victim
attention  decode attention over the two-tier cache (float64); post-attention top-k ("oracle eviction")
perturbation  the step after attention: o . W_O and the CriticalKV per-head perturbation
channel_quant  per-channel key quantisation with pending-token buffering (Appendix C alternative)
pipeline   prefill + decode steps composed into one cache, the whole path

Parity pins for every function live in ``tests/test_oracle_*.py``.
"""
from . import attention, balance, pipeline, quant, scores, select  # noqa: F401
