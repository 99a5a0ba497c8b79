"""CPU oracle for direct-access tiered-memory decode (DAK-style). TEST INFRASTRUCTURE ONLY.

Plain, slow, fp64 reference implementations of what the direct-access path computes.
Only the tests, the smoke check and the benchmark's CPU-baseline leg may import this
package; the product library never does, and this package imports nothing from it.

Sources (cited by page title and section):
* [DAK] "DAK: Direct-Access-Enabled GPU Memory Offloading with Optimal Efficiency for
  LLM Inference" (arXiv 2604.26074v1) -- the authority on what is computed.
* [DAK-explainer] "DAK 完全拆解：绕过 HBM 预取，用 TMA 直连远端内存" -- a blog post that
  restates the paper's performance model with clean formulas.

Modules:
* ``bf16``       -- bf16 decode / round-to-nearest-even (the oracle's own copy).
* ``gemm``       -- C = A.B over a tile-row partitioned A ([DAK] section 4.1).
* ``attention``  -- single-query GQA scaled dot-product attention ([DAK] section 5).
* ``placement``  -- tile rows / requests per tier, global offload ratio, host-link traffic.
* ``planner``    -- the per-operation offload optimisation problem ([DAK] section 4.2,
  Appendix A eq. (1)) solved by exhaustive search.
* ``decoder``    -- one decode step of a Llama-shaped transformer around those two
  operations ([DAK] sections 3, 5 and 6.1).

Parity status of each function is stated in its module docstring; none is unpinned.
"""
from . import bf16, gemm, attention, placement, planner, decoder  # noqa: F401
