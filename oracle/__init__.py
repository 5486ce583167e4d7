"""CPU oracle for the persistent tiled GEMM, its tile schedulers and the persistent add.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the ``persistent_gemm_tile_gb300``
package and its CUDA library) imports, links or executes anything here; only the tests,
the smoke check and the CPU-baseline leg of the benchmark do.  The oracle shares no code,
header, table or helper with the CUDA path.

Sources (three public pull-request pages on persistent tile scheduling):

* "Work Stealing Scheduler Kernel" (ROCm/tritonBLAS PR #65): per-group atomic tile
  counters, the counter-buffer sizing review, the edge-masking and small-K reviews.
* "[Feature] Introduce tile scheduler" (tile-ai/tilelang PR #2441),
  ``gemm_mxfp8_blockscaled_1d1d.py``: the cluster-interleaved wave order, the swizzled
  tile-id -> (bx, by) decode with 2-CTA pairing, the stage/parity ring, MXFP8 with one
  scale per 1 x 128 K block.
* "Implement persistent kernels" (pytorch-labs/helion PR #238): persistent_blocked and
  persistent_interleaved tile loops, the linear decode, the L2-grouping decode and the
  persistent elementwise add.

Modules:

* :mod:`oracle.numerics` - exact decoders (bf16, E4M3FN, E8M0) and fp64 -> bf16 RNE.
* :mod:`oracle.schedule` - every scheduler's tile-visit enumeration and the
  work-stealing ticket protocol (sequential model and trace validator).
* :mod:`oracle.gemm` - fp64 GEMM from exactly dequantised operands, |A|.|B| bound,
  tolerance checks.  The fp64 inner loops are in ``gemm_f64.c`` (plain C + OpenMP).
* :mod:`oracle.add` - the fp32 elementwise add.

Parity status: every function here is pinned by ``tests/test_oracle_*.py`` against
closed forms, the pages' own formulas written literally, library routines on special
cases, hand-evaluated fixtures under ``tests/golden/`` or brute force on tiny inputs.
"""
