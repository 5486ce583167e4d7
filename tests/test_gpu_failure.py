"""Failure detection on the GPU without a fault: a bounded wait that nothing completes runs
out, the kernel records PGT_ERR_TIMEOUT and returns, the host reads the status, and the
context stays usable for the next launch."""
import time

import numpy as np
import pytest
import torch

import persistent_gemm_tile_gb300 as pgt
import synthetic
from gpu_helpers import dev_u16, need_gpu

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    need_gpu()
    ctx = pgt.Context(0)
    ctx.wait_probe(arrive=True)
    assert ctx.last_error()[0] == pgt.OK
    t0 = time.perf_counter()
    ctx.wait_probe(arrive=False)  # nothing ever arrives
    rc, detail = ctx.last_error()
    waited = time.perf_counter() - t0
    assert rc == pgt.ERR_TIMEOUT
    assert detail == [1, 3, 0, 12]  # code, role (scheduler), block, wait site
    assert 0.5 < waited < 30.0
    assert ctx.last_error()[0] == pgt.OK  # read and cleared
    # the context and the GPU keep working: a GEMM and the work-stealing counters are fine
    M = N = K = 512
    A, B = synthetic.gemm_bf16_inputs(M, N, K, seed=111)
    ref = torch.empty((M, N), dtype=torch.int16, device="cuda")
    C = torch.empty((M, N), dtype=torch.int16, device="cuda")
    ctx.gemm_ex(pgt.make_desc(M, N, K, sched_mode=pgt.SWIZZLED), dev_u16(A), dev_u16(B), ref)
    ctx.gemm_ex(pgt.make_desc(M, N, K, sched_mode=pgt.WORK_STEALING), dev_u16(A), dev_u16(B), C)
    torch.cuda.synchronize()
    assert ctx.last_error()[0] == pgt.OK
    assert torch.equal(C, ref)
    ctx.close()
