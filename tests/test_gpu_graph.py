"""GEMM, add and multi-loop launches captured in a CUDA graph replay with the same results
as eager launches (work stealing included: its counters reset in-kernel between replays)."""
import numpy as np
import pytest
import torch

import persistent_gemm_tile_gb300 as pgt
import synthetic
from gpu_helpers import dev_u16, need_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode", [pgt.SWIZZLED, pgt.WORK_STEALING, pgt.LAUNCH_CONTROL])
def test_gemm_graph_replay_matches_eager(mode):
    need_gpu()
    ctx = pgt.Context(0)
    M, N, K = 1024, 1536, 512
    A, B = synthetic.gemm_bf16_inputs(M, N, K, seed=121)
    dA, dB = dev_u16(A), dev_u16(B)
    d = pgt.make_desc(M, N, K, sched_mode=mode)
    ref = torch.empty((M, N), dtype=torch.int16, device="cuda")
    ctx.gemm_ex(d, dA, dB, ref)  # eager first: also does the per-device set-up
    torch.cuda.synchronize()
    outs = [torch.zeros((M, N), dtype=torch.int16, device="cuda") for _ in range(3)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for o in outs:
            ctx.gemm_ex(d, dA, dB, o)
    for _ in range(3):
        for o in outs:
            o.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert ctx.last_error()[0] == 0
        for o in outs:
            assert torch.equal(o, ref)
    ctx.close()


def test_add_graph_replay():
    need_gpu()
    ctx = pgt.Context(0)
    x, y = synthetic.add_inputs(1000, 1024, seed=122)
    tx, ty = torch.from_numpy(x).cuda(), torch.from_numpy(y).cuda()
    out = torch.empty_like(tx)
    ctx.add(tx, ty, out)
    torch.cuda.synchronize()
    ref = out.clone()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ctx.add(tx, ty, out)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    ctx.close()
