"""Edge cases on the GPU: degenerate GEMM shapes, very large tile counts, long K, and
work-stealing counters under heavy contention; all against the CPU oracle."""
import numpy as np
import pytest
import torch

import persistent_gemm_tile_gb300 as pgt
import synthetic
from gpu_helpers import dev_u16, host_u16, need_gpu
from oracle import gemm as OG
from oracle import schedule as S

pytestmark = pytest.mark.gpu

CFGS = [pgt.CFG_1CTA_128x128, pgt.CFG_1CTA_128x256, pgt.CFG_2CTA_256x128, pgt.CFG_2CTA_256x256]


@pytest.fixture(scope="module")
def ctx():
    need_gpu()
    c = pgt.Context(0, max_groups=16)
    yield c
    c.close()


def run(ctx, A, B, M, N, K, **kw):
    desc = pgt.make_desc(M, N, K, **kw)
    C = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
    ctx.gemm_ex(desc, dev_u16(A), dev_u16(B), C)
    torch.cuda.synchronize()
    assert ctx.last_error()[0] == 0
    return host_u16(C)


@pytest.mark.parametrize("cfg", CFGS)
@pytest.mark.parametrize("M,N,K", [(1, 8, 8), (1, 8, 1000), (129, 72, 40), (257, 8, 64), (3, 264, 129)])
@pytest.mark.parametrize("mode", [pgt.SWIZZLED, pgt.WORK_STEALING, pgt.BLOCKED_GROUPED_M, pgt.LAUNCH_CONTROL])
def test_tiny_and_odd_shapes(ctx, cfg, M, N, K, mode):
    lda = -(-K // 8) * 8
    A, B = synthetic.gemm_bf16_inputs(M, N, K, seed=101, lda=lda)
    c = run(ctx, A, B, M, N, K, lda=lda, kernel_cfg=cfg, sched_mode=mode, group_size=3)
    C64, Abs = OG.gemm_full(OG.dequant_bf16(A), OG.dequant_bf16(B), True, M, N, K)
    OG.check(c, C64, Abs)


@pytest.mark.parametrize("mode", [pgt.BLOCKED, pgt.SWIZZLED, pgt.WORK_STEALING, pgt.LAUNCH_CONTROL])
def test_many_tiles_tall_skinny(ctx, mode):
    # 1M rows x 64 columns: 8192 tiles of 128 rows (4096 for a pair), K = 64
    M, N, K = 1 << 20, 64, 64
    A, B = synthetic.gemm_bf16_inputs(M, N, K, seed=102)
    c = run(ctx, A, B, M, N, K, kernel_cfg=pgt.CFG_2CTA_256x128, sched_mode=mode, group_size=16)
    C64, Abs = OG.gemm_full(OG.dequant_bf16(A), OG.dequant_bf16(B), True, M, N, K)
    OG.check(c, C64, Abs)


def test_long_k(ctx):
    M, N, K = 256, 512, 65536  # 1024 k-iterations: the stage ring wraps many times
    A, B = synthetic.gemm_bf16_inputs(M, N, K, seed=103, dist="normal")
    c1 = run(ctx, A, B, M, N, K, sched_mode=pgt.SWIZZLED)
    c2 = run(ctx, A, B, M, N, K, sched_mode=pgt.WORK_STEALING, kernel_cfg=pgt.CFG_2CTA_256x256)
    assert np.array_equal(c1, c2)
    C64, Abs = OG.gemm_full(OG.dequant_bf16(A), OG.dequant_bf16(B), True, M, N, K)
    OG.check(c1, C64, Abs)


@pytest.mark.parametrize("G_ws", [1, 8, 16])
def test_work_stealing_contention_100k_tiles(ctx, G_ws):
    mb, nb, P = 400, 250, 64  # 100,000 tiles
    grid = S.Grid(mb, nb, 1)
    for _ in range(2):  # the second launch depends on the in-kernel reset
        tb = pgt.TraceBuffers(P, grid.tiles)
        ctx.schedule_log(mb, nb, 1, pgt.WORK_STEALING, 16, G_ws, P, tb.struct)
        torch.cuda.synchronize()
        visits, _ = tb.read()
        S.check_ws_trace([[t for (t, _, _, _) in v] for v in visits], grid.tiles, G_ws)
        del tb
