"""Tile-ring stress on the GPU: many one-stage tiles per worker and few workers, so the
scheduler thread posts far ahead and the four-entry tile ring wraps dozens of times per
worker, in both CTAs of a pair.  Every order and configuration against the CPU oracle, the
orders bit-identical to each other, and every visit log valid for its order."""
import numpy as np
import pytest
import torch

import persistent_gemm_tile_gb300 as pgt
import synthetic
from gpu_helpers import dev_u8, dev_u16, host_u16, need_gpu
from oracle import gemm as OG
from oracle import schedule as S

pytestmark = pytest.mark.gpu

M, N = 1 << 16, 512
ORDERS = [(pgt.SWIZZLED, 0), (pgt.BLOCKED, 0), (pgt.INTERLEAVED, 0), (pgt.BLOCKED_GROUPED_M, 0),
          (pgt.WORK_STEALING, pgt.WS_RANGES), (pgt.WORK_STEALING, pgt.WS_STRIPED), (pgt.LAUNCH_CONTROL, 0)]
WORKERS = 6


@pytest.fixture(scope="module")
def ctx():
    need_gpu()
    c = pgt.Context(0, max_groups=16)
    yield c
    c.close()


@pytest.fixture(scope="module")
def bf16_case():
    K = 64  # one stage per tile
    A, B = synthetic.gemm_bf16_inputs(M, N, K, seed=211, dist="normal")
    C64, Abs = OG.gemm_full(OG.dequant_bf16(A), OG.dequant_bf16(B), True, M, N, K)
    return K, dev_u16(A), dev_u16(B), C64, Abs


@pytest.fixture(scope="module")
def mx_case():
    K = 128  # one stage per tile
    qa, sa, qb, sb = synthetic.gemm_mxfp8_inputs(M, N, K, seed=212)
    C64, Abs = OG.gemm_full(OG.dequant_mxfp8(qa, sa), OG.dequant_mxfp8(qb, sb), False, M, N, K)
    return K, [dev_u8(x) for x in (qa, qb, sa, sb)], C64, Abs


def check_visits(plan, tb, mode, layout):
    visits, _ = tb.read()
    cs = plan["cluster_size"]
    grid = S.Grid(plan["m_blocks"], plan["n_blocks"], cs)
    tmn = [[(t, m, n) for (t, m, n, _) in v] for v in visits]
    # both CTAs of a pair see the same entries of the ring
    for w in range(plan["workers"]):
        for r in range(1, cs):
            assert tmn[w * cs + r] == tmn[w * cs], (w, r)
    wv = [tmn[w * cs] for w in range(plan["workers"])]
    if mode == pgt.WORK_STEALING:
        S.check_ws_trace([[t for (t, _, _) in v] for v in wv], grid.tiles, plan["ws_groups"], layout)
    else:
        want = S.static_schedule(mode, grid, plan["workers"], 16)
        assert wv == [[(t, m, n) for (_, t, m, n) in v] for v in want]
    # the ring wrapped many times for the busiest worker
    assert max(len(v) for v in wv) >= 4 * 8


@pytest.mark.parametrize("cfg", [pgt.CFG_2CTA_256x256, pgt.CFG_2CTA_256x128, pgt.CFG_1CTA_128x128])
def test_bf16_one_stage_tiles_every_order(ctx, bf16_case, cfg):
    K, tA, tB, C64, Abs = bf16_case
    ref = None
    for mode, layout in ORDERS:
        workers = 0 if mode == pgt.LAUNCH_CONTROL else WORKERS
        desc = pgt.make_desc(M, N, K, sched_mode=mode, group_size=16, ws_groups=4, ws_layout=layout,
                             kernel_cfg=cfg, num_workers=workers)
        plan = ctx.gemm_plan(desc)
        tb = pgt.TraceBuffers(plan["ctas"], plan["tiles"])
        C = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
        ctx.gemm_ex(desc, tA, tB, C, trace=tb.struct)
        torch.cuda.synchronize()
        rc, detail = ctx.last_error()
        assert rc == 0, (mode, layout, detail)
        c = host_u16(C)
        if ref is None:
            OG.check(c, C64, Abs)
            ref = c
        else:
            assert np.array_equal(c, ref), (mode, layout)
        if mode != pgt.LAUNCH_CONTROL:
            check_visits(plan, tb, mode, layout)


@pytest.mark.parametrize("cfg", [pgt.CFG_2CTA_256x256, pgt.CFG_2CTA_256x224, pgt.CFG_1CTA_128x256])
def test_mxfp8_one_stage_tiles_every_order(ctx, mx_case, cfg):
    K, (qa, qb, sa, sb), C64, Abs = mx_case
    ref = None
    for mode, layout in ORDERS:
        workers = 0 if mode == pgt.LAUNCH_CONTROL else WORKERS
        desc = pgt.make_desc(M, N, K, dtype=pgt.MXFP8, b_layout=pgt.B_NK, sched_mode=mode, group_size=16,
                             ws_groups=4, ws_layout=layout, kernel_cfg=cfg, num_workers=workers)
        plan = ctx.gemm_plan(desc)
        ws = torch.zeros(max(ctx.gemm_workspace_bytes(desc), 16), dtype=torch.uint8, device="cuda")
        tb = pgt.TraceBuffers(plan["ctas"], plan["tiles"])
        C = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
        ctx.gemm_ex(desc, qa, qb, C, sfa=sa, sfb=sb, workspace=ws, trace=tb.struct)
        torch.cuda.synchronize()
        rc, detail = ctx.last_error()
        assert rc == 0, (mode, layout, detail)
        c = host_u16(C)
        if ref is None:
            OG.check(c, C64, Abs)
            ref = c
        else:
            assert np.array_equal(c, ref), (mode, layout)
        if mode != pgt.LAUNCH_CONTROL:
            check_visits(plan, tb, mode, layout)
