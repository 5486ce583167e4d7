"""GPU checks of cooperative release for work stealing: raised flags stop workers homed on
released groups, the others steal the rest, and the GEMM output is complete and identical."""
import numpy as np
import pytest
import torch

import persistent_gemm_tile_gb300 as pgt
import synthetic
from gpu_helpers import dev_u16, need_gpu
from oracle import schedule as S

pytestmark = pytest.mark.gpu


@pytest.fixture()
def ctx():
    need_gpu()
    c = pgt.Context(0, max_groups=8)
    yield c
    c.set_release(np.zeros(8, np.int32))
    torch.cuda.synchronize()
    c.close()


def implied_first_tile(T, G, layout, w, P):
    """The tile a work-stealing worker of P is given at launch: ticket w div G of its home
    group w mod G (none when the group has fewer tickets)."""
    tiles = S.ws_group_tiles(T, G, layout, P)[w % G]
    return tiles[w // G: w // G + 1]


def test_schedule_log_release_from_start(ctx):
    G, P = 4, 64
    ctx.set_release([1, 1, 1, 0])  # group 0's flag is ignored
    torch.cuda.synchronize()
    grid = S.Grid(40, 13, 1)
    tb = pgt.TraceBuffers(P, grid.tiles)
    ctx.schedule_log(40, 13, 1, pgt.WORK_STEALING, 16, G, P, tb.struct)
    torch.cuda.synchronize()
    visits, _ = tb.read()
    S.check_ws_trace([[t for (t, _, _, _) in v] for v in visits], grid.tiles, G)
    for c, v in enumerate(visits):
        if c % G in (1, 2):  # released before launch: only the tile assigned at launch
            assert [t for (t, _, _, _) in v] == implied_first_tile(grid.tiles, G, S.WS_RANGES, c, P), c


@pytest.mark.parametrize("cfg", [pgt.CFG_1CTA_128x256, pgt.CFG_2CTA_256x256])
def test_gemm_release_from_start_same_bits(ctx, cfg):
    M, N, K = 2048, 2048, 1024
    A, B = synthetic.gemm_bf16_inputs(M, N, K, seed=81)
    dA, dB = dev_u16(A), dev_u16(B)
    ref = torch.empty((M, N), dtype=torch.int16, device="cuda")
    ctx.gemm_ex(pgt.make_desc(M, N, K, sched_mode=pgt.SWIZZLED, kernel_cfg=cfg), dA, dB, ref)
    ctx.set_release([0, 1, 1, 1, 1, 1, 1, 1])
    desc = pgt.make_desc(M, N, K, sched_mode=pgt.WORK_STEALING, ws_groups=8, kernel_cfg=cfg)
    plan = ctx.gemm_plan(desc)
    tb = pgt.TraceBuffers(plan["ctas"], plan["tiles"])
    C = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
    ctx.gemm_ex(desc, dA, dB, C, trace=tb.struct)
    torch.cuda.synchronize()
    assert ctx.last_error()[0] == 0
    assert torch.equal(C, ref)
    visits, _ = tb.read()
    cs = plan["cluster_size"]
    wv = [visits[w * cs] for w in range(plan["workers"])]
    assert plan["ws_groups"] == 8
    S.check_ws_trace([[t for (t, _, _, _) in v] for v in wv], plan["tiles"], 8)
    for w, v in enumerate(wv):
        if w % 8 != 0:  # released before launch: only the tile assigned at launch
            assert [t for (t, _, _, _) in v] == implied_first_tile(plan["tiles"], 8, S.WS_RANGES, w, plan["workers"]), w


def test_gemm_release_mid_launch_from_another_stream(ctx):
    M = N = K = 8192
    A, B = synthetic.gemm_bf16_inputs(M, N, K, seed=82, dist="normal")
    dA, dB = dev_u16(A), dev_u16(B)
    ref = torch.empty((M, N), dtype=torch.int16, device="cuda")
    ctx.gemm_ex(pgt.make_desc(M, N, K, sched_mode=pgt.SWIZZLED), dA, dB, ref)
    torch.cuda.synchronize()
    desc = pgt.make_desc(M, N, K, sched_mode=pgt.WORK_STEALING, ws_groups=8)
    plan = ctx.gemm_plan(desc)
    tb = pgt.TraceBuffers(plan["ctas"], plan["tiles"])
    C = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
    ctx.set_release(np.zeros(8, np.int32))  # arm the flags: launches read them from now on
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    flags = torch.ones(8, dtype=torch.int32).pin_memory()
    ctx.gemm_ex(desc, dA, dB, C, trace=tb.struct)  # current stream
    pgt.lib().pgt_set_release(ctx.handle, flags.data_ptr(), 8, side.cuda_stream)  # lands while it runs
    torch.cuda.synchronize()
    assert ctx.last_error()[0] == 0
    assert torch.equal(C, ref)
    visits, _ = tb.read()
    wv = [visits[w * plan["cluster_size"]] for w in range(plan["workers"])]
    S.check_ws_trace([[t for (t, _, _, _) in v] for v in wv], plan["tiles"], 8)
