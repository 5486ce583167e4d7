"""GPU checks of the hardware launch-control scheduler (Blackwell cluster launch control):
one worker per tile, running workers cancel workers not yet started and take their tiles.
The visit logs must satisfy oracle.schedule.check_launch_control_trace; GEMM outputs must
be bit-identical to the static schedulers' for the same kernel configuration."""
import numpy as np
import pytest
import torch

import persistent_gemm_tile_gb300 as pgt
import synthetic
from gpu_helpers import dev_u16, host_u16, need_gpu
from oracle import gemm as OG
from oracle import schedule as S

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    need_gpu()
    c = pgt.Context(0)
    yield c
    c.close()


@pytest.mark.parametrize("mb,nb,cs", [(1, 1, 1), (3, 5, 1), (40, 13, 1), (64, 64, 2), (200, 100, 1)])
@pytest.mark.parametrize("G", [1, 16])
def test_schedule_log_launch_control(ctx, mb, nb, cs, G):
    grid = S.Grid(mb, nb, cs)
    T = grid.tiles
    tb = pgt.TraceBuffers(T, T)
    ctx.schedule_log(mb, nb, cs, pgt.LAUNCH_CONTROL, G, 1, T, tb.struct)
    torch.cuda.synchronize()
    assert ctx.last_error()[0] == 0
    visits, _ = tb.read()
    S.check_launch_control_trace([[t for (t, _, _, _) in v] for v in visits], T)
    for v in visits:
        for (t, m, n, _) in v:
            assert (m, n) == S.decode(S.LAUNCH_CONTROL, t, grid, G)


@pytest.mark.parametrize("cfg", [pgt.CFG_1CTA_128x128, pgt.CFG_1CTA_128x256, pgt.CFG_2CTA_256x128,
                                 pgt.CFG_2CTA_256x256])
def test_gemm_launch_control_matches_static(ctx, cfg):
    M, N, K = 2000, 2048, 512
    A, B = synthetic.gemm_bf16_inputs(M, N, K, seed=91)
    dA, dB = dev_u16(A), dev_u16(B)
    ref = torch.empty((M, N), dtype=torch.int16, device="cuda")
    ctx.gemm_ex(pgt.make_desc(M, N, K, sched_mode=pgt.SWIZZLED, group_size=4, kernel_cfg=cfg), dA, dB, ref)
    desc = pgt.make_desc(M, N, K, sched_mode=pgt.LAUNCH_CONTROL, group_size=4, kernel_cfg=cfg)
    plan = ctx.gemm_plan(desc)
    assert plan["workers"] == plan["tiles"]
    tb = pgt.TraceBuffers(plan["ctas"], plan["tiles"])
    C = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
    ctx.gemm_ex(desc, dA, dB, C, trace=tb.struct)
    torch.cuda.synchronize()
    assert ctx.last_error()[0] == 0
    assert torch.equal(C, ref)
    visits, _ = tb.read()
    cs = plan["cluster_size"]
    wv = []
    for w in range(plan["workers"]):
        lists = [[t for (t, _, _, _) in v] for v in visits[w * cs:(w + 1) * cs]]
        assert all(x == lists[0] for x in lists[1:])
        wv.append(lists[0])
    S.check_launch_control_trace(wv, plan["tiles"])
    C64, Abs = OG.gemm_full(OG.dequant_bf16(A), OG.dequant_bf16(B), True, M, N, K)
    OG.check(host_u16(C), C64, Abs)


def test_gemm_8192_launch_control_same_bits(ctx):
    M = N = K = 8192
    A, B = synthetic.gemm_bf16_inputs(M, N, K, seed=2, dist="normal")
    dA, dB = dev_u16(A), dev_u16(B)
    ref = torch.empty((M, N), dtype=torch.int16, device="cuda")
    C = torch.empty((M, N), dtype=torch.int16, device="cuda")
    ctx.gemm_ex(pgt.make_desc(M, N, K, sched_mode=pgt.SWIZZLED, group_size=16), dA, dB, ref)
    ctx.gemm_ex(pgt.make_desc(M, N, K, sched_mode=pgt.LAUNCH_CONTROL, group_size=16), dA, dB, C)
    torch.cuda.synchronize()
    assert ctx.last_error()[0] == 0
    assert torch.equal(C, ref)


def test_launch_control_rejects_worker_count(ctx):
    t = torch.zeros((256, 256), dtype=torch.int16, device="cuda")
    with pytest.raises(pgt.PgtError):
        ctx.gemm_ex(pgt.make_desc(256, 256, 256, sched_mode=pgt.LAUNCH_CONTROL, num_workers=3), t, t, t)
