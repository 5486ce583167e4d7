"""GPU parity for work stealing with striped tile ownership (PGT_WS_STRIPED: counter group g
owns the tiles t = g mod G) against oracle.schedule: the protocol's invariants on
schedule logs and traced GEMMs, the in-kernel counter reset, release, GEMM outputs
bit-identical to the static schedule, and the argument check."""
import pytest
import torch

import persistent_gemm_tile_gb300 as pgt
import synthetic
from gpu_helpers import dev_u16, need_gpu
from oracle import schedule as S

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    need_gpu()
    c = pgt.Context(0, max_groups=16)
    yield c
    c.close()


def log(ctx, mb, nb, cs, G, G_ws, P):
    grid = S.Grid(mb, nb, cs)
    tb = pgt.TraceBuffers(P, max(grid.tiles, 1))
    ctx.schedule_log(mb, nb, cs, pgt.WORK_STEALING, G, G_ws, P, tb.struct, ws_layout=pgt.WS_STRIPED)
    torch.cuda.synchronize()
    visits, _ = tb.read()
    return grid, visits


@pytest.mark.parametrize("mb,nb,cs", [(1, 1, 1), (3, 5, 1), (7, 4, 2), (19, 32, 1), (64, 64, 2), (40, 13, 1)])
@pytest.mark.parametrize("P,G_ws", [(1, 1), (4, 2), (152, 8), (152, 16), (300, 8), (7, 3)])
def test_schedule_log_invariants(ctx, mb, nb, cs, P, G_ws):
    for _ in range(2):  # the second launch relies on the in-kernel counter reset
        grid, visits = log(ctx, mb, nb, cs, 16, G_ws, P)
        S.check_ws_trace([[t for (t, _, _, _) in v] for v in visits], grid.tiles, G_ws, S.WS_STRIPED)
        for v in visits:
            for (t, m, n, _) in v:
                assert (m, n) == S.decode(S.WORK_STEALING, t, grid, 16)


def test_first_tiles_are_the_static_first_wave(ctx):
    # every worker's first tile is taken from its home group before any group runs dry:
    # with P a multiple of G_ws and T >= P, the first tiles are exactly 0 .. P-1
    grid, visits = log(ctx, 64, 64, 1, 16, 8, 152)
    assert sorted(v[0][0] for v in visits) == list(range(152))


def test_release_from_start(ctx):
    G, P = 4, 64
    ctx.set_release([1, 1, 1, 0])  # group 0's flag is ignored
    torch.cuda.synchronize()
    grid, visits = log(ctx, 40, 13, 1, 16, G, P)
    ctx.set_release([0, 0, 0, 0])
    torch.cuda.synchronize()
    S.check_ws_trace([[t for (t, _, _, _) in v] for v in visits], grid.tiles, G, S.WS_STRIPED)
    for c, v in enumerate(visits):
        if c % G in (1, 2):  # released before launch: only ticket c div G of the home group
            tiles = S.ws_group_tiles(grid.tiles, G, S.WS_STRIPED, P)[c % G]
            assert [t for (t, _, _, _) in v] == tiles[c // G: c // G + 1], c


@pytest.mark.parametrize("cfg", [pgt.CFG_1CTA_128x256, pgt.CFG_2CTA_256x256])
@pytest.mark.parametrize("M,N,K", [(2048, 2048, 512), (1000, 1104, 200)])
def test_gemm_bit_identical_to_static_with_valid_trace(ctx, cfg, M, N, K):
    A, B = synthetic.gemm_bf16_inputs(M, N, K, seed=91)
    dA, dB = dev_u16(A), dev_u16(B)
    ref = torch.empty((M, N), dtype=torch.int16, device="cuda")
    ctx.gemm_ex(pgt.make_desc(M, N, K, sched_mode=pgt.SWIZZLED, kernel_cfg=cfg), dA, dB, ref)
    for G_ws in (1, 8, 16):
        desc = pgt.make_desc(M, N, K, sched_mode=pgt.WORK_STEALING, ws_groups=G_ws, kernel_cfg=cfg,
                             ws_layout=pgt.WS_STRIPED)
        plan = ctx.gemm_plan(desc)
        tb = pgt.TraceBuffers(plan["ctas"], plan["tiles"])
        C = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
        ctx.gemm_ex(desc, dA, dB, C, trace=tb.struct)
        torch.cuda.synchronize()
        assert ctx.last_error()[0] == 0
        assert torch.equal(C, ref), G_ws
        visits, _ = tb.read()
        cs = plan["cluster_size"]
        wv = [visits[w * cs] for w in range(plan["workers"])]
        S.check_ws_trace([[t for (t, _, _, _) in v] for v in wv], plan["tiles"], plan["ws_groups"], S.WS_STRIPED)
        if cs == 2:  # both CTAs of a pair visit the same tiles
            assert [[t for (t, _, _, _) in visits[w * 2 + 1]] for w in range(plan["workers"])] == \
                   [[t for (t, _, _, _) in v] for v in wv]


def test_gemm_8192_matches_static(ctx):
    M = N = K = 8192
    A, B = synthetic.gemm_bf16_inputs(M, N, K, seed=92, dist="normal")
    dA, dB = dev_u16(A), dev_u16(B)
    ref = torch.empty((M, N), dtype=torch.int16, device="cuda")
    C = torch.empty((M, N), dtype=torch.int16, device="cuda")
    ctx.gemm_ex(pgt.make_desc(M, N, K, sched_mode=pgt.SWIZZLED), dA, dB, ref)
    ctx.gemm_ex(pgt.make_desc(M, N, K, sched_mode=pgt.WORK_STEALING, ws_groups=8, ws_layout=pgt.WS_STRIPED),
                dA, dB, C)
    torch.cuda.synchronize()
    assert ctx.last_error()[0] == 0
    assert torch.equal(C, ref)


def test_unknown_layout_rejected(ctx):
    A = torch.zeros((64, 64), dtype=torch.int16, device="cuda")
    desc = pgt.make_desc(64, 64, 64, sched_mode=pgt.WORK_STEALING, ws_layout=2)
    with pytest.raises(pgt.PgtError) as e:
        ctx.gemm_ex(desc, A, A, A)
    assert e.value.status == pgt.ERR_ARG
    tb = pgt.TraceBuffers(4, 16)
    with pytest.raises(pgt.PgtError) as e:
        ctx.schedule_log(4, 4, 1, pgt.WORK_STEALING, 1, 2, 4, tb.struct, ws_layout=2)
    assert e.value.status == pgt.ERR_ARG



def test_worker_limit_for_work_stealing(ctx):
    """Work stealing's group arithmetic is 32-bit for P <= 65535: more workers are refused on
    the host before anything is launched (other modes are not limited)."""
    tb = pgt.TraceBuffers(1, 1)
    with pytest.raises(pgt.PgtError) as e:
        ctx.schedule_log(4, 4, 1, pgt.WORK_STEALING, 1, 2, 65536, tb.struct)
    assert e.value.status == pgt.ERR_ARG
    A = torch.zeros((64, 64), dtype=torch.int16, device="cuda")
    desc = pgt.make_desc(64, 64, 64, sched_mode=pgt.WORK_STEALING, num_workers=65536)
    with pytest.raises(pgt.PgtError) as e:
        ctx.gemm_ex(desc, A, A, A)
    assert e.value.status == pgt.ERR_ARG


@pytest.mark.parametrize("layout", [pgt.WS_RANGES, pgt.WS_STRIPED])
@pytest.mark.parametrize("K", [64, 576, 2048])
def test_uneven_home_counts_and_short_tiles(ctx, layout, K):
    """7 workers on 3 counter groups (homes 3, 2, 2: shares in proportion), with K from one
    stage (the next tile asked for at the tile's first load) to many: exact-once visits in
    each worker's order, the launch tiles, and the static order's bits."""
    M, N = 1280, 1536
    A, B = synthetic.gemm_bf16_inputs(M, N, K, seed=93)
    dA, dB = dev_u16(A), dev_u16(B)
    ref = torch.empty((M, N), dtype=torch.int16, device="cuda")
    ctx.gemm_ex(pgt.make_desc(M, N, K, sched_mode=pgt.SWIZZLED, kernel_cfg=pgt.CFG_1CTA_128x128), dA, dB, ref)
    desc = pgt.make_desc(M, N, K, sched_mode=pgt.WORK_STEALING, ws_groups=3, ws_layout=layout, num_workers=7,
                         kernel_cfg=pgt.CFG_1CTA_128x128)
    plan = ctx.gemm_plan(desc)
    assert plan["workers"] == 7 and plan["ws_groups"] == 3
    for _ in range(2):  # the second launch relies on the in-kernel counter reset
        tb = pgt.TraceBuffers(plan["ctas"], plan["tiles"])
        C = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
        ctx.gemm_ex(desc, dA, dB, C, trace=tb.struct)
        torch.cuda.synchronize()
        assert ctx.last_error()[0] == 0
        assert torch.equal(C, ref)
        visits, _ = tb.read()
        lists = [[t for (t, _, _, _) in v] for v in visits]
        S.check_ws_trace(lists, plan["tiles"], 3, layout)
        groups = S.ws_group_tiles(plan["tiles"], 3, layout, 7)
        for w, v in enumerate(lists):
            assert v[0] == groups[w % 3][w // 3]  # the launch ticket
