"""GPU parity for the device tile scheduler (pgt_schedule_log) against oracle.schedule:
static modes bit-exact per worker, work stealing by the protocol's invariants."""
import pytest
import torch

import persistent_gemm_tile_gb300 as pgt
from gpu_helpers import need_gpu
from oracle import schedule as S

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    need_gpu()
    c = pgt.Context(0, max_groups=16)
    yield c
    c.close()


def run_log(ctx, mb, nb, cs, mode, G, G_ws, P):
    grid = S.Grid(mb, nb, cs)
    tb = pgt.TraceBuffers(P, max(grid.tiles, 1))
    ctx.schedule_log(mb, nb, cs, mode, G, G_ws, P, tb.struct)
    torch.cuda.synchronize()
    visits, times = tb.read()
    return grid, visits, times


GRIDS = [(1, 1, 1), (3, 5, 1), (7, 4, 2), (19, 32, 1), (5, 17, 2), (32, 64, 1), (64, 64, 2), (40, 13, 1)]
STATIC = [S.BLOCKED, S.INTERLEAVED, S.SWIZZLED, S.BLOCKED_GROUPED_M]


@pytest.mark.parametrize("mb,nb,cs", GRIDS)
@pytest.mark.parametrize("P", [1, 3, 8, 152, 200])
@pytest.mark.parametrize("G", [1, 2, 3, 16])
def test_static_schedules_bit_exact(ctx, mb, nb, cs, P, G):
    for mode in STATIC:
        grid, visits, _ = run_log(ctx, mb, nb, cs, mode, G, 1, P)
        expect = S.static_schedule(mode, grid, P, G)
        got = [[(t, m, n) for (t, m, n, _) in v] for v in visits]
        want = [[(t, m, n) for (_, t, m, n) in v] for v in expect]
        assert got == want, S.MODE_NAMES[mode]


@pytest.mark.parametrize("mb,nb,cs", GRIDS)
@pytest.mark.parametrize("P,G_ws", [(1, 1), (4, 2), (152, 8), (152, 16), (300, 8), (7, 3)])
@pytest.mark.parametrize("G", [1, 16])
def test_work_stealing_invariants(ctx, mb, nb, cs, P, G_ws, G):
    for rep in range(2):  # the second launch relies on the in-kernel counter reset
        grid, visits, _ = run_log(ctx, mb, nb, cs, S.WORK_STEALING, G, G_ws, P)
        S.check_ws_trace([[t for (t, _, _, _) in v] for v in visits], grid.tiles, G_ws)
        for v in visits:
            for (t, m, n, _) in v:
                assert (m, n) == S.decode(S.WORK_STEALING, t, grid, G)


def test_work_stealing_host_reset_flag():
    need_gpu()
    c = pgt.Context(0, max_groups=8, flags=pgt.FLAG_HOST_RESET)
    for _ in range(3):
        grid, visits, _ = run_log(c, 19, 32, 1, S.WORK_STEALING, 16, 8, 152)
        S.check_ws_trace([[t for (t, _, _, _) in v] for v in visits], grid.tiles, 8)
    c.close()


def test_ws_groups_above_max_rejected(ctx):
    tb = pgt.TraceBuffers(4, 16)
    with pytest.raises(pgt.PgtError) as e:
        ctx.schedule_log(4, 4, 1, S.WORK_STEALING, 1, 17, 4, tb.struct)
    assert e.value.status == pgt.ERR_GROUPS
