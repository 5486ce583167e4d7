"""GPU parity for the fused multi-space persistent loop (pgt_multi_loop): outputs bit-exact
against oracle.add.scale_f32, traced tile order equal to oracle.schedule.multi_space_schedule."""
import numpy as np
import pytest
import torch

import persistent_gemm_tile_gb300 as pgt
import synthetic
from gpu_helpers import need_gpu
from oracle import add as OA
from oracle import schedule as S

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    need_gpu()
    c = pgt.Context(0)
    yield c
    c.close()


def bits(a):
    return np.ascontiguousarray(a).view(np.uint32)


@pytest.mark.parametrize("mode", [pgt.BLOCKED, pgt.INTERLEAVED])
@pytest.mark.parametrize("tile", [(32, 16), (0, 0), (5, 12)])
def test_two_spaces_page_scales_bit_exact(ctx, mode, tile):
    x, _ = synthetic.add_inputs(3000, 4100, seed=51)
    y, _ = synthetic.add_inputs(1234, 2048, seed=52)
    tx, ty = torch.from_numpy(x).cuda(), torch.from_numpy(y).cuda()
    o1, o2 = torch.full_like(tx, float("nan")), torch.full_like(ty, float("nan"))
    ctx.multi_loop([(tx, o1, 2.0), (ty, o2, 3.0)], sched_mode=mode, tile_r=tile[0], tile_c=tile[1])
    torch.cuda.synchronize()
    assert np.array_equal(bits(o1.cpu().numpy()), bits(OA.scale_f32(x, 2.0)))
    assert np.array_equal(bits(o2.cpu().numpy()), bits(OA.scale_f32(y, 3.0)))


@pytest.mark.parametrize("mode", [pgt.BLOCKED, pgt.INTERLEAVED])
@pytest.mark.parametrize("P", [1, 3, 7, 152])
def test_traced_order_matches_oracle(ctx, mode, P):
    shapes = [(64, 32), (32, 48), (100, 70), (33, 17)]
    arrays = [synthetic.add_inputs(r, c, seed=60 + i)[0] for i, (r, c) in enumerate(shapes)]
    dev = [torch.from_numpy(a).cuda() for a in arrays]
    outs = [torch.empty_like(d) for d in dev]
    scales = [2.0, 3.0, -0.5, 1.0 / 3.0]
    grids = [S.grid_for(r, c, 32, 16) for (r, c) in shapes]
    total = sum(g.tiles for g in grids)
    tb = pgt.TraceBuffers(P, total)
    ctx.multi_loop(list(zip(dev, outs, scales)), sched_mode=mode, tile_r=32, tile_c=16, num_workers=P,
                   trace=tb.struct)
    torch.cuda.synchronize()
    visits, _ = tb.read()
    got = [[(t, f >> 24, m, n) for (t, m, n, f) in v] for v in visits]
    want = [[(t, s, m, n) for (_, t, s, m, n) in v] for v in S.multi_space_schedule(mode, grids, P)]
    assert got == want
    for a, o, sc in zip(arrays, outs, scales):
        assert np.array_equal(bits(o.cpu().numpy()), bits(OA.scale_f32(a, sc)))


def test_in_place_and_unaligned(ctx):
    x, _ = synthetic.add_inputs(257, 301, seed=70)
    big = torch.zeros((257, 320), dtype=torch.float32, device="cuda")
    view = big[:, 3:304]  # 12-byte offset: scalar path
    view.copy_(torch.from_numpy(x))
    y, _ = synthetic.add_inputs(128, 512, seed=71)
    ty = torch.from_numpy(y).cuda()
    ctx.multi_loop([(view, view, 2.0), (ty, ty, 3.0)])
    torch.cuda.synchronize()
    assert np.array_equal(bits(view.cpu().numpy()), bits(OA.scale_f32(x, 2.0)))
    assert np.array_equal(bits(ty.cpu().numpy()), bits(OA.scale_f32(y, 3.0)))
    assert torch.count_nonzero(big[:, :3]) == 0 and torch.count_nonzero(big[:, 304:]) == 0


def test_multi_loop_argument_errors(ctx):
    t = torch.zeros((8, 8), device="cuda")
    with pytest.raises(pgt.PgtError):
        ctx.multi_loop([])
    with pytest.raises(pgt.PgtError):
        ctx.multi_loop([(t, t, 1.0)] * 9)
    with pytest.raises(pgt.PgtError):
        ctx.multi_loop([(t, t, 1.0)], sched_mode=pgt.SWIZZLED)
