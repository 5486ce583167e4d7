"""GPU parity for the persistent add: bit-exact against oracle.add on the 8192 x 8192
workload and on ragged, strided, misaligned and aliased cases; the traced tile order
matches oracle.schedule."""
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


@pytest.fixture(scope="module")
def big():
    x, y = synthetic.add_inputs(8192, 8192, seed=1)
    return x, y, OA.add_f32(x, y)


@pytest.mark.parametrize("tile", [(32, 16), (0, 0), (16, 512), (4, 2048)])
@pytest.mark.parametrize("mode", [pgt.BLOCKED, pgt.INTERLEAVED])
def test_add_8192_bit_exact(ctx, big, tile, mode):
    x, y, ref = big
    tx, ty = torch.from_numpy(x).cuda(), torch.from_numpy(y).cuda()
    out = torch.full_like(tx, float("nan"))
    ctx.add(tx, ty, out, sched_mode=mode, tile_r=tile[0], tile_c=tile[1])
    torch.cuda.synchronize()
    assert np.array_equal(bits(out.cpu().numpy()), bits(ref))


@pytest.mark.parametrize("rows,cols", [(1, 1), (1, 5), (33, 17), (1000, 1001), (517, 4096), (4099, 3)])
@pytest.mark.parametrize("tile", [(32, 16), (0, 0), (7, 12)])
def test_add_ragged_shapes(ctx, rows, cols, tile):
    x, y = synthetic.add_inputs(rows, cols, seed=5)
    ref = OA.add_f32(x, y)
    tx, ty = torch.from_numpy(x).cuda(), torch.from_numpy(y).cuda()
    out = torch.full_like(tx, float("nan"))
    ctx.add(tx, ty, out, sched_mode=pgt.INTERLEAVED, tile_r=tile[0], tile_c=tile[1])
    torch.cuda.synchronize()
    assert np.array_equal(bits(out.cpu().numpy()), bits(ref))


def test_add_strided_and_unaligned(ctx):
    x, y = synthetic.add_inputs(300, 257, seed=6)
    ref = OA.add_f32(x, y)
    big_x = torch.zeros((300, 300), dtype=torch.float32, device="cuda")
    big_y = torch.zeros((300, 264), dtype=torch.float32, device="cuda")
    big_o = torch.full((300, 280), float("nan"), dtype=torch.float32, device="cuda")
    vx, vy, vo = big_x[:, :257], big_y[:, 3:260], big_o[:, 1:258]  # y and out start off 16-byte
    vx.copy_(torch.from_numpy(x))
    vy.copy_(torch.from_numpy(y))
    ctx.add(vx, vy, vo, sched_mode=pgt.BLOCKED)
    torch.cuda.synchronize()
    assert np.array_equal(bits(vo.cpu().numpy()), bits(ref))
    assert torch.isnan(big_o[:, 0]).all() and torch.isnan(big_o[:, 258:]).all()  # nothing outside written


def test_add_in_place(ctx):
    x, y = synthetic.add_inputs(640, 512, seed=7)
    ref = OA.add_f32(x, y)
    tx, ty = torch.from_numpy(x).cuda(), torch.from_numpy(y).cuda()
    ctx.add(tx, ty, tx)
    torch.cuda.synchronize()
    assert np.array_equal(bits(tx.cpu().numpy()), bits(ref))


def test_add_special_values_no_flush(ctx):
    x = np.array([[2.0 ** -149, 1.0, np.inf, 3e38, -0.0, 1.0 + 2.0 ** -23, 2.0 ** -126, np.nan]], np.float32)
    y = np.array([[2.0 ** -149, 2.0 ** -24, -np.inf, 3e38, 0.0, 2.0 ** -24, -2.0 ** -127, 1.0]], np.float32)
    tx, ty = torch.from_numpy(x).cuda(), torch.from_numpy(y).cuda()
    out = torch.empty_like(tx)
    ctx.add(tx, ty, out, tile_r=32, tile_c=16)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    ref = OA.add_f32(x, y)
    same = (bits(got) == bits(ref)) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


@pytest.mark.parametrize("mode", [pgt.BLOCKED, pgt.INTERLEAVED])
@pytest.mark.parametrize("P,rows,cols", [(1, 200, 300), (5, 200, 300), (152, 200, 300), (3000, 200, 300),
                                         (2500, 2048, 2048)])
def test_add_trace_matches_oracle_schedule(ctx, mode, P, rows, cols):
    """Per-worker visit lists equal the oracle's.  With more workers than CTAs fit on the
    GPU (2500, 3000), each CTA runs several workers in turn."""
    tr, tc = 32, 16
    x, y = synthetic.add_inputs(rows, cols, seed=8)
    tx, ty = torch.from_numpy(x).cuda(), torch.from_numpy(y).cuda()
    out = torch.empty_like(tx)
    grid = S.Grid(-(-rows // tr), -(-cols // tc), 1)
    tb = pgt.TraceBuffers(P, grid.tiles)
    ctx.add(tx, ty, out, sched_mode=mode, tile_r=tr, tile_c=tc, num_workers=P, trace=tb.struct)
    torch.cuda.synchronize()
    visits, _ = tb.read()
    want = S.static_schedule(mode, grid, P, 1)
    assert [[(t, m, n) for (t, m, n, _) in v] for v in visits] == [[(t, m, n) for (_, t, m, n) in v] for v in want]
    assert np.array_equal(bits(out.cpu().numpy()), bits(OA.add_f32(x, y)))


def test_default_workers_keep_line_partners_together(ctx):
    """32 x 16 tiles are half a 128-byte line wide: the default worker count makes workers on
    neighbouring tile columns read the same rows together (blocked: whole columns split
    evenly, interleaved: waves of whole column pairs, two workers per resident CTA); the wide
    tile takes every CTA that fits, whatever the order."""
    m_tiles, n_tiles = 8192 // 32, 8192 // 16
    P = ctx.add_workers(8192, 8192, 32, 16, sched_mode=pgt.BLOCKED)
    assert P % n_tiles == 0 and m_tiles % (P // n_tiles) == 0, P
    P = ctx.add_workers(8192, 8192, 32, 16, sched_mode=pgt.INTERLEAVED)
    assert P % (2 * m_tiles) == 0 and P > n_tiles, P  # about two workers per resident CTA
    wide = ctx.add_workers(8192, 8192, 0, 0, sched_mode=pgt.BLOCKED)
    assert wide == ctx.add_workers(8192, 8192, 0, 0, sched_mode=pgt.INTERLEAVED)
    assert wide % ctx.num_sms == 0
    assert ctx.add_workers(100, 100, 32, 16, num_workers=7) == 7


def test_add_rejects_bad_arguments(ctx):
    t = torch.zeros((4, 4), device="cuda")
    with pytest.raises(pgt.PgtError):
        ctx.add(t, t, t, sched_mode=pgt.SWIZZLED)
    with pytest.raises(pgt.PgtError):
        ctx.add(t, t, t, tile_r=2048, tile_c=16)
