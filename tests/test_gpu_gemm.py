"""GPU parity for the persistent bf16 GEMM against oracle.gemm / oracle.schedule.

Bars: exact equality for closed forms; relative Frobenius <= 1e-3 against bf16(C64) and
per-element |C - C64| <= 1e-2 * (|A|.|B|) against the fp64 oracle; bit-identical output
across scheduler modes for one kernel configuration; traced schedules equal to the
oracle's (static modes) or valid under the ticket protocol (work stealing)."""
import numpy as np
import pytest
import torch

import persistent_gemm_tile_gb300 as pgt
import synthetic
from gpu_helpers import dev_u16, host_u16, need_gpu
from oracle import gemm as OG
from oracle import numerics as NM
from oracle import schedule as S

pytestmark = pytest.mark.gpu

ALL_MODES = [pgt.BLOCKED, pgt.INTERLEAVED, pgt.SWIZZLED, pgt.WORK_STEALING, pgt.BLOCKED_GROUPED_M]
BF16_CFGS = [pgt.CFG_1CTA_128x128, pgt.CFG_1CTA_128x256, pgt.CFG_2CTA_256x128, pgt.CFG_2CTA_256x256]


@pytest.fixture(scope="module")
def ctx():
    need_gpu()
    c = pgt.Context(0, max_groups=16)
    yield c
    c.close()


def run(ctx, A, B, M, N, K, *, b_layout=pgt.B_KN, mode=pgt.SWIZZLED, G=16, cfg=pgt.CFG_AUTO, lda=0, ldb=0,
        ldc=0, ws_groups=0, workers=0, trace=False, ws_layout=pgt.WS_RANGES):
    desc = pgt.make_desc(M, N, K, lda=lda, ldb=ldb, ldc=ldc, b_layout=b_layout, sched_mode=mode, group_size=G,
                         ws_groups=ws_groups, kernel_cfg=cfg, num_workers=workers, ws_layout=ws_layout)
    plan = ctx.gemm_plan(desc)
    C = torch.full((M, ldc or N), -1, dtype=torch.int16, device="cuda")
    tb = pgt.TraceBuffers(plan["ctas"], plan["tiles"]) if trace else None
    ctx.gemm_ex(desc, A, B, C, trace=tb.struct if tb else None)
    torch.cuda.synchronize()
    rc, detail = ctx.last_error()
    assert rc == 0, f"device error {detail}"
    return C, plan, tb


def oracle_full(A_bits, B_bits, M, N, K, b_kn=True):
    return OG.gemm_full(OG.dequant_bf16(A_bits), OG.dequant_bf16(B_bits), b_kn, M, N, K)


# ------------------------------------------------------------------ closed forms
@pytest.mark.parametrize("cfg", BF16_CFGS)
@pytest.mark.parametrize("b_layout", [pgt.B_KN, pgt.B_NK])
def test_identity_gives_b_exactly(ctx, cfg, b_layout):
    M = N = K = 256
    eye = synthetic.f64_to_bf16_bits(np.eye(K))
    _, Bb = synthetic.gemm_bf16_inputs(M, N, K, seed=11, b_layout="kn")
    Bstore = Bb if b_layout == pgt.B_KN else np.ascontiguousarray(Bb.T)
    C, _, _ = run(ctx, dev_u16(eye), dev_u16(Bstore), M, N, K, b_layout=b_layout, cfg=cfg)
    assert np.array_equal(host_u16(C), Bb)


@pytest.mark.parametrize("cfg", BF16_CFGS)
@pytest.mark.parametrize("K", [256, 8192])
def test_all_ones_gives_k(ctx, cfg, K):
    M, N = 256, 384
    one = np.uint16(0x3F80)
    A = np.full((M, K), one, np.uint16)
    B = np.full((K, N), one, np.uint16)
    C, _, _ = run(ctx, dev_u16(A), dev_u16(B), M, N, K, cfg=cfg)
    assert np.all(host_u16(C) == NM.f64_to_bf16_rne(np.float64(K)))


@pytest.mark.parametrize("cfg", BF16_CFGS)
def test_k1_outer_product(ctx, cfg):
    M, N, K, lda = 300, 200, 1, 8
    A, B = synthetic.gemm_bf16_inputs(M, N, K, seed=12, lda=lda)
    C, _, _ = run(ctx, dev_u16(A), dev_u16(B), M, N, K, lda=lda, cfg=cfg)
    a = NM.bf16_bits_to_f64(A[:, 0])
    b = NM.bf16_bits_to_f64(B[0])
    assert np.array_equal(host_u16(C), NM.f64_to_bf16_rne(a[:, None] * b[None, :]))


# ---------------------------------------------------- 256^3, 4 tiles, every mode
def test_256_all_modes_schedule_and_values(ctx):
    M = N = K = 256
    A, B = synthetic.gemm_bf16_inputs(M, N, K, seed=0, dist="uniform")
    C64, Abs = oracle_full(A, B, M, N, K)
    outs = []
    for mode in ALL_MODES:
        G = 2 if mode in (pgt.SWIZZLED, pgt.WORK_STEALING) else 2
        C, plan, tb = run(ctx, dev_u16(A), dev_u16(B), M, N, K, mode=mode, G=G, cfg=pgt.CFG_1CTA_128x128,
                          trace=True)
        assert plan["tiles"] == 4 and plan["workers"] == 4
        assert plan["ws_groups"] == 4  # eight requested, one per worker in use
        c = host_u16(C)
        OG.check(c, C64, Abs)
        outs.append(c)
        visits, _ = tb.read()
        grid = S.Grid(plan["m_blocks"], plan["n_blocks"], 1)
        if mode == pgt.WORK_STEALING:
            S.check_ws_trace([[t for (t, _, _, _) in v] for v in visits], grid.tiles, plan["ws_groups"])
        else:
            want = S.static_schedule(mode, grid, plan["workers"], G)
            assert [[(t, m, n) for (t, m, n, _) in v] for v in visits] == \
                   [[(t, m, n) for (_, t, m, n) in v] for v in want]
    for c in outs[1:]:
        assert np.array_equal(c, outs[0])


def worker_visits(visits, cs):
    """Per-worker visit lists from per-CTA traces; both CTAs of a pair must agree."""
    out = []
    for w in range(len(visits) // cs):
        lists = [[(t, m, n) for (t, m, n, _) in v] for v in visits[w * cs:(w + 1) * cs]]
        for other in lists[1:]:
            assert other == lists[0], f"CTAs of pair {w} visited different tiles"
        out.append(visits[w * cs])
    return out


# ------------------------------------------------------------- K tails, layouts
@pytest.mark.parametrize("cfg", BF16_CFGS)
@pytest.mark.parametrize("K", [1, 63, 64, 65, 130, 1000])
@pytest.mark.parametrize("b_layout", [pgt.B_KN, pgt.B_NK])
def test_k_tails_and_layouts(ctx, cfg, K, b_layout):
    M, N = 200, 328
    lda = -(-K // 8) * 8
    lay = "kn" if b_layout == pgt.B_KN else "nk"
    ldb = N if lay == "kn" else lda
    A, B = synthetic.gemm_bf16_inputs(M, N, K, seed=13, lda=lda, b_layout=lay, ldb=ldb)
    C, _, _ = run(ctx, dev_u16(A), dev_u16(B), M, N, K, b_layout=b_layout, lda=lda, ldb=ldb, cfg=cfg)
    C64, Abs = OG.gemm_full(OG.dequant_bf16(A), OG.dequant_bf16(B), lay == "kn", M, N, K)
    OG.check(host_u16(C), C64, Abs)


@pytest.mark.parametrize("cfg", BF16_CFGS)
def test_ldc_padding_untouched(ctx, cfg):
    M, N, K, ldc = 130, 72, 96, 88
    A, B = synthetic.gemm_bf16_inputs(M, N, K, seed=14)
    C, _, _ = run(ctx, dev_u16(A), dev_u16(B), M, N, K, ldc=ldc, cfg=cfg)
    c = host_u16(C)
    assert np.all(c[:, N:] == 0xFFFF)  # -1 fill, never written
    C64, Abs = oracle_full(A, B, M, N, K)
    OG.check(np.ascontiguousarray(c[:, :N]), C64, Abs)


# ------------------------------------------- workers, groups: schedule + identity
@pytest.mark.parametrize("cfg", BF16_CFGS)
@pytest.mark.parametrize("workers", [1, 3, 7, 0])
def test_modes_bit_identical_with_traces(ctx, cfg, workers):
    M, N, K = 1000, 1104, 320
    A, B = synthetic.gemm_bf16_inputs(M, N, K, seed=15)
    C64, Abs = oracle_full(A, B, M, N, K)
    ref = None
    for mode in ALL_MODES:
        for G in (1, 3, 16):
            C, plan, tb = run(ctx, dev_u16(A), dev_u16(B), M, N, K, mode=mode, G=G, cfg=cfg, workers=workers,
                              trace=True, ws_groups=4)
            c = host_u16(C)
            if ref is None:
                OG.check(c, C64, Abs)
                ref = c
            else:
                assert np.array_equal(c, ref), (mode, G)
            visits, _ = tb.read()
            cs = plan["cluster_size"]
            visits = worker_visits(visits, cs)
            grid = S.Grid(plan["m_blocks"], plan["n_blocks"], cs)
            if mode == pgt.WORK_STEALING:
                S.check_ws_trace([[t for (t, _, _, _) in v] for v in visits], grid.tiles, plan["ws_groups"])
            else:
                want = S.static_schedule(mode, grid, plan["workers"], G)
                assert [[(t, m, n) for (t, m, n, _) in v] for v in visits] == \
                       [[(t, m, n) for (_, t, m, n) in v] for v in want]


# -------------------------------------------------------- ragged-tail GEMM set
RAGGED = [(4864, 4096, 2048), (128, 16384, 16384), (3000, 5000, 1024)]


@pytest.fixture(scope="module")
def ragged_inputs():
    return synthetic.gemm_bf16_sequence(RAGGED, seed=3, dist="uniform")


@pytest.fixture(scope="module")
def ragged_oracle(ragged_inputs):
    """fp64 C and |A|.|B| of each ragged shape, computed once per module."""
    cache = {}

    def get(idx):
        if idx not in cache:
            M, N, K = RAGGED[idx]
            A, B = ragged_inputs[idx]
            cache[idx] = oracle_full(A, B, M, N, K)
        return cache[idx]
    return get


@pytest.mark.parametrize("cfg", [pgt.CFG_AUTO, pgt.CFG_1CTA_128x256, pgt.CFG_2CTA_256x128])
@pytest.mark.parametrize("idx", [0, 1, 2])
def test_ragged_set_all_modes(ctx, ragged_inputs, ragged_oracle, idx, cfg):
    """Every element of C against the fp64 oracle (first mode), then bit identity across
    the other schedulers."""
    M, N, K = RAGGED[idx]
    A, B = ragged_inputs[idx]
    dA, dB = dev_u16(A), dev_u16(B)
    ref = None
    for mode in ALL_MODES + [pgt.LAUNCH_CONTROL]:
        C, plan, _ = run(ctx, dA, dB, M, N, K, mode=mode, G=16, cfg=cfg)
        if ref is None:
            ref = C
            C64, Abs = ragged_oracle(idx)
            OG.check(host_u16(C), C64, Abs)
        else:
            assert torch.equal(C, ref), mode


# ----------------------------------------------------------- 8192^3 bf16 (full)
@pytest.fixture(scope="module")
def big_inputs():
    M = N = K = 8192
    A, B = synthetic.gemm_bf16_inputs(M, N, K, seed=2, dist="normal")
    return A, B


@pytest.fixture(scope="module")
def big_oracle(big_inputs):
    A, B = big_inputs
    return oracle_full(A, B, 8192, 8192, 8192)


@pytest.mark.parametrize("cfg", [pgt.CFG_AUTO, pgt.CFG_1CTA_128x128, pgt.CFG_1CTA_128x256, pgt.CFG_2CTA_256x128])
def test_8192_full_matrix_swizzled_vs_work_stealing(ctx, big_inputs, big_oracle, cfg):
    """The benchmark workload: all 8192 x 8192 outputs against the fp64 oracle, and work
    stealing (both tile ownerships) and launch control bit-identical to the swizzled order.
    AUTO must keep the pair 256 x 256 tile at this size."""
    M = N = K = 8192
    A, B = big_inputs
    dA, dB = dev_u16(A), dev_u16(B)
    C1, plan, _ = run(ctx, dA, dB, M, N, K, mode=pgt.SWIZZLED, G=16, cfg=cfg)
    if cfg == pgt.CFG_AUTO:
        assert plan["kernel_cfg"] == pgt.CFG_2CTA_256x256
    C64, Abs = big_oracle
    OG.check(host_u16(C1), C64, Abs)
    for kw in (dict(mode=pgt.WORK_STEALING), dict(mode=pgt.WORK_STEALING, ws_layout=pgt.WS_STRIPED),
               dict(mode=pgt.LAUNCH_CONTROL)):
        C2, _, _ = run(ctx, dA, dB, M, N, K, G=16, cfg=cfg, **kw)
        assert torch.equal(C1, C2), kw


# ------------------------------------------------------------------ AUTO per shape
@pytest.mark.parametrize("M,N,K,b_layout", [(256, 256, 256, pgt.B_KN), (128, 16384, 16384, pgt.B_KN),
                                            (8192, 8192, 8192, pgt.B_KN), (3000, 5000, 1024, pgt.B_NK),
                                            (1, 8, 8, pgt.B_KN)])
def test_auto_picks_a_candidate_whatever_the_scheduler(ctx, M, N, K, b_layout):
    """AUTO resolves to one of its candidate tiles, and to the same one for every scheduler
    and worker count (the choice depends on the problem alone)."""
    cfgs = set()
    for mode in ALL_MODES + [pgt.LAUNCH_CONTROL]:
        for workers in (0, 1):
            if mode == pgt.LAUNCH_CONTROL and workers:
                continue
            d = pgt.make_desc(M, N, K, b_layout=b_layout, sched_mode=mode, num_workers=workers)
            cfgs.add(ctx.gemm_plan(d)["kernel_cfg"])
    assert len(cfgs) == 1
    assert cfgs.pop() in (pgt.CFG_1CTA_128x128, pgt.CFG_1CTA_128x256, pgt.CFG_2CTA_256x256)


# ------------------------------------------------------------- the flat form
def test_flat_gemm_ws_groups(ctx):
    """pgt_gemm's counter-group count: work stealing on 1, 3 and 16 groups gives the bits of
    the swizzled order; a count above the context's max_groups is rejected."""
    M, N, K = 1000, 1104, 320
    A, B = synthetic.gemm_bf16_inputs(M, N, K, seed=16)
    dA, dB = dev_u16(A), dev_u16(B)
    ref = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
    ctx.gemm(dA, dB, ref, M, N, K, sched_mode=pgt.SWIZZLED)
    torch.cuda.synchronize()
    C64, Abs = oracle_full(A, B, M, N, K)
    OG.check(host_u16(ref), C64, Abs)
    for g in (1, 3, 16, 0):
        C = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
        ctx.gemm(dA, dB, C, M, N, K, sched_mode=pgt.WORK_STEALING, ws_groups=g)
        torch.cuda.synchronize()
        assert ctx.last_error()[0] == 0
        assert torch.equal(C, ref), g
    with pytest.raises(pgt.PgtError) as e:
        ctx.gemm(dA, dB, ref, M, N, K, sched_mode=pgt.WORK_STEALING, ws_groups=ctx.max_groups + 1)
    assert e.value.status == pgt.ERR_GROUPS


# ------------------------------------------------------------------- errors
def test_argument_errors(ctx):
    A = torch.zeros((64, 64), dtype=torch.int16, device="cuda")
    C = torch.zeros((64, 64), dtype=torch.int16, device="cuda")
    bad = [
        (dict(M=0), pgt.ERR_ARG),
        (dict(lda=60), pgt.ERR_ARG),        # lda < K
        (dict(lda=68), pgt.ERR_ALIGN),      # 136-byte rows
        (dict(ws_groups=17), pgt.ERR_GROUPS),
        (dict(group_size=0), pgt.ERR_ARG),
        (dict(sched_mode=9), pgt.ERR_ARG),
        (dict(kernel_cfg=99), pgt.ERR_UNSUPPORTED),
        (dict(kernel_cfg=pgt.CFG_2CTA_256x224), pgt.ERR_UNSUPPORTED),  # MXFP8 only
        (dict(dtype=pgt.MXFP8, b_layout=pgt.B_KN), pgt.ERR_ARG),  # MXFP8 needs B stored N x K
    ]
    for kw, status in bad:
        args = dict(M=64, N=64, K=64)
        args.update(kw)
        desc = pgt.make_desc(args.pop("M"), args.pop("N"), args.pop("K"), **args)
        with pytest.raises(pgt.PgtError) as e:
            ctx.gemm_ex(desc, A, A, C)
        assert e.value.status == status, kw
    desc = pgt.make_desc(64, 64, 64)
    with pytest.raises(pgt.PgtError) as e:  # misaligned base pointer
        ctx.gemm_ex(desc, A.data_ptr() + 2, A, C)
    assert e.value.status == pgt.ERR_ALIGN
    with pytest.raises(pgt.PgtError) as e:  # scales given for bf16
        ctx.gemm_ex(desc, A, A, C, sfa=A)
    assert e.value.status == pgt.ERR_ARG
