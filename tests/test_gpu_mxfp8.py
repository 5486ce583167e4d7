"""GPU parity for the MXFP8 block-scaled GEMM (E4M3 payloads, one E8M0 scale per row and
128-wide K block) against oracle.gemm.

Exact pins: unit payloads with per-row/per-block scales make every fp32 partial sum exact,
so the result must equal bf16_rne of the fp64 oracle bit for bit; this fixes the scale
layout, the K-block -> scale mapping and the row/column -> scale mapping.  Random data is
held to the GEMM bars (relative Frobenius <= 1e-3 against bf16(C64), per element
|C - C64| <= 1e-2 |A|.|B|), and results are bit-identical across scheduler modes."""
import numpy as np
import pytest
import torch

import persistent_gemm_tile_gb300 as pgt
import synthetic
from gpu_helpers import dev_u8, host_u16, need_gpu
from oracle import gemm as OG
from oracle import numerics as NM
from oracle import schedule as S

pytestmark = pytest.mark.gpu

MX_CFGS = [pgt.CFG_1CTA_128x128, pgt.CFG_1CTA_128x256, pgt.CFG_2CTA_256x128, pgt.CFG_2CTA_256x256,
           pgt.CFG_2CTA_256x224]
MODES = [pgt.BLOCKED, pgt.INTERLEAVED, pgt.SWIZZLED, pgt.WORK_STEALING, pgt.BLOCKED_GROUPED_M]


@pytest.fixture(scope="module")
def ctx():
    need_gpu()
    c = pgt.Context(0, max_groups=16)
    yield c
    c.close()


def run_mx(ctx, qa, sa, qb, sb, M, N, K, cfg=pgt.CFG_AUTO, mode=pgt.SWIZZLED, G=16, workers=0, trace=False,
           ldc=0):
    desc = pgt.make_desc(M, N, K, dtype=pgt.MXFP8, b_layout=pgt.B_NK, sched_mode=mode, group_size=G,
                         kernel_cfg=cfg, num_workers=workers, ldc=ldc)
    plan = ctx.gemm_plan(desc)
    ws = torch.zeros(max(ctx.gemm_workspace_bytes(desc), 16), dtype=torch.uint8, device="cuda")
    C = torch.full((M, ldc or N), -1, dtype=torch.int16, device="cuda")
    tb = pgt.TraceBuffers(plan["ctas"], plan["tiles"]) if trace else None
    args = [qa, qb, C]
    ctx.gemm_ex(desc, *args, sfa=sa, sfb=sb, workspace=ws, trace=tb.struct if tb else None)
    torch.cuda.synchronize()
    rc, detail = ctx.last_error()
    assert rc == 0, f"device error {detail}"
    return C, plan, tb


def dev(*arrays):
    return [dev_u8(a) for a in arrays]


@pytest.mark.parametrize("cfg", MX_CFGS)
@pytest.mark.parametrize("M,N,K", [(256, 256, 128), (300, 392, 384), (512, 1024, 640), (1000, 1104, 2048)])
def test_unit_payload_random_scales_exact(ctx, cfg, M, N, K):
    rng = np.random.default_rng(31)
    kb = K // 128
    qa = np.full((M, K), 0x38, np.uint8)  # 1.0
    qb = np.full((N, K), 0x38, np.uint8)
    # exponents in [-3, 3]: every partial sum is a multiple of 2**-1 below 2**17, exact in fp32
    sa = (127 + rng.integers(-3, 4, (M, kb))).astype(np.uint8)
    sb = (127 + rng.integers(-3, 4, (N, kb))).astype(np.uint8)
    C, _, _ = run_mx(ctx, *dev(qa, sa, qb, sb), M, N, K, cfg=cfg)
    C64, _ = OG.gemm_full(OG.dequant_mxfp8(qa, sa), OG.dequant_mxfp8(qb, sb), False, M, N, K)
    assert np.array_equal(host_u16(C), NM.f64_to_bf16_rne(C64))


@pytest.mark.parametrize("cfg", MX_CFGS)
def test_signed_payloads_single_block_exact(ctx, cfg):
    # K = 128: one scale per row; payloads +-1, +-2, +-0.5 keep every fp32 sum exact
    M, N, K = 256, 256, 128
    rng = np.random.default_rng(32)
    codes = np.array([0x38, 0xB8, 0x40, 0xC0, 0x30, 0xB0], np.uint8)
    qa = codes[rng.integers(0, 6, (M, K))]
    qb = codes[rng.integers(0, 6, (N, K))]
    sa = (127 + rng.integers(-3, 4, (M, 1))).astype(np.uint8)
    sb = (127 + rng.integers(-3, 4, (N, 1))).astype(np.uint8)
    C, _, _ = run_mx(ctx, *dev(qa, sa, qb, sb), M, N, K, cfg=cfg)
    C64, _ = OG.gemm_full(OG.dequant_mxfp8(qa, sa), OG.dequant_mxfp8(qb, sb), False, M, N, K)
    assert np.array_equal(host_u16(C), NM.f64_to_bf16_rne(C64))


@pytest.mark.parametrize("cfg", MX_CFGS)
def test_random_modes_bit_identical_with_traces(ctx, cfg):
    M, N, K = 1000, 1104, 1536
    qa, sa, qb, sb = synthetic.gemm_mxfp8_inputs(M, N, K, seed=33)
    d = dev(qa, sa, qb, sb)
    C64, Abs = OG.gemm_full(OG.dequant_mxfp8(qa, sa), OG.dequant_mxfp8(qb, sb), False, M, N, K)
    ref = None
    for mode in MODES:
        C, plan, tb = run_mx(ctx, *d, M, N, K, cfg=cfg, mode=mode, G=3, workers=5, trace=True)
        c = host_u16(C)
        if ref is None:
            OG.check(c, C64, Abs)
            ref = c
        else:
            assert np.array_equal(c, ref), mode
        visits, _ = tb.read()
        cs = plan["cluster_size"]
        wv = [visits[w * cs] for w in range(plan["workers"])]
        grid = S.Grid(plan["m_blocks"], plan["n_blocks"], cs)
        if mode == pgt.WORK_STEALING:
            S.check_ws_trace([[t for (t, _, _, _) in v] for v in wv], grid.tiles, plan["ws_groups"])
        else:
            want = S.static_schedule(mode, grid, plan["workers"], 3)
            assert [[(t, m, n) for (t, m, n, _) in v] for v in wv] == [[(t, m, n) for (_, t, m, n) in v] for v in want]


@pytest.mark.parametrize("mode", MODES + [pgt.LAUNCH_CONTROL])
def test_224_tile_ragged_tail_columns(ctx, mode):
    """The 224-column pair tile stores its last 32 columns with direct global stores.  N =
    1100 ends inside that tail chunk (at a column that is not a multiple of 8), M = 1000 is
    ragged, and ldc = 1104: the padding columns must stay untouched."""
    M, N, K, ldc = 1000, 1100, 1664, 1104
    qa, sa, qb, sb = synthetic.gemm_mxfp8_inputs(M, N, K, seed=34)
    C, plan, _ = run_mx(ctx, *dev(qa, sa, qb, sb), M, N, K, cfg=pgt.CFG_2CTA_256x224, mode=mode, G=2, ldc=ldc)
    assert plan["bn"] == 224 and plan["n_blocks"] == 5
    c = host_u16(C)
    assert np.all(c[:, N:] == 0xFFFF)
    C64, Abs = OG.gemm_full(OG.dequant_mxfp8(qa, sa), OG.dequant_mxfp8(qb, sb), False, M, N, K)
    OG.check(c[:, :N], C64, Abs)
    C2, _, _ = run_mx(ctx, *dev(qa, sa, qb, sb), M, N, K, cfg=pgt.CFG_2CTA_256x224, mode=pgt.BLOCKED, G=2, ldc=ldc)
    assert torch.equal(C, C2)


def test_224_tile_unsupported_for_bf16(ctx):
    A = torch.zeros((256, 256), dtype=torch.int16, device="cuda")
    desc = pgt.make_desc(256, 256, 256, kernel_cfg=pgt.CFG_2CTA_256x224)
    with pytest.raises(pgt.PgtError) as e:
        ctx.gemm_ex(desc, A, A, A)
    assert e.value.status == pgt.ERR_UNSUPPORTED


@pytest.fixture(scope="module")
def big_mx():
    M = N = K = 8192
    return synthetic.gemm_mxfp8_inputs(M, N, K, seed=4)


@pytest.fixture(scope="module")
def big_mx_oracle(big_mx):
    qa, sa, qb, sb = big_mx
    return OG.gemm_full(OG.dequant_mxfp8(qa, sa), OG.dequant_mxfp8(qb, sb), False, 8192, 8192, 8192)


@pytest.mark.parametrize("cfg", [pgt.CFG_AUTO, pgt.CFG_1CTA_128x256, pgt.CFG_2CTA_256x224])
def test_8192_mxfp8_full_matrix(ctx, big_mx, big_mx_oracle, cfg):
    """The MXFP8 benchmark workload: every output against the fp64 oracle, and work
    stealing bit-identical to the swizzled order."""
    M = N = K = 8192
    qa, sa, qb, sb = big_mx
    d = dev(qa, sa, qb, sb)
    C, plan, _ = run_mx(ctx, *d, M, N, K, cfg=cfg, mode=pgt.SWIZZLED, G=16)
    C64, Abs = big_mx_oracle
    OG.check(host_u16(C), C64, Abs)
    C2, _, _ = run_mx(ctx, *d, M, N, K, cfg=cfg, mode=pgt.WORK_STEALING, G=16)
    assert torch.equal(C, C2)


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (128, 16384, 1024), (2048, 2048, 2048), (8192, 8192, 8192),
                                   (3000, 5000, 1024)])
def test_auto_configuration_and_workspace_agree(ctx, M, N, K):
    """AUTO picks per shape among the 128-multiple tiles, whose packed-scale layout is the
    same, so the workspace size (queried without a context) fits whatever AUTO picks."""
    auto = pgt.make_desc(M, N, K, dtype=pgt.MXFP8, b_layout=pgt.B_NK)
    plan = ctx.gemm_plan(auto)
    assert plan["kernel_cfg"] in (pgt.CFG_1CTA_128x128, pgt.CFG_1CTA_128x256, pgt.CFG_2CTA_256x256)
    fixed = pgt.make_desc(M, N, K, dtype=pgt.MXFP8, b_layout=pgt.B_NK, kernel_cfg=plan["kernel_cfg"])
    assert ctx.gemm_workspace_bytes(auto) == ctx.gemm_workspace_bytes(fixed)


def test_mxfp8_argument_errors(ctx):
    t8 = torch.zeros((256, 256), dtype=torch.uint8, device="cuda")
    s8 = torch.full((256, 2), 127, dtype=torch.uint8, device="cuda")
    C = torch.zeros((256, 256), dtype=torch.int16, device="cuda")
    desc = pgt.make_desc(256, 256, 256, dtype=pgt.MXFP8, b_layout=pgt.B_NK)
    with pytest.raises(pgt.PgtError) as e:  # no workspace
        ctx.gemm_ex(desc, t8, t8, C, sfa=s8, sfb=s8)
    assert e.value.status == pgt.ERR_WORKSPACE
    ws = torch.zeros(ctx.gemm_workspace_bytes(desc), dtype=torch.uint8, device="cuda")
    with pytest.raises(pgt.PgtError) as e:  # no scales
        ctx.gemm_ex(desc, t8, t8, C, workspace=ws)
    assert e.value.status == pgt.ERR_ARG
    with pytest.raises(pgt.PgtError) as e:  # K not a multiple of 128
        ctx.gemm_ex(pgt.make_desc(256, 256, 192, dtype=pgt.MXFP8, b_layout=pgt.B_NK), t8, t8, C, sfa=s8, sfb=s8,
                    workspace=ws)
    assert e.value.status == pgt.ERR_ARG
