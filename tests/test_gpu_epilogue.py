"""GPU parity for the fused GEMM epilogue C = alpha * (A . B) + bias[n] against
oracle.gemm.epilogue (exact on closed forms, the GEMM bars on random data)."""
import numpy as np
import pytest
import torch

import persistent_gemm_tile_gb300 as pgt
import synthetic
from gpu_helpers import dev_u8, dev_u16, host_u16, need_gpu
from oracle import gemm as OG
from oracle import numerics as NM

pytestmark = pytest.mark.gpu

CFGS = [pgt.CFG_1CTA_128x128, pgt.CFG_1CTA_128x256, pgt.CFG_2CTA_256x128, pgt.CFG_2CTA_256x256]


@pytest.fixture(scope="module")
def ctx():
    need_gpu()
    c = pgt.Context(0)
    yield c
    c.close()


def gemm(ctx, A, B, M, N, K, cfg, alpha=None, bias=None, mode=pgt.SWIZZLED):
    desc = pgt.make_desc(M, N, K, kernel_cfg=cfg, sched_mode=mode, alpha=alpha, bias=bias)
    C = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
    ctx.gemm_ex(desc, A, B, C)
    torch.cuda.synchronize()
    assert ctx.last_error()[0] == 0
    return host_u16(C)


@pytest.mark.parametrize("cfg", CFGS)
def test_all_ones_scale_and_bias_exact(ctx, cfg):
    M, N, K = 256, 512, 256
    one = np.uint16(0x3F80)
    A = dev_u16(np.full((M, K), one, np.uint16))
    B = dev_u16(np.full((K, N), one, np.uint16))
    bias = (np.arange(N) % 17 - 8).astype(np.float32) * 0.5
    c = gemm(ctx, A, B, M, N, K, cfg, alpha=0.25, bias=torch.from_numpy(bias).cuda())
    expect = NM.f64_to_bf16_rne(0.25 * K + bias.astype(np.float64))
    assert np.array_equal(c, np.tile(expect, (M, 1)))


@pytest.mark.parametrize("cfg", CFGS)
@pytest.mark.parametrize("alpha,use_bias", [(-1.5, True), (None, True), (0.75, False)])
def test_random_scale_bias_ragged(ctx, cfg, alpha, use_bias):
    M, N, K = 1000, 1104, 512  # N is not a multiple of any tile width: bias reads must stop at N
    A, B = synthetic.gemm_bf16_inputs(M, N, K, seed=41)
    bias = np.random.default_rng(42).uniform(-3, 3, N).astype(np.float32) if use_bias else None
    c = gemm(ctx, dev_u16(A), dev_u16(B), M, N, K, cfg, alpha=alpha,
             bias=torch.from_numpy(bias).cuda() if use_bias else None)
    C64, Abs = OG.gemm_full(OG.dequant_bf16(A), OG.dequant_bf16(B), True, M, N, K)
    Ce, Ae = OG.epilogue(C64, Abs, 1.0 if alpha is None else alpha, bias)
    OG.check(c, Ce, Ae)


@pytest.mark.parametrize("cfg", [pgt.CFG_AUTO, pgt.CFG_2CTA_256x224])
def test_mxfp8_with_scale_and_bias(ctx, cfg):
    M, N, K = 512, 872, 1024  # 872 = 3 * 224 + 200: the last 224-column tile's 32-column tail holds 8
    qa, sa, qb, sb = synthetic.gemm_mxfp8_inputs(M, N, K, seed=43)
    bias = np.random.default_rng(44).uniform(-2, 2, N).astype(np.float32)
    dbias = torch.from_numpy(bias).cuda()  # the descriptor holds only its address: keep it alive
    desc = pgt.make_desc(M, N, K, dtype=pgt.MXFP8, b_layout=pgt.B_NK, alpha=0.5, bias=dbias, kernel_cfg=cfg)
    ws = torch.zeros(ctx.gemm_workspace_bytes(desc), dtype=torch.uint8, device="cuda")
    C = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
    ctx.gemm_ex(desc, dev_u8(qa), dev_u8(qb), C, sfa=dev_u8(sa), sfb=dev_u8(sb), workspace=ws)
    torch.cuda.synchronize()
    assert ctx.last_error()[0] == 0
    C64, Abs = OG.gemm_full(OG.dequant_mxfp8(qa, sa), OG.dequant_mxfp8(qb, sb), False, M, N, K)
    Ce, Ae = OG.epilogue(C64, Abs, 0.5, bias)
    OG.check(host_u16(C), Ce, Ae)


def test_epilogue_argument_errors(ctx):
    t = torch.zeros((64, 64), dtype=torch.int16, device="cuda")
    desc = pgt.make_desc(64, 64, 64)
    desc.epilogue = pgt.EPI_BIAS  # bias flag without a bias pointer
    with pytest.raises(pgt.PgtError) as e:
        ctx.gemm_ex(desc, t, t, t)
    assert e.value.status == pgt.ERR_ARG
    desc.epilogue = 4  # unknown flag
    with pytest.raises(pgt.PgtError) as e:
        ctx.gemm_ex(desc, t, t, t)
    assert e.value.status == pgt.ERR_ARG
