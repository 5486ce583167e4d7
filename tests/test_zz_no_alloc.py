"""The allocation-free GEMM entry point (pgt_gemm_noalloc), called through the C ABI.

It serves callers that cannot allocate device memory (allocator hooks, pre-budgeted
plugins, real-time paths), so its scratch is a static array inside the library.  Its
output must match the regular entry point's work-stealing GEMM (the same kernel: the same
bits) on two calls in a row, the second one reusing the array the first left behind.
This file is named to be collected last."""
import numpy as np
import pytest
import torch

import persistent_gemm_tile_gb300 as pgt
import synthetic
from gpu_helpers import dev_u16, host_u16, need_gpu
from oracle import gemm as OG

pytestmark = pytest.mark.gpu


def test_noalloc_matches_regular_entry_point_on_two_calls():
    need_gpu()
    lib = pgt.lib()
    M, N, K = 1000, 1104, 512
    A, B = synthetic.gemm_bf16_inputs(M, N, K, seed=21)
    dA, dB = dev_u16(A), dev_u16(B)
    ctx = pgt.Context(0)
    desc = pgt.make_desc(M, N, K, b_layout=pgt.B_KN, sched_mode=pgt.WORK_STEALING, group_size=16, ws_groups=8)
    ref = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
    ctx.gemm_ex(desc, dA, dB, ref)
    torch.cuda.synchronize()
    assert ctx.last_error()[0] == 0
    C64, Abs = OG.gemm_full(OG.dequant_bf16(A), OG.dequant_bf16(B), True, M, N, K)
    OG.check(host_u16(ref), C64, Abs)
    err = torch.zeros(4, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        C = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
        rc = lib.pgt_gemm_noalloc(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), M, N, K, pgt.B_KN, 16, 8,
                                  err.data_ptr(), stream)
        assert rc == pgt.OK, pgt.strerror(rc)
        torch.cuda.synchronize()
        assert torch.count_nonzero(err).item() == 0, err.tolist()
        OG.check(host_u16(C), C64, Abs)
        assert torch.equal(C, ref), f"call {call} differs from pgt_gemm_ex"
    ctx.close()


def test_noalloc_rejects_groups_beyond_its_scratch():
    need_gpu()
    t = torch.zeros((64, 64), dtype=torch.int16, device="cuda")
    with pytest.raises(pgt.PgtError) as e:
        pgt.gemm_noalloc(t, t, t, 64, 64, 64, ws_groups=pgt.NOALLOC_MAX_GROUPS + 1)
    assert e.value.status == pgt.ERR_GROUPS
