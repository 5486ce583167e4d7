"""The allocation-free GEMM entry point (pgt_gemm_noalloc), called through the C ABI.

It serves callers that cannot allocate device memory (allocator hooks, pre-budgeted
plugins, real-time paths), so its scratch is a static array inside the library.  Its
output must match the regular entry point's work-stealing GEMM with the same counter
groups (the same kernel: the same bits) on two calls in a row, the second one reusing the
array the first left behind.  This file is named to be collected last."""
import os
import subprocess
import sys

import pytest
import torch

import persistent_gemm_tile_gb300 as pgt
import synthetic
from gpu_helpers import dev_u16, host_u16, need_gpu
from oracle import gemm as OG

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
M, N, K = 1000, 1104, 512


@pytest.fixture(scope="module")
def problem():
    need_gpu()
    A, B = synthetic.gemm_bf16_inputs(M, N, K, seed=21)
    C64, Abs = OG.gemm_full(OG.dequant_bf16(A), OG.dequant_bf16(B), True, M, N, K)
    ctx = pgt.Context(0, max_groups=pgt.NOALLOC_MAX_GROUPS)
    yield dev_u16(A), dev_u16(B), C64, Abs, ctx
    ctx.close()


@pytest.mark.parametrize("with_err", [True, False])
@pytest.mark.parametrize("ws_groups", [0, 1, pgt.NOALLOC_MAX_GROUPS])
def test_noalloc_matches_regular_entry_point_on_two_calls(problem, ws_groups, with_err):
    """ws_groups 0 (eight groups), 1, and the largest count, whose last counter line sits
    next to the done counter; with a caller error word and without one (then the array's
    own error line is cleared as well)."""
    dA, dB, C64, Abs, ctx = problem
    lib = pgt.lib()
    desc = pgt.make_desc(M, N, K, b_layout=pgt.B_KN, sched_mode=pgt.WORK_STEALING, group_size=16,
                         ws_groups=ws_groups)
    ref = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
    ctx.gemm_ex(desc, dA, dB, ref)
    torch.cuda.synchronize()
    assert ctx.last_error()[0] == 0
    OG.check(host_u16(ref), C64, Abs)
    err = torch.zeros(4, dtype=torch.int32, device="cuda") if with_err else None
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        C = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
        rc = lib.pgt_gemm_noalloc(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), M, N, K, pgt.B_KN, 16, ws_groups,
                                  err.data_ptr() if with_err else None, stream)
        assert rc == pgt.OK, pgt.strerror(rc)
        torch.cuda.synchronize()
        if with_err:
            assert torch.count_nonzero(err).item() == 0, err.tolist()
        assert torch.equal(C, ref), f"call {call} differs from pgt_gemm_ex"


def test_noalloc_rejects_groups_beyond_its_scratch():
    need_gpu()
    t = torch.zeros((64, 64), dtype=torch.int16, device="cuda")
    with pytest.raises(pgt.PgtError) as e:
        pgt.gemm_noalloc(t, t, t, 64, 64, 64, ws_groups=pgt.NOALLOC_MAX_GROUPS + 1)
    assert e.value.status == pgt.ERR_GROUPS


_FIRST_CALL_UNDER_CAPTURE = r"""
import sys, torch
sys.path.insert(0, sys.argv[1])
import persistent_gemm_tile_gb300 as pgt
lib = pgt.lib()
a = torch.zeros((256, 256), dtype=torch.int16, device="cuda")
c = torch.zeros((256, 256), dtype=torch.int16, device="cuda")
s = torch.cuda.Stream()
g = torch.cuda.CUDAGraph()
with torch.cuda.graph(g, stream=s):
    rc_captured = lib.pgt_gemm_noalloc(a.data_ptr(), a.data_ptr(), c.data_ptr(), 256, 256, 256, pgt.B_KN, 16, 8,
                                       None, s.cuda_stream)
rc_after = lib.pgt_gemm_noalloc(a.data_ptr(), a.data_ptr(), c.data_ptr(), 256, 256, 256, pgt.B_KN, 16, 8, None,
                                torch.cuda.current_stream().cuda_stream)
torch.cuda.synchronize()
print("rc", rc_captured, rc_after)
"""


def test_first_call_under_capture_is_refused():
    """In a fresh process (so that this is the first call on the device), a call made while
    its stream is capturing returns PGT_ERR_ARG and enqueues nothing; the next call outside
    the capture does the set-up and runs."""
    need_gpu()
    r = subprocess.run([sys.executable, "-c", _FIRST_CALL_UNDER_CAPTURE, ROOT], capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert f"rc {pgt.ERR_ARG} {pgt.OK}" in r.stdout, r.stdout + r.stderr
