"""Host-only checks of the C ABI: the library builds and loads, exports every function
include/pgt.h declares, and the binding's constants agree with the header's."""
import ctypes
import os
import re

import pytest

import persistent_gemm_tile_gb300 as pgt
from persistent_gemm_tile_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pgt.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return pgt.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pgt_[a-z_0-9]+)\s*\(", text)))


def _defines():
    out = {}
    for name, val in re.findall(r"#define\s+(PGT_[A-Za-z0-9_]+)\s+\(?(-?\d+)\)?", open(HEADER).read()):
        out[name] = int(val)
    return out


def test_every_declared_symbol_is_exported(lib):
    declared = _declared_functions()
    assert len(declared) >= 14
    assert set(declared) == set(pgt.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def test_binding_constants_match_header():
    d = _defines()
    pairs = {
        "PGT_OK": pgt.OK, "PGT_ERR_ARG": pgt.ERR_ARG, "PGT_ERR_ALIGN": pgt.ERR_ALIGN,
        "PGT_ERR_UNSUPPORTED": pgt.ERR_UNSUPPORTED, "PGT_ERR_CUDA": pgt.ERR_CUDA,
        "PGT_ERR_TIMEOUT": pgt.ERR_TIMEOUT, "PGT_ERR_GROUPS": pgt.ERR_GROUPS,
        "PGT_ERR_WORKSPACE": pgt.ERR_WORKSPACE, "PGT_ERR_CAPACITY": pgt.ERR_CAPACITY,
        "PGT_BF16": pgt.BF16, "PGT_MXFP8": pgt.MXFP8, "PGT_B_KN": pgt.B_KN, "PGT_B_NK": pgt.B_NK,
        "PGT_BLOCKED": pgt.BLOCKED, "PGT_INTERLEAVED": pgt.INTERLEAVED, "PGT_SWIZZLED": pgt.SWIZZLED,
        "PGT_WORK_STEALING": pgt.WORK_STEALING, "PGT_BLOCKED_GROUPED_M": pgt.BLOCKED_GROUPED_M,
        "PGT_LAUNCH_CONTROL": pgt.LAUNCH_CONTROL,
        "PGT_CFG_AUTO": pgt.CFG_AUTO, "PGT_CFG_1CTA_128x128": pgt.CFG_1CTA_128x128,
        "PGT_CFG_1CTA_128x256": pgt.CFG_1CTA_128x256, "PGT_CFG_2CTA_256x128": pgt.CFG_2CTA_256x128,
        "PGT_CFG_2CTA_256x256": pgt.CFG_2CTA_256x256, "PGT_CFG_2CTA_256x224": pgt.CFG_2CTA_256x224,
        "PGT_FLAG_HOST_RESET": pgt.FLAG_HOST_RESET, "PGT_WS_RANGES": pgt.WS_RANGES, "PGT_WS_STRIPED": pgt.WS_STRIPED,
        "PGT_VISIT_FIELDS": pgt.VISIT_FIELDS, "PGT_NOALLOC_MAX_GROUPS": pgt.NOALLOC_MAX_GROUPS,
        "PGT_EPI_ALPHA": pgt.EPI_ALPHA, "PGT_EPI_BIAS": pgt.EPI_BIAS, "PGT_MAX_SPACES": pgt.MAX_SPACES,
    }
    for k, v in pairs.items():
        assert d[k] == v, k


def test_struct_sizes_match_c_layout():
    assert ctypes.sizeof(pgt.GemmDesc) == 6 * 8 + 10 * 4 + 8
    assert ctypes.sizeof(pgt.PlanInfo) == 15 * 4
    assert ctypes.sizeof(pgt.Trace) == 32
    assert ctypes.sizeof(pgt.ScaleSpace) == 2 * 8 + 4 * 8 + 8


def test_strerror_names_every_status(lib):
    for st in range(0, -9, -1):
        assert pgt.strerror(st) != "unknown status"
    assert pgt.strerror(-100) == "unknown status"


def test_null_arguments_rejected_without_touching_a_gpu(lib):
    assert lib.pgt_preamble(0, 8, 0, None) == pgt.ERR_ARG
    assert lib.pgt_num_sms(None) == pgt.ERR_ARG
    assert lib.pgt_destroy(None) == pgt.OK
    assert lib.pgt_gemm_plan(None, None, None) == pgt.ERR_ARG
    assert lib.pgt_gemm_workspace_bytes(None) == 0
    h = ctypes.c_void_p()
    assert lib.pgt_preamble(0, 0, 0, ctypes.byref(h)) == pgt.ERR_ARG  # max_groups < 1
    assert lib.pgt_preamble(0, 65, 0, ctypes.byref(h)) == pgt.ERR_ARG
    assert lib.pgt_preamble(0, 8, 4, ctypes.byref(h)) == pgt.ERR_ARG  # unknown flag


def test_flat_gemm_checks_counter_groups_first(lib):
    """pgt_gemm's ws_groups must lie in [0, 64] whatever the context; a valid count with no
    context is an argument error."""
    def flat(ws_groups):
        return lib.pgt_gemm(None, None, None, None, None, None, 64, 64, 64, pgt.BF16, pgt.B_KN, pgt.WORK_STEALING,
                            16, ws_groups, None, 0, None)
    assert flat(65) == pgt.ERR_GROUPS
    assert flat(-1) == pgt.ERR_GROUPS
    assert flat(0) == pgt.ERR_ARG
    assert flat(64) == pgt.ERR_ARG


def test_mxfp8_workspace_bytes_per_configuration(lib):
    """Packed-scale workspace: k groups of four 128-wide K blocks x (A blocks + B blocks) x
    512 bytes.  A and B use 128-row blocks rounded up to even counts, except that for the
    224-column pair tile B's blocks are cut per tile (two per 224-row tile)."""
    def ws(M, N, K, cfg):
        d = pgt.make_desc(M, N, K, dtype=pgt.MXFP8, b_layout=pgt.B_NK, kernel_cfg=cfg)
        return lib.pgt_gemm_workspace_bytes(ctypes.byref(d))
    even = lambda v: (v + 1) // 2 * 2  # noqa: E731
    for M, N, K in ((8192, 8192, 8192), (1000, 1100, 1664), (128, 224, 128), (384, 448, 512)):
        kg = (K // 128 + 3) // 4
        ma = even(-(-M // 128))
        for cfg in (pgt.CFG_AUTO, pgt.CFG_1CTA_128x128, pgt.CFG_2CTA_256x256):
            assert ws(M, N, K, cfg) == kg * (ma + even(-(-N // 128))) * 512, (M, N, K, cfg)
        assert ws(M, N, K, pgt.CFG_2CTA_256x224) == kg * (ma + 2 * -(-N // 224)) * 512, (M, N, K)
    assert ws(8192, 8192, 8192, 99) == 0  # unknown configuration
    d = pgt.make_desc(256, 256, 256, kernel_cfg=pgt.CFG_2CTA_256x224)  # bf16 needs none
    assert lib.pgt_gemm_workspace_bytes(ctypes.byref(d)) == 0


def test_oracle_and_library_share_no_code():
    """The CUDA path never imports the oracle, and the oracle never imports the package."""
    root = os.path.dirname(os.path.dirname(HEADER))
    pkg = os.path.join(root, "persistent_gemm_tile_gb300")
    imp_oracle = re.compile(r"^\s*(import|from)\s+oracle\b|#include\s+[<\"].*oracle", re.M)
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                assert not imp_oracle.search(open(os.path.join(dirpath, f)).read()), f
    imp_pkg = re.compile(r"^\s*(import|from)\s+persistent_gemm_tile_gb300\b|#include\s+[<\"]pgt", re.M)
    for f in os.listdir(os.path.join(root, "oracle")):
        if f.endswith((".py", ".c")):
            assert not imp_pkg.search(open(os.path.join(root, "oracle", f)).read()), f
