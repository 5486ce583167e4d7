"""Python binding of libpgt.so: the GB300 persistent tiled GEMM, its tile schedulers and
the persistent elementwise add.

Argument marshalling only: every step of the computation runs in the library's CUDA
kernels.  Function and argument names mirror ``include/pgt.h``.  Tensors may be torch
tensors (their ``data_ptr()`` is passed) or raw integer addresses; streams default to
torch's current CUDA stream.  The library must have been built (``__graft_entry__.build()``
or ``python -m persistent_gemm_tile_gb300._build``); nothing here falls back to any other
implementation.
"""
from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpgt.so")

# ------------------------------------------------------------------ constants (pgt.h)
OK = 0
ERR_ARG, ERR_ALIGN, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_GROUPS, ERR_WORKSPACE, ERR_CAPACITY = (
    -1, -2, -3, -4, -5, -6, -7, -8)
BF16, MXFP8 = 0, 1
B_KN, B_NK = 0, 1
BLOCKED, INTERLEAVED, SWIZZLED, WORK_STEALING, BLOCKED_GROUPED_M, LAUNCH_CONTROL = 0, 1, 2, 3, 4, 5
SCHED = {"blocked": BLOCKED, "interleaved": INTERLEAVED, "swizzled": SWIZZLED,
         "work_stealing": WORK_STEALING, "blocked_grouped_m": BLOCKED_GROUPED_M, "launch_control": LAUNCH_CONTROL}
CFG_AUTO, CFG_1CTA_128x128, CFG_1CTA_128x256, CFG_2CTA_256x128, CFG_2CTA_256x256 = 0, 1, 2, 3, 4
CFG_2CTA_256x224 = 5  # MXFP8 only
WS_RANGES, WS_STRIPED = 0, 1
FLAG_HOST_RESET = 1
EPI_ALPHA, EPI_BIAS = 1, 2
VISIT_FIELDS = 4

# every symbol include/pgt.h declares
EXPORTS = (
    "pgt_preamble", "pgt_destroy", "pgt_num_sms", "pgt_max_groups", "pgt_last_error", "pgt_strerror",
    "pgt_gemm_workspace_bytes", "pgt_gemm_plan", "pgt_gemm_ex", "pgt_gemm", "pgt_gemm_host",
    "pgt_add", "pgt_add_workers", "pgt_schedule_log", "pgt_gemm_noalloc", "pgt_multi_loop", "pgt_set_release",
    "pgt_wait_probe",
)
MAX_SPACES = 8
NOALLOC_MAX_GROUPS = 16


class GemmDesc(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("lda", ctypes.c_int64), ("ldb", ctypes.c_int64), ("ldc", ctypes.c_int64),
                ("dtype", ctypes.c_int32), ("b_layout", ctypes.c_int32), ("sched_mode", ctypes.c_int32),
                ("group_size", ctypes.c_int32), ("ws_groups", ctypes.c_int32), ("kernel_cfg", ctypes.c_int32),
                ("num_workers", ctypes.c_int32), ("epilogue", ctypes.c_int32), ("alpha", ctypes.c_float),
                ("ws_layout", ctypes.c_int32), ("bias", ctypes.c_void_p)]


class PlanInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "kernel_cfg", "bm", "bn", "bk", "cluster_size", "stages", "m_blocks", "n_blocks", "m_tiles",
        "tiles", "workers", "ctas", "k_iters", "smem_bytes", "ws_groups")]

    def as_dict(self) -> dict:
        return {n: getattr(self, n) for n, _ in self._fields_}


class Trace(ctypes.Structure):
    _fields_ = [("visits", ctypes.c_void_p), ("max_visits", ctypes.c_int64),
                ("counts", ctypes.c_void_p), ("times_ns", ctypes.c_void_p)]


class ScaleSpace(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("out", ctypes.c_void_p), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("ldx", ctypes.c_int64), ("ldo", ctypes.c_int64), ("scale", ctypes.c_float),
                ("reserved", ctypes.c_int32)]


class PgtError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        super().__init__(f"{where}: {strerror(status)} ({status})" if where else f"{strerror(status)} ({status})")


_lib = None


def lib() -> ctypes.CDLL:
    """Load libpgt.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() (nvcc, sm_103a)")
        L = ctypes.CDLL(LIB_PATH)
        P, I, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        L.pgt_preamble.argtypes = [I, I, I, ctypes.POINTER(P)]
        L.pgt_destroy.argtypes = [P]
        L.pgt_num_sms.argtypes = [P]
        L.pgt_max_groups.argtypes = [P]
        L.pgt_last_error.argtypes = [P, P, P]
        L.pgt_strerror.argtypes = [I]
        L.pgt_strerror.restype = ctypes.c_char_p
        L.pgt_gemm_workspace_bytes.argtypes = [P]
        L.pgt_gemm_workspace_bytes.restype = SZ
        L.pgt_gemm_plan.argtypes = [P, P, P]
        L.pgt_gemm_ex.argtypes = [P, P, P, P, P, P, P, P, SZ, P, P]
        L.pgt_gemm.argtypes = [P, P, P, P, P, P, I64, I64, I64, I, I, I, I, I, P, SZ, P]
        L.pgt_gemm_host.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, P, SZ, P]
        L.pgt_add.argtypes = [P, P, P, P, I64, I64, I64, I64, I64, I, I, I, I, P, P]
        L.pgt_add_workers.argtypes = [P, I64, I64, I, I, I, I]
        L.pgt_schedule_log.argtypes = [P, I64, I64, I, I, I, I, I, I, P, P]
        L.pgt_gemm_noalloc.argtypes = [P, P, P, I64, I64, I64, I, I, I, P, P]
        L.pgt_multi_loop.argtypes = [P, P, I, I, I, I, I, P, P]
        L.pgt_set_release.argtypes = [P, P, I, P]
        L.pgt_wait_probe.argtypes = [P, I, P]
        _lib = L
    return _lib


def strerror(status: int) -> str:
    try:
        return lib().pgt_strerror(int(status)).decode()
    except RuntimeError:
        return f"status {status}"


def _check(rc: int, where: str) -> int:
    if rc < 0:
        raise PgtError(rc, where)
    return rc


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_desc(M, N, K, *, lda=0, ldb=0, ldc=0, dtype=BF16, b_layout=B_KN, sched_mode=SWIZZLED,
              group_size=16, ws_groups=0, kernel_cfg=CFG_AUTO, num_workers=0, alpha=None, bias=None,
              ws_layout=WS_RANGES) -> GemmDesc:
    """A pgt_gemm_desc; alpha (a_scale * b_scale) and bias (device fp32[N]) enable the epilogue.

    The descriptor stores only the bias tensor's address: keep the tensor alive until the
    GEMMs that use this descriptor have finished."""
    if isinstance(sched_mode, str):
        sched_mode = SCHED[sched_mode]
    epi = (EPI_ALPHA if alpha is not None else 0) | (EPI_BIAS if bias is not None else 0)
    return GemmDesc(M, N, K, lda, ldb, ldc, dtype, b_layout, sched_mode, group_size, ws_groups, kernel_cfg,
                    num_workers, epi, 1.0 if alpha is None else float(alpha), ws_layout, _ptr(bias))


def gemm_noalloc(A, B, C, M, N, K, b_layout=B_KN, group_size=16, ws_groups=0, err=None, stream=None) -> None:
    """pgt_gemm_noalloc: the work-stealing bf16 GEMM on the current device for callers that
    cannot allocate device memory (its scratch is a static array inside the library)."""
    _check(lib().pgt_gemm_noalloc(_ptr(A), _ptr(B), _ptr(C), M, N, K, b_layout, group_size, ws_groups, _ptr(err),
                                  _stream(stream)), "pgt_gemm_noalloc")


class Context:
    """A pgt context (pgt_preamble): SM count plus the preallocated work-stealing counters."""

    def __init__(self, device: int = 0, max_groups: int = 8, flags: int = 0):
        h = ctypes.c_void_p()
        _check(lib().pgt_preamble(device, max_groups, flags, ctypes.byref(h)), "pgt_preamble")
        self.handle = h.value
        self.device = device

    def close(self):
        if getattr(self, "handle", None):
            lib().pgt_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_release(self, flags, stream=None) -> None:
        """pgt_set_release: raise (nonzero) or clear the per-group release flags."""
        import numpy as np
        arr = np.ascontiguousarray(flags, dtype=np.int32)
        self._release_host = arr  # the copy is asynchronous: keep the host buffer alive
        _check(lib().pgt_set_release(self.handle, arr.ctypes.data, arr.size, _stream(stream)), "pgt_set_release")

    @property
    def num_sms(self) -> int:
        return _check(lib().pgt_num_sms(self.handle), "pgt_num_sms")

    @property
    def max_groups(self) -> int:
        return _check(lib().pgt_max_groups(self.handle), "pgt_max_groups")

    def last_error(self, stream=None):
        detail = (ctypes.c_int32 * 4)()
        rc = lib().pgt_last_error(self.handle, _stream(stream), ctypes.cast(detail, ctypes.c_void_p))
        return rc, list(detail)

    def wait_probe(self, arrive: bool, stream=None) -> None:
        """pgt_wait_probe: exercise the bounded-wait path (arrive=False makes it time out)."""
        _check(lib().pgt_wait_probe(self.handle, int(bool(arrive)), _stream(stream)), "pgt_wait_probe")

    def gemm_plan(self, desc: GemmDesc) -> dict:
        info = PlanInfo()
        _check(lib().pgt_gemm_plan(self.handle, ctypes.byref(desc), ctypes.byref(info)), "pgt_gemm_plan")
        return info.as_dict()

    @staticmethod
    def gemm_workspace_bytes(desc: GemmDesc) -> int:
        return lib().pgt_gemm_workspace_bytes(ctypes.byref(desc))

    def gemm_ex(self, desc: GemmDesc, A, B, C, sfa=None, sfb=None, workspace=None, workspace_bytes=0,
                trace: Trace | None = None, stream=None) -> None:
        if workspace is not None and not workspace_bytes:
            workspace_bytes = workspace.numel() * workspace.element_size()
        _check(lib().pgt_gemm_ex(self.handle, ctypes.byref(desc), _ptr(A), _ptr(B), _ptr(sfa), _ptr(sfb), _ptr(C),
                                 _ptr(workspace), workspace_bytes, ctypes.byref(trace) if trace else None,
                                 _stream(stream)), "pgt_gemm_ex")

    def gemm(self, A, B, C, M, N, K, dtype=BF16, b_layout=B_KN, sched_mode=SWIZZLED, group_size=16, ws_groups=0,
             sfa=None, sfb=None, workspace=None, workspace_bytes=0, stream=None) -> None:
        """pgt_gemm, the flat form: packed operands, automatic kernel configuration."""
        if isinstance(sched_mode, str):
            sched_mode = SCHED[sched_mode]
        if workspace is not None and not workspace_bytes:
            workspace_bytes = workspace.numel() * workspace.element_size()
        _check(lib().pgt_gemm(self.handle, _ptr(A), _ptr(B), _ptr(sfa), _ptr(sfb), _ptr(C), M, N, K, dtype,
                              b_layout, sched_mode, group_size, ws_groups, _ptr(workspace), workspace_bytes,
                              _stream(stream)), "pgt_gemm")

    def gemm_host(self, desc: GemmDesc, hA, hB, hC, dA, dB, dC, h_sfa=None, h_sfb=None, d_sfa=None, d_sfb=None,
                  workspace=None, workspace_bytes=0, stream=None) -> None:
        if workspace is not None and not workspace_bytes:
            workspace_bytes = workspace.numel() * workspace.element_size()
        _check(lib().pgt_gemm_host(self.handle, ctypes.byref(desc), _ptr(hA), _ptr(hB), _ptr(h_sfa), _ptr(h_sfb),
                                   _ptr(hC), _ptr(dA), _ptr(dB), _ptr(d_sfa), _ptr(d_sfb), _ptr(dC),
                                   _ptr(workspace), workspace_bytes, _stream(stream)), "pgt_gemm_host")

    def add(self, x, y, out, rows=None, cols=None, ldx=0, ldy=0, ldo=0, sched_mode=BLOCKED, tile_r=0, tile_c=0,
            num_workers=0, trace: Trace | None = None, stream=None) -> None:
        if isinstance(sched_mode, str):
            sched_mode = SCHED[sched_mode]
        if rows is None:
            rows, cols = x.shape
            ldx, ldy, ldo = x.stride(0), y.stride(0), out.stride(0)
        _check(lib().pgt_add(self.handle, _ptr(x), _ptr(y), _ptr(out), rows, cols, ldx, ldy, ldo, sched_mode,
                             tile_r, tile_c, num_workers, ctypes.byref(trace) if trace else None,
                             _stream(stream)), "pgt_add")

    def multi_loop(self, spaces, sched_mode=BLOCKED, tile_r=0, tile_c=0, num_workers=0,
                   trace: Trace | None = None, stream=None) -> None:
        """pgt_multi_loop over [(x, out, scale), ...] 2-D fp32 tensors: out = scale * x."""
        if isinstance(sched_mode, str):
            sched_mode = SCHED[sched_mode]
        arr = (ScaleSpace * len(spaces))()
        for i, (x, out, scale) in enumerate(spaces):
            arr[i] = ScaleSpace(_ptr(x), _ptr(out), x.shape[0], x.shape[1], x.stride(0), out.stride(0),
                                float(scale), 0)
        _check(lib().pgt_multi_loop(self.handle, ctypes.cast(arr, ctypes.c_void_p), len(spaces), sched_mode, tile_r,
                                    tile_c, num_workers, ctypes.byref(trace) if trace else None, _stream(stream)),
               "pgt_multi_loop")

    def add_workers(self, rows, cols, tile_r=0, tile_c=0, num_workers=0, sched_mode=BLOCKED) -> int:
        if isinstance(sched_mode, str):
            sched_mode = SCHED[sched_mode]
        return _check(lib().pgt_add_workers(self.handle, rows, cols, tile_r, tile_c, sched_mode, num_workers),
                      "pgt_add_workers")

    def schedule_log(self, m_blocks, n_blocks, cluster_size, sched_mode, group_size, ws_groups, num_workers,
                     trace: Trace, stream=None, ws_layout=WS_RANGES) -> None:
        if isinstance(sched_mode, str):
            sched_mode = SCHED[sched_mode]
        _check(lib().pgt_schedule_log(self.handle, m_blocks, n_blocks, cluster_size, sched_mode, group_size,
                                      ws_groups, ws_layout, num_workers, ctypes.byref(trace), _stream(stream)),
               "pgt_schedule_log")


class TraceBuffers:
    """Device buffers for a traced launch (torch-allocated), and their decoding."""

    def __init__(self, ctas: int, max_visits: int, device="cuda"):
        import torch
        self.ctas, self.max_visits = ctas, max_visits
        self.visits = torch.full((ctas, max_visits, VISIT_FIELDS), -1, dtype=torch.int32, device=device)
        self.counts = torch.full((ctas,), -1, dtype=torch.int32, device=device)
        self.times = torch.zeros((ctas, 2), dtype=torch.int64, device=device)
        self.struct = Trace(self.visits.data_ptr(), max_visits, self.counts.data_ptr(), self.times.data_ptr())

    def read(self):
        """Per CTA: list of (tile_id, m_idx, n_idx, smid) in visit order; plus times (ns)."""
        v = self.visits.cpu().numpy()
        c = self.counts.cpu().numpy()
        out = []
        for i in range(self.ctas):
            n = int(c[i])
            if n > self.max_visits:
                raise PgtError(ERR_CAPACITY, "trace")
            out.append([tuple(int(x) for x in v[i, j]) for j in range(max(n, 0))])
        return out, self.times.cpu().numpy()
