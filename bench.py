"""Benchmark of the persistent tiled GEMM and the persistent add on GB300.

Headline (``value``): bf16 GEMM C = A . B at M = N = K = 8192 (A, B ~ N(0,1)/sqrt(K), seed 2,
B stored K x N), swizzled scheduler with group_size 16, in TFLOP/s over the whole job.
One step = one GEMM launch through the C ABI.  The same run also reports, outside the
timed headline loop: TFLOP/s per scheduler mode, the persistent add's GB/s on fp32
8192 x 8192 (seed 1), tail idle per scheduler from traced launches, the end-to-end figure
from host memory, and the CPU oracle timed on a bounded sample.

``--impl reference`` times the CPU oracle (the benchmark's reference arm) on the same
workload and prints the same JSON line with ``"impl": "reference"``.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

M = N = K = 8192
FLOP = 2.0 * M * N * K
ADD_ROWS = ADD_COLS = 8192
ADD_BYTES = 12.0 * ADD_ROWS * ADD_COLS  # read x, read y, write out (fp32)
METRIC = "GEMM TFLOP/s & % tensor peak per scheduler mode; persistent add GB/s vs HBM"
WORKLOAD = "bf16 GEMM M=N=K=8192, A,B ~ N(0,1)/sqrt(K) seed 2, B stored KxN, swizzled group_size=16"
L2_NOTE = "inputs larger than L2: A+B+C = 384 MiB per GEMM > 129 MB L2; add x+y+out = 768 MiB"


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from one ncu capture
# of each kernel (summaries under profiles/).  A figure is reported only while the kernel's
# sources hash to the fingerprint taken with it (comments and blank lines left out, so an
# edit of comments alone keeps a capture); after any change of code the roofline says null.
GEMM_SOURCES = ["csrc/pgt_gemm_kernel.cuh", "csrc/pgt_device.cuh", "csrc/pgt_sched.cuh"]
ADD_SOURCES = ["csrc/pgt_add.cu", "csrc/pgt_device.cuh", "csrc/pgt_sched.cuh"]
PROFILED_TRAFFIC = {
    "gemm_bf16_2cta_256x256": (8.66333440e+08 + 1.27151360e+08, GEMM_SOURCES, "95db09673622310a"),
    "gemm_mxfp8_2cta_256x256": (2.47468288e+08 + 1.15645952e+08, GEMM_SOURCES, "95db09673622310a"),
    "add_wide_8x1024_blocked": (5.36939520e+08 + 2.31422720e+08, ADD_SOURCES, "ea072a4ea074ca89"),
    "add_wide_8x1024_interleaved": (5.36960768e+08 + 2.30933504e+08, ADD_SOURCES, "ea072a4ea074ca89"),
    "add_page_32x16_blocked": (5.36942848e+08 + 2.33459456e+08, ADD_SOURCES, "ea072a4ea074ca89"),
    "add_page_32x16_interleaved": (5.66916352e+08 + 2.37809920e+08, ADD_SOURCES, "ea072a4ea074ca89"),
}


def source_fingerprint(files) -> str:
    """First 16 hex digits of the sha256 of the kernel sources' code: every line up to a `//`
    comment, trailing blanks removed, empty lines dropped (the sources use no block
    comments and no `//` inside strings)."""
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "persistent_gemm_tile_gb300", f), encoding="utf-8") as fh:
            for line in fh:
                code = line.split("//", 1)[0].rstrip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def profiled_traffic(key: str):
    if key not in PROFILED_TRAFFIC:
        return None
    nbytes, files, fingerprint = PROFILED_TRAFFIC[key]
    return nbytes if source_fingerprint(files) == fingerprint else None


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cfg", type=int, default=0, help="kernel configuration (PGT_CFG_*), 0 = auto")
    ap.add_argument("--kernel", default="gemm", choices=["gemm", "add", "mxfp8", "ragged"],
                    help="headline kernel: the bf16 GEMM (default), or the persistent add / the MXFP8 GEMM "
                         "(for timing and profiling those kernels alone), or one launch per scheduler and "
                         "configuration of the ragged set (for profiling)")
    ap.add_argument("--no-extras", action="store_true", help="headline only")
    ap.add_argument("--sched", default="swizzled",
                    choices=["blocked", "interleaved", "swizzled", "work_stealing", "blocked_grouped_m",
                             "launch_control"], help="scheduler of the bf16 headline GEMM")
    ap.add_argument("--group", type=int, default=16, help="group_size of the bf16 headline GEMM")
    ap.add_argument("--ws-groups", type=int, default=8, help="work-stealing counter groups of the bf16 headline GEMM")
    ap.add_argument("--ws-layout", default="ranges", choices=["ranges", "striped"],
                    help="work-stealing tile ownership of the bf16 headline GEMM")
    ap.add_argument("--add-tile", default="wide", help="tile of the --kernel add headline: 'wide' (8x1024) or RxC, "
                                                         "e.g. 32x16 (the page's tile)")
    ap.add_argument("--add-sched", default="blocked", choices=["blocked", "interleaved"],
                    help="scheduler of the --kernel add headline")
    ap.add_argument("--cublas", action="store_true",
                    help="with --kernel mxfp8: also time cuBLAS's MXFP8 GEMM on the same operands after the "
                         "timed loop (for profiling the two side by side)")
    ap.add_argument("--no-ragged", action="store_true",
                    help="skip the ragged-tail GEMM set (timed per scheduler, with tail idle from traces)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU oracle sample budget")
    ap.add_argument("--size", type=int, default=8192,
                    help="M = N = K of the GEMM workloads (8192 is the benchmark; smaller sizes are for "
                         "quick checks and small profiling cases)")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_burst": p["bf16_tflops"],
                "bf16_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_burst": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


class NvmlClockReader:
    """Read-only NVML queries through ctypes (libnvidia-ml ships with the driver): the SM
    clock, its maximum and the active clock-event reasons of one device.  Nothing is set."""

    SM = 1  # NVML_CLOCK_SM
    # nvmlClocksEventReasons bits (NVML's public header)
    BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
            0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index: int, pci_bus_id: str | None = None):
        import ctypes
        self.ct = ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.lib = lib
        self.h = ctypes.c_void_p()
        rc = 1
        if pci_bus_id:
            rc = lib.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(), ctypes.byref(self.h))
        if rc != 0:
            rc = lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(device_index), ctypes.byref(self.h))
        if rc != 0:
            raise OSError("no NVML handle for the device")
        reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
        self.reasons_fn = reasons if reasons is not None else lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.max_mhz = self._clock(lib.nvmlDeviceGetMaxClockInfo)

    def _clock(self, fn):
        v = self.ct.c_uint(0)
        return float(v.value) if fn(self.h, self.SM, self.ct.byref(v)) == 0 else None

    def sample(self):
        """(SM MHz, max SM MHz, set of active reasons), or None if a query failed."""
        sm = self._clock(self.lib.nvmlDeviceGetClockInfo)
        bits = self.ct.c_ulonglong(0)
        if sm is None or self.reasons_fn(self.h, self.ct.byref(bits)) != 0:
            return None
        return sm, self.max_mhz, {n for b, n in self.BITS.items() if bits.value & b}


def summarize_clocks(rows, t_begin, t_end, period_ms, source):
    """rows: (host time, SM MHz, max MHz, active reasons).  The figures describe the samples
    taken between t_begin and t_end (the timed launches); *_around describe all of them."""
    inside = [r for r in rows if r[0] is not None and t_begin is not None and t_end is not None
              and t_begin <= r[0] <= t_end]

    def summary(rs):
        return (float(np.median([r[1] for r in rs])) if rs else None,
                sorted(set().union(*[r[3] for r in rs])) if rs else [])
    sm_in, reasons_in = summary(inside)
    sm_all, reasons_all = summary(rows)
    return {"sm_mhz": sm_in, "sm_max_mhz": max((r[2] for r in rows if r[2] is not None), default=None),
            "reasons": reasons_in, "samples": len(inside), "period_ms": period_ms, "source": source,
            "region_s": (t_end - t_begin) if t_begin and t_end else None,
            "sm_mhz_around": sm_all, "reasons_around": reasons_all, "samples_around": len(rows)}


class Clocks:
    """SM clocks and clock-event reasons sampled while the timed launches run.  NVML is
    polled every millisecond from a host thread (read-only queries); without NVML,
    nvidia-smi samples every ``period_ms``.  Samples carry host timestamps; ``stop`` keeps
    only those taken between ``begin()`` and ``end()`` (just before the first timed launch
    is enqueued and just after the last one has finished), so the figures describe the
    timed launches.  A region that holds no sample reports ``samples`` 0 and null figures,
    while ``*_around`` give the samples taken around it."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
    NVML_PERIOD_MS = 1

    def __init__(self, device_index: int, period_ms: int = 20, reader=None):
        self.dev = device_index
        self.period_ms = period_ms
        self.proc = None
        self.reader = reader
        self.thread = None
        self.rows = []
        self.t_begin = self.t_end = None
        self.path = os.path.join(tempfile.gettempdir(), f"pgt_clocks_{os.getpid()}.csv")

    def _open_reader(self):
        if self.reader is not None:
            return self.reader
        bus = None
        try:
            import torch
            pr = torch.cuda.get_device_properties(self.dev)
            if isinstance(getattr(pr, "pci_bus_id", None), int):
                bus = f"{getattr(pr, 'pci_domain_id', 0):08x}:{pr.pci_bus_id:02x}:{getattr(pr, 'pci_device_id', 0):02x}.0"
        except Exception:
            bus = None
        try:
            return NvmlClockReader(self.dev, bus)
        except (OSError, AttributeError):
            return None

    def _poll(self):
        while not self.stop_flag:
            smp = self.reader.sample()
            if smp is not None:
                self.rows.append((time.time(), *smp))
            time.sleep(self.NVML_PERIOD_MS / 1000.0)

    def start(self):
        self.reader = self._open_reader()
        if self.reader is not None:
            import threading
            self.stop_flag = False
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            time.sleep(0.02)
            return
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.15)
        except (OSError, FileNotFoundError):
            self.proc = None

    def begin(self):
        self.t_begin = time.time()

    def end(self):
        self.t_end = time.time()

    @staticmethod
    def _parse_time(text: str):
        import datetime
        try:
            return datetime.datetime.strptime(text.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def stop(self) -> dict:
        if self.thread is not None:
            time.sleep(0.02)
            self.stop_flag = True
            self.thread.join()
            return summarize_clocks(self.rows, self.t_begin, self.t_end, self.NVML_PERIOD_MS, "nvml")
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clock sampling unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        self.proc.wait()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    sm, smax = float(parts[2]), float(parts[3])
                except ValueError:
                    continue
                active = {n for n, v in zip(self.REASONS, parts[6:10]) if v.lower().startswith("active")}
                rows.append((self._parse_time(parts[0]), sm, smax, active))
        os.unlink(self.path)
        return summarize_clocks(rows, self.t_begin, self.t_end, self.period_ms, "nvidia-smi")


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        dist.init_process_group(backend=backend)
        pg = dist
    return world, rank, local, pg


def barrier(pg, torch=None):
    if pg is not None:
        pg.barrier()


def max_over_ranks(pg, value: float, device) -> float:
    if pg is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------- helpers
def time_launches(torch, launch, steps: int, warmup: int):
    """Run `warmup` untimed launches, then `steps` launches bracketed by CUDA events on the
    current stream; returns (total ms, list of per-launch ms)."""
    for _ in range(warmup):
        launch()
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    evs[0].record()
    for i in range(steps):
        launch()
        evs[i + 1].record()
    torch.cuda.synchronize()
    per = [evs[i].elapsed_time(evs[i + 1]) for i in range(steps)]
    return evs[0].elapsed_time(evs[-1]), per


def time_sustained(torch, launch, seconds: float, block: int = 50) -> list:
    """Launch back to back for about `seconds`, with CUDA events every `block` launches on
    the current stream; returns the mean per-launch ms of each block."""
    for _ in range(3):
        launch()
    torch.cuda.synchronize()
    out = []
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(block):
            launch()
        b.record()
        b.synchronize()
        out.append(a.elapsed_time(b) / block)
    return out


def time_protocol(torch, launch, flush, warmup: int = 10, reps: int = 50) -> list:
    """The measurement protocol of the benchmark plan: `warmup` untimed launches, then `reps`
    launches each bracketed by its own CUDA events on the current stream, with `flush` (a
    write larger than L2) before each one, outside the events.  Returns per-launch ms."""
    for _ in range(warmup):
        launch()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for a, b in evs:
        flush()
        a.record()
        launch()
        b.record()
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def tail_idle(times_ns: np.ndarray, slots: int | None = None) -> float:
    """1 - sum(busy) / (P * span): the share of worker time spent idle in the launch, over
    the workers that ran (under launch control most launched workers are cancelled before
    they start and record no times).  With `slots` (e.g. the SM count, one CTA per SM), the
    idle share of that many slots instead: the quantity ncu's 1 - sm__cycles_active.avg /
    sm__cycles_elapsed.max measures, SMs that ran no CTA counting as idle."""
    t = times_ns[(times_ns[:, 0] > 0) & (times_ns[:, 1] > 0)]
    if len(t) == 0:
        return float("nan")
    span = float(t[:, 1].max() - t[:, 0].min())
    n = len(t) if slots is None else slots
    return 1.0 - float((t[:, 1] - t[:, 0]).sum()) / (n * span) if span > 0 else 0.0


def cpu_baseline(budget_s: float, A_bits, B_bits, rows_hint: int | None = None) -> dict:
    """The CPU oracle, as it stands, on a bounded sample of rows of the same GEMM."""
    from oracle import gemm as OG
    cores = OG.num_threads()
    B64 = OG.dequant_bf16(B_bits)
    probe_rows = max(1, cores)
    A64 = OG.dequant_bf16(A_bits[:probe_rows])
    t0 = time.perf_counter()
    OG.gemm_rows(A64, B64, True, K, N, np.arange(probe_rows))
    t_probe = time.perf_counter() - t0
    rows = rows_hint or int(max(probe_rows, min(M, probe_rows * budget_s / max(t_probe, 1e-3))))
    rows = (rows // probe_rows) * probe_rows or probe_rows
    A64 = OG.dequant_bf16(A_bits[:rows])
    t0 = time.perf_counter()
    OG.gemm_rows(A64, B64, True, K, N, np.arange(rows))
    dt = time.perf_counter() - t0
    out = {"value": 2.0 * rows * N * K / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
           "sample": f"first {rows} rows of C for the {M}^3 bf16 GEMM (fp64 C loops, OpenMP over rows), "
                     f"{dt:.1f} s; operand decode not timed"}
    # the other oracle parts, as they stand: the fp32 add (numpy, one core) on 1024 rows of
    # the add workload, and the static schedule enumeration of the headline GEMM
    import synthetic
    from oracle import add as OA
    from oracle import schedule as OS
    x, y = synthetic.add_inputs(1024, ADD_COLS, seed=1)
    t0 = time.perf_counter()
    OA.add_f32(x, y)
    dt_add = time.perf_counter() - t0
    grid = OS.grid_for(M, N, 128, 256, cs=2)
    t0 = time.perf_counter()
    OS.static_schedule(OS.SWIZZLED, grid, 76, 16)
    dt_sched = time.perf_counter() - t0
    out["others"] = {
        "add_f32": {"value": 12.0 * x.size / dt_add / 1e9, "unit": "GB/s", "cores": 1,
                    "sample": f"1024 rows x {ADD_COLS} columns of the fp32 add workload"},
        "schedule": {"value": grid.tiles / dt_sched, "unit": "tiles/s", "cores": 1,
                     "sample": f"swizzled G=16 visit lists, {grid.tiles} pair tiles on 76 workers"},
    }
    return out


# ----------------------------------------------------------------- reference arm
def run_reference(args, world, rank):
    if rank != 0:
        return
    import synthetic
    from oracle import gemm as OG
    A, B = synthetic.gemm_bf16_inputs(M, N, K, seed=2, dist="normal")
    cores = OG.num_threads()
    B64 = OG.dequant_bf16(B)
    rows = max(1, cores)
    A64 = OG.dequant_bf16(A[:rows])
    t0 = time.perf_counter()
    OG.gemm_rows(A64, B64, True, K, N, np.arange(rows))
    t_step = time.perf_counter() - t0
    total_budget = 150.0
    while rows > 1 and t_step * (args.steps + args.warmup) > total_budget:
        rows //= 2
        t_step /= 2
    A64 = OG.dequant_bf16(A[:rows])
    sel = np.arange(rows)
    for _ in range(args.warmup):
        OG.gemm_rows(A64, B64, True, K, N, sel)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        OG.gemm_rows(A64, B64, True, K, N, sel)
    dt = time.perf_counter() - t0
    val = 2.0 * rows * N * K * args.steps / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample_rows_per_step": rows},
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{rows} rows of C per step of the {M}^3 bf16 GEMM, fp64 oracle"},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------ our arm
def run_ours(args, world, rank, local, pg):
    import torch

    import persistent_gemm_tile_gb300 as pgt
    import synthetic

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    peaks = load_peaks()
    ctx = pgt.Context(local, max_groups=16)
    if args.kernel == "add":
        return run_add_headline(args, world, rank, local, pg, torch, pgt, ctx, device, peaks)
    if args.kernel == "ragged":
        return run_ragged_launches(args, pgt, ctx, device)
    dC = torch.empty((M, N), dtype=torch.int16, device=device)
    if args.kernel == "mxfp8":
        return run_mx_headline(args, world, rank, local, pg, torch, pgt, ctx, device, peaks, dC)
    A, B = synthetic.gemm_bf16_inputs(M, N, K, seed=2, dist="normal")
    dA = torch.from_numpy(A.view(np.int16)).to(device)
    dB = torch.from_numpy(B.view(np.int16)).to(device)

    def desc_for(mode, cfg=args.cfg):
        return pgt.make_desc(M, N, K, b_layout=pgt.B_KN, sched_mode=mode, group_size=16, ws_groups=8,
                             kernel_cfg=cfg)

    default_head = args.sched == "swizzled" and args.group == 16
    head = desc_for(pgt.SCHED[args.sched]) if default_head else pgt.make_desc(
        M, N, K, b_layout=pgt.B_KN, sched_mode=pgt.SCHED[args.sched], group_size=args.group,
        ws_groups=args.ws_groups, kernel_cfg=args.cfg,
        ws_layout=pgt.WS_STRIPED if args.ws_layout == "striped" else pgt.WS_RANGES)
    plan = ctx.gemm_plan(head)
    launch = lambda: ctx.gemm_ex(head, dA, dB, dC)  # noqa: E731

    # ------------------------------------------------------------------ headline
    for _ in range(args.warmup):
        launch()
    torch.cuda.synchronize()
    barrier(pg)
    torch.cuda.synchronize()
    clocks = Clocks(local)
    clocks.start()
    clocks.begin()
    total_ms, per = time_launches(torch, launch, args.steps, 0)
    torch.cuda.synchronize()
    clocks.end()
    clk = clocks.stop()
    barrier(pg)
    rc, detail = ctx.last_error()
    if rc != 0:
        raise RuntimeError(f"device-side timeout during the timed region: {detail}")
    total_ms = max_over_ranks(pg, total_ms, device)
    ms_per_step = total_ms / args.steps
    value = world * FLOP * args.steps / (total_ms * 1e-3) / 1e12
    kern_ms = float(np.mean(per))
    achieved = FLOP / (kern_ms * 1e-3) / 1e12
    long_region = total_ms > 500.0
    peak = peaks["bf16_sustained"] if long_region else peaks["bf16_burst"]
    out = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "kernel_cfg": plan["kernel_cfg"],
                   "tile": f"{plan['bm'] * plan['cluster_size']}x{plan['bn']}",
                   "ctas_per_worker": plan["cluster_size"], "workers": plan["workers"], "stages": plan["stages"],
                   "l2": L2_NOTE, "parallelism": f"{world} independent GEMMs (one per GPU)"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak,
                     "traffic": profiled_traffic("gemm_bf16_2cta_256x256")
                     if plan["kernel_cfg"] == 4 and default_head else None,
                     "peak_kind": ("sustained" if long_region else "burst") + f" bf16 ({peaks['source']})"},
        "gpu_launches": args.steps,
        "clocks": clk,
    }
    if rank != 0:
        return
    if not args.no_extras:
        extras(args, torch, pgt, ctx, device, dA, dB, dC, desc_for, peaks, out, head)
    print(json.dumps(out), flush=True)
    ctx.close()


def run_add_headline(args, world, rank, local, pg, torch, pgt, ctx, device, peaks):
    """The persistent add as the timed kernel (tile and order from --add-tile / --add-sched):
    GB/s against HBM."""
    import synthetic
    x, y = synthetic.add_inputs(ADD_ROWS, ADD_COLS, seed=1)
    tx, ty = torch.from_numpy(x).to(device), torch.from_numpy(y).to(device)
    to = torch.empty_like(tx)
    tile = (0, 0) if args.add_tile == "wide" else tuple(int(v) for v in args.add_tile.split("x"))
    tname = "wide 8x1024" if tile == (0, 0) else f"{tile[0]}x{tile[1]}"
    traffic_key = f"add_page_32x16_{args.add_sched}" if tile == (32, 16) else f"add_wide_8x1024_{args.add_sched}"
    mode = pgt.SCHED[args.add_sched]
    launch = lambda: ctx.add(tx, ty, to, sched_mode=mode, tile_r=tile[0], tile_c=tile[1])  # noqa: E731
    for _ in range(args.warmup):
        launch()
    torch.cuda.synchronize()
    barrier(pg)
    clocks = Clocks(local)
    clocks.start()
    clocks.begin()
    total_ms, per = time_launches(torch, launch, args.steps, 0)
    clocks.end()
    clk = clocks.stop()
    barrier(pg)
    total_ms = max_over_ranks(pg, total_ms, device)
    kern_ms = float(np.mean(per))
    achieved = ADD_BYTES / (kern_ms * 1e-3) / 1e9
    out = {"metric": "persistent add GB/s vs HBM", "value": world * ADD_BYTES * args.steps / (total_ms * 1e-3) / 1e9,
           "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": "f32", "data": "synthetic",
           "config": {"workload": f"fp32 add 8192x8192, {tname} tile, {args.add_sched}", "l2": L2_NOTE},
           "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                        "frac": achieved / peaks["hbm_gbs"], "traffic": profiled_traffic(traffic_key)},
           "gpu_launches": args.steps, "clocks": clk}
    if rank == 0:
        print(json.dumps(out), flush=True)
    ctx.close()


def run_mx_headline(args, world, rank, local, pg, torch, pgt, ctx, device, peaks, dC):
    """The MXFP8 GEMM 8192^3 (2 launches per step: scale repack + GEMM) as the timed kernel."""
    import synthetic
    qa, sa, qb, sb = synthetic.gemm_mxfp8_inputs(M, N, K, seed=4)
    tqa, tsa = torch.from_numpy(qa).to(device), torch.from_numpy(sa).to(device)
    tqb, tsb = torch.from_numpy(qb).to(device), torch.from_numpy(sb).to(device)
    d = pgt.make_desc(M, N, K, dtype=pgt.MXFP8, b_layout=pgt.B_NK, sched_mode=pgt.SWIZZLED, group_size=16,
                      kernel_cfg=args.cfg)
    plan = ctx.gemm_plan(d)
    ws = torch.empty(ctx.gemm_workspace_bytes(d), dtype=torch.uint8, device=device)
    launch = lambda: ctx.gemm_ex(d, tqa, tqb, dC, sfa=tsa, sfb=tsb, workspace=ws)  # noqa: E731
    for _ in range(args.warmup):
        launch()
    torch.cuda.synchronize()
    barrier(pg)
    clocks = Clocks(local)
    clocks.start()
    clocks.begin()
    total_ms, per = time_launches(torch, launch, args.steps, 0)
    clocks.end()
    clk = clocks.stop()
    barrier(pg)
    total_ms = max_over_ranks(pg, total_ms, device)
    kern_ms = float(np.mean(per))
    achieved = FLOP / (kern_ms * 1e-3) / 1e12
    fp8_peak = 2.0 * peaks["bf16_burst"]
    out = {"metric": "MXFP8 GEMM TFLOP/s vs fp8 tensor peak", "value": world * FLOP * args.steps / (total_ms * 1e-3) / 1e12,
           "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": "e4m3+e8m0", "data": "synthetic",
           "config": {"workload": f"MXFP8 {M}^3 seed 4, swizzled group 16", "kernel_cfg": plan["kernel_cfg"],
                      "tile": f"{plan['bm'] * plan['cluster_size']}x{plan['bn']}", "l2": L2_NOTE},
           "roofline": {"bound": "tensor", "achieved": achieved, "peak": fp8_peak, "unit": "TFLOP/s",
                        "frac": achieved / fp8_peak,
                        "traffic": profiled_traffic("gemm_mxfp8_2cta_256x256") if plan["kernel_cfg"] == 4 else None,
                        "peak_kind": f"2 x bf16 burst ({peaks['source']})"},
           "gpu_launches": 2 * args.steps, "clocks": clk}
    if args.cublas:
        lib_launch, lib_out = cublas_mxfp8(torch, qa, sa, qb, sb, device)
        if lib_launch is None:
            out["vs_cublas"] = {"unavailable": lib_out}
        else:
            _, lper = time_launches(torch, lib_launch, max(3, args.steps), args.warmup)
            lms = float(np.median(lper))
            out["vs_cublas"] = {"cublas_tflops": FLOP / (lms * 1e-3) / 1e12, "ours_tflops": achieved,
                                "bit_identical_outputs": bool(torch.equal(dC.view(torch.bfloat16), lib_out))}
    if rank == 0:
        print(json.dumps(out), flush=True)
    ctx.close()


def extras(args, torch, pgt, ctx, device, dA, dB, dC, desc_for, peaks, out, head):
    import synthetic
    A_host = dA.cpu().numpy().view(np.uint16)
    B_host = dB.cpu().numpy().view(np.uint16)
    launch = lambda: ctx.gemm_ex(head, dA, dB, dC)  # noqa: E731
    # the headline GEMM over a 2-second back-to-back loop, clocks sampled inside it: the
    # power-capped steady state, against the sustained peak
    clocks = Clocks(device.index or 0, period_ms=50)
    clocks.start()
    clocks.begin()
    blocks = time_sustained(torch, launch, 2.0)
    clocks.end()
    clk = clocks.stop()
    ms = float(np.median(blocks))
    tf = FLOP / (ms * 1e-3) / 1e12
    out["sustained"] = {"tflops": tf, "ms": ms, "seconds": 2.0, "launches": 50 * len(blocks),
                        "peak": peaks["bf16_sustained"], "frac": tf / peaks["bf16_sustained"],
                        "peak_kind": f"sustained bf16 ({peaks['source']})", "clocks": clk,
                        "tflops_per_sm_ghz": tf / (clk["sm_mhz"] / 1e3) if clk.get("sm_mhz") else None}
    # the benchmark plan's protocol: 10 warm-ups, 50 individually timed launches, L2 flushed
    # (256 MiB written) before each; median and best
    flush_buf = torch.empty(64 << 20, dtype=torch.float32, device=device)
    per = time_protocol(torch, launch, lambda: flush_buf.fill_(1.0))
    del flush_buf
    out["protocol"] = {"warmup": 10, "reps": 50, "l2_flush": "256 MiB written before each launch, outside the events",
                       "median_ms": float(np.median(per)), "min_ms": float(np.min(per)),
                       "tflops_median": FLOP / (float(np.median(per)) * 1e-3) / 1e12,
                       "tflops_best": FLOP / (float(np.min(per)) * 1e-3) / 1e12}
    # per scheduler mode: 1-second back-to-back loops, modes interleaved over 3 rounds so that
    # each sees the same mix of power and clock states (the GPU is power-capped within a
    # fraction of a second); median of the 50-launch block means
    per_mode = {}
    names = {pgt.BLOCKED: "blocked", pgt.INTERLEAVED: "interleaved", pgt.SWIZZLED: "swizzled",
             pgt.WORK_STEALING: "work_stealing", pgt.BLOCKED_GROUPED_M: "blocked_grouped_m",
             pgt.LAUNCH_CONTROL: "launch_control"}
    descs = {name: desc_for(mode) for mode, name in names.items()}
    # work stealing with striped tile ownership (counter group g owns tiles t = g mod 8)
    descs["work_stealing_striped"] = pgt.make_desc(M, N, K, b_layout=pgt.B_KN, sched_mode=pgt.WORK_STEALING,
                                                   group_size=16, ws_groups=8, kernel_cfg=args.cfg,
                                                   ws_layout=pgt.WS_STRIPED)
    samples = {name: [] for name in descs}
    for _ in range(3):
        for name, d in descs.items():
            samples[name].extend(time_sustained(torch, lambda: ctx.gemm_ex(d, dA, dB, dC), 1.0))
    for name, per in samples.items():
        ms = float(np.median(per))
        tf = FLOP / (ms * 1e-3) / 1e12
        per_mode[name] = {"tflops": tf, "ms": ms, "frac_of_burst_peak": tf / peaks["bf16_burst"]}
    out["per_mode"] = per_mode
    # work stealing with 1..16 counter groups, contiguous ranges and striped ownership,
    # 1-second loops interleaved over 2 rounds
    wdescs = {f"{lay}_groups_{g}": pgt.make_desc(M, N, K, b_layout=pgt.B_KN, sched_mode=pgt.WORK_STEALING,
                                                 group_size=16, ws_groups=g, kernel_cfg=args.cfg, ws_layout=code)
              for lay, code in (("ranges", pgt.WS_RANGES), ("striped", pgt.WS_STRIPED)) for g in (1, 2, 4, 8, 16)}
    wsamples = {k: [] for k in wdescs}
    for _ in range(2):
        for k, d in wdescs.items():
            wsamples[k].extend(time_sustained(torch, lambda: ctx.gemm_ex(d, dA, dB, dC), 1.0))
    out["work_stealing_groups"] = {k: {"tflops": FLOP / (float(np.median(v)) * 1e-3) / 1e12,
                                       "ms": float(np.median(v))} for k, v in wsamples.items()}
    # swizzle group width (column blocks per group), interleaved rounds
    gsamples = {g: [] for g in (2, 4, 8, 16, 32)}
    gdescs = {g: pgt.make_desc(M, N, K, b_layout=pgt.B_KN, sched_mode=pgt.SWIZZLED, group_size=g,
                               kernel_cfg=args.cfg) for g in gsamples}
    for _ in range(4):
        for g, d in gdescs.items():
            _, per = time_launches(torch, lambda: ctx.gemm_ex(d, dA, dB, dC), 10, 2)
            gsamples[g].extend(per)
    out["swizzle_groups"] = {f"group_{g}": {"tflops": FLOP / (float(np.median(v)) * 1e-3) / 1e12,
                                            "ms": float(np.median(v))} for g, v in gsamples.items()}
    # per kernel configuration (swizzled, group 16), interleaved the same way
    per_cfg = {}
    cfgs = ((pgt.CFG_1CTA_128x128, "1cta_128x128"), (pgt.CFG_1CTA_128x256, "1cta_128x256"),
            (pgt.CFG_2CTA_256x128, "2cta_256x128"), (pgt.CFG_2CTA_256x256, "2cta_256x256"))
    csamples = {cname: [] for _, cname in cfgs}
    cdescs = {cname: desc_for(pgt.SWIZZLED, cfg) for cfg, cname in cfgs}
    for _ in range(4):
        for _, cname in cfgs:
            d = cdescs[cname]
            _, per = time_launches(torch, lambda: ctx.gemm_ex(d, dA, dB, dC), 10, 2)
            csamples[cname].extend(per)
    for cname, per in csamples.items():
        ms = float(np.median(per))
        per_cfg[cname] = {"tflops": FLOP / (ms * 1e-3) / 1e12, "ms": ms}
    out["per_cfg"] = per_cfg
    # cuBLAS through torch.matmul on the same bf16 operands, rounds interleaved with this
    # kernel (swizzled, group 16): a library point of comparison on the same GPU and power
    # state, not part of the path
    a16, b16 = dA.view(torch.bfloat16), dB.view(torch.bfloat16)
    c16 = torch.empty((M, N), dtype=torch.bfloat16, device=device)
    head = desc_for(pgt.SWIZZLED)
    lsamples = {"ours": [], "cublas": []}
    for _ in range(6):
        _, per = time_launches(torch, lambda: ctx.gemm_ex(head, dA, dB, dC), 10, 2)
        lsamples["ours"].extend(per)
        _, per = time_launches(torch, lambda: torch.matmul(a16, b16, out=c16), 10, 2)
        lsamples["cublas"].extend(per)
    out["vs_cublas"] = {name: {"tflops": FLOP / (float(np.median(v)) * 1e-3) / 1e12, "ms": float(np.median(v))}
                        for name, v in lsamples.items()}
    out["vs_cublas"]["ratio"] = out["vs_cublas"]["ours"]["tflops"] / out["vs_cublas"]["cublas"]["tflops"]
    del c16
    # tail idle from traced launches (not timed)
    tails = {}
    for name, d in descs.items():
        plan = ctx.gemm_plan(d)
        tb = pgt.TraceBuffers(plan["ctas"], plan["tiles"], device=device)
        ctx.gemm_ex(d, dA, dB, dC, trace=tb.struct)
        torch.cuda.synchronize()
        tails[name] = tail_idle(tb.times.cpu().numpy())
    out["tail_idle"] = {"workload": f"{M}^3 bf16", **tails}
    # persistent add
    x, y = synthetic.add_inputs(ADD_ROWS, ADD_COLS, seed=1)
    tx, ty = torch.from_numpy(x).to(device), torch.from_numpy(y).to(device)
    to = torch.empty_like(tx)
    add = {}
    best = None
    for tile, tname in (((0, 0), "wide_8x1024"), ((32, 16), "page_32x16")):
        for mode, mname in ((pgt.BLOCKED, "blocked"), (pgt.INTERLEAVED, "interleaved")):
            fn = lambda: ctx.add(tx, ty, to, sched_mode=mode, tile_r=tile[0], tile_c=tile[1])  # noqa: E731
            _, per = time_launches(torch, fn, 30, 3)
            ms = float(np.median(per))
            gbs = ADD_BYTES / (ms * 1e-3) / 1e9
            add[f"{tname}_{mname}"] = {"gbs": gbs, "ms": ms}
            if best is None or gbs > best[1]:
                best = (f"{tname}_{mname}", gbs, ms)
    # the page's 32 x 16 tile against the worker count (0 = the library's default); the SM
    # count is the pages' own choice
    sweep = {}
    for mode, mname in ((pgt.BLOCKED, "blocked"), (pgt.INTERLEAVED, "interleaved")):
        for P in (0, ctx.num_sms, 512, 1024, 2048, 4096):
            fn = lambda: ctx.add(tx, ty, to, sched_mode=mode, tile_r=32, tile_c=16, num_workers=P)  # noqa: E731
            _, per = time_launches(torch, fn, 20, 3)
            sweep[f"{mname}_{P or 'default'}"] = ADD_BYTES / (float(np.median(per)) * 1e-3) / 1e9
        sweep[f"{mname}_default_workers"] = ctx.add_workers(ADD_ROWS, ADD_COLS, 32, 16, sched_mode=mode)
    add["page_32x16_workers_gbs"] = sweep
    add["roofline"] = {"bound": "hbm", "achieved": best[1], "peak": peaks["hbm_gbs"], "unit": "GB/s",
                       "frac": best[1] / peaks["hbm_gbs"],
                       "traffic": profiled_traffic("add_" + best[0]),
                       "kernel": best[0],
                       "algorithmic_bytes": ADD_BYTES}
    add["workload"] = "fp32 8192x8192 x,y ~ N(0,1) seed 1, out = x + y"
    out["add"] = add
    # fused multi-space loop (helion multi-loop): result1 = 2 x, result2 = 3 y in one launch
    r1, r2 = torch.empty_like(tx), torch.empty_like(ty)
    ml = {}
    for mode, mname in ((pgt.BLOCKED, "blocked"), (pgt.INTERLEAVED, "interleaved")):
        fn = lambda: ctx.multi_loop([(tx, r1, 2.0), (ty, r2, 3.0)], sched_mode=mode)  # noqa: E731
        _, per = time_launches(torch, fn, 30, 3)
        ms = float(np.median(per))
        ml[mname] = {"gbs": 2 * 8.0 * ADD_ROWS * ADD_COLS / (ms * 1e-3) / 1e9, "ms": ms}
    ml["workload"] = "two fp32 8192x8192 spaces in one launch, wide 8x1024 tile; 8 bytes per element"
    out["multi_loop"] = ml
    del r1, r2
    del tx, ty, to
    # MXFP8 block-scaled GEMM 8192^3 (E4M3 payload from N(0,1), E8M0 exponents in [-4, 4], seed 4)
    qa, sa, qb, sb = synthetic.gemm_mxfp8_inputs(M, N, K, seed=4)
    tqa, tsa = torch.from_numpy(qa).to(device), torch.from_numpy(sa).to(device)
    tqb, tsb = torch.from_numpy(qb).to(device), torch.from_numpy(sb).to(device)
    mx = {}
    fp8_peak = 2.0 * peaks["bf16_burst"]  # fp8 dense is twice bf16 dense (4.5 vs 2.25 PFLOP/s nominal)
    for cfg, cname in ((pgt.CFG_2CTA_256x256, "2cta_256x256"), (pgt.CFG_2CTA_256x224, "2cta_256x224"),
                       (pgt.CFG_1CTA_128x256, "1cta_128x256"), (pgt.CFG_2CTA_256x128, "2cta_256x128")):
        d = pgt.make_desc(M, N, K, dtype=pgt.MXFP8, b_layout=pgt.B_NK, sched_mode=pgt.SWIZZLED, group_size=16,
                          kernel_cfg=cfg)
        ws = torch.empty(ctx.gemm_workspace_bytes(d), dtype=torch.uint8, device=device)
        _, per = time_launches(torch, lambda: ctx.gemm_ex(d, tqa, tqb, dC, sfa=tsa, sfb=tsb, workspace=ws), 40, 5)
        ms = float(np.median(per))
        tf = FLOP / (ms * 1e-3) / 1e12
        mx[cname] = {"tflops": tf, "ms": ms, "frac_of_fp8_peak": tf / fp8_peak}
    best = max(mx, key=lambda k: mx[k]["tflops"])
    mx["roofline"] = {"bound": "tensor", "achieved": mx[best]["tflops"], "peak": fp8_peak, "unit": "TFLOP/s",
                      "frac": mx[best]["tflops"] / fp8_peak,
                      "traffic": profiled_traffic("gemm_mxfp8_2cta_256x256") if best == "2cta_256x256" else None,
                      "kernel": best,
                      "peak_kind": f"2 x measured bf16 burst ({peaks['source']}), nominal fp8/bf16 ratio"}
    mx["workload"] = f"MXFP8 {M}^3, E4M3 payload N(0,1), E8M0 per 1x128 K block, exps U{{-4..4}}, seed 4, " \
                     "swizzled group 16; time includes the per-call scale repack"
    # cuBLAS MXFP8 on the same operands, rounds interleaved with this library's AUTO kernel
    lib_launch, lib_out = cublas_mxfp8(torch, qa, sa, qb, sb, device)
    if lib_launch is None:
        mx["vs_cublas"] = {"unavailable": lib_out}
    else:
        d = pgt.make_desc(M, N, K, dtype=pgt.MXFP8, b_layout=pgt.B_NK, sched_mode=pgt.SWIZZLED, group_size=16)
        ws = torch.empty(ctx.gemm_workspace_bytes(d), dtype=torch.uint8, device=device)
        ours = lambda: ctx.gemm_ex(d, tqa, tqb, dC, sfa=tsa, sfb=tsb, workspace=ws)  # noqa: E731
        ours()
        torch.cuda.synchronize()
        same = bool(torch.equal(dC.view(torch.bfloat16), lib_out))
        vs = {"ours": [], "cublas": []}
        for _ in range(6):
            vs["ours"].extend(time_launches(torch, ours, 10, 2)[1])
            vs["cublas"].extend(time_launches(torch, lib_launch, 10, 2)[1])
        mx["vs_cublas"] = {k: {"tflops": FLOP / (float(np.median(v)) * 1e-3) / 1e12, "ms": float(np.median(v))}
                           for k, v in vs.items()}
        mx["vs_cublas"]["ratio"] = mx["vs_cublas"]["ours"]["tflops"] / mx["vs_cublas"]["cublas"]["tflops"]
        mx["vs_cublas"]["bit_identical_outputs"] = same
        mx["vs_cublas"]["how"] = "torch._scaled_mm, E8M0 scales repeated per 32-wide K block, bf16 out"
        del ws
    del lib_launch, lib_out
    out["mxfp8"] = mx
    del tqa, tsa, tqb, tsb
    if not args.no_ragged:
        out["ragged"] = ragged_set(torch, pgt, ctx, device)
    out["small_256"] = small_256(torch, pgt, ctx, device)
    # end to end from pinned host memory through pgt_gemm_host: every step copies its A and B
    # host -> device, runs the GEMM and copies C back.  Two streams with two device buffer
    # sets let one step's GEMM and D2H overlap the next step's H2D (the link carries H2D and
    # D2H concurrently); the single-stream figure is reported beside it.
    hA = torch.from_numpy(A_host.view(np.int16)).pin_memory()
    hB = torch.from_numpy(B_host.view(np.int16)).pin_memory()
    hCs = [torch.empty((M, N), dtype=torch.int16).pin_memory() for _ in range(2)]
    d = desc_for(pgt.SWIZZLED)
    e2e_steps = max(4, min(args.steps, 20))
    single, _ = time_launches(torch, lambda: ctx.gemm_host(d, hA, hB, hCs[0], dA, dB, dC), e2e_steps, 2)
    bufs = [(dA, dB, dC), (torch.empty_like(dA), torch.empty_like(dB), torch.empty_like(dC))]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]

    def pipelined(steps):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record()
        for st in streams:
            st.wait_event(start)
        for i in range(steps):
            k = i % 2
            ctx.gemm_host(d, hA, hB, hCs[k], *bufs[k], stream=streams[k])
        for st in streams:
            torch.cuda.current_stream().wait_stream(st)
        end.record()
        torch.cuda.synchronize()
        return start.elapsed_time(end)

    pipelined(2)
    total = pipelined(e2e_steps)
    h2d_b = int(hA.numel() * 2 + hB.numel() * 2)
    d2h_b = int(hCs[0].numel() * 2)
    link = link_bandwidth(torch, hA, dA, hCs[1], dC, streams)
    # the link bound of one step: its H2D and D2H bytes with both directions busy at once,
    # and never less than its H2D bytes alone (the GEMM overlaps the other stream's copies)
    bound_ms = max((h2d_b + d2h_b) / (link["both_gbs"] * 1e9), h2d_b / (link["h2d_gbs"] * 1e9)) * 1e3
    step_ms = total / e2e_steps
    out["e2e"] = {"value": FLOP * e2e_steps / (total * 1e-3) / 1e12, "unit": "TFLOP/s",
                  "h2d_bytes_per_step": h2d_b, "d2h_bytes_per_step": d2h_b, "steps": e2e_steps, "streams": 2,
                  "single_stream_value": FLOP * e2e_steps / (single * 1e-3) / 1e12,
                  "link": link, "ms_per_step": step_ms, "link_bound_ms_per_step": bound_ms,
                  "frac_of_link_bound": bound_ms / step_ms}
    del bufs
    # the oracle on the host cores
    out["cpu_baseline"] = cpu_baseline(args.cpu_seconds, A_host, B_host)


def block_scale_tiles(s: np.ndarray) -> np.ndarray:
    """E8M0 scales (rows x blocks) in the tiled layout the library's block-scaled GEMMs read:
    128-row x 4-block tiles of 512 bytes, tile-major over (row tile, block tile), inside a
    tile byte (r mod 32) * 16 + ((r mod 128) div 32) * 4 + (block mod 4); padding zero."""
    R, C = s.shape
    Rp, Cp = -(-R // 128) * 128, -(-C // 4) * 4
    pad = np.zeros((Rp, Cp), np.uint8)
    pad[:R, :C] = s
    r = np.arange(Rp)[:, None]
    c = np.arange(Cp)[None, :]
    off = ((r // 128) * (Cp // 4) + c // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + c % 4
    out = np.empty(Rp * Cp, np.uint8)
    out[off.ravel()] = pad.ravel()
    return out


def cublas_mxfp8(torch, qa, sa, qb, sb, device):
    """cuBLAS's MXFP8 GEMM (torch._scaled_mm) on the same operands, as a measured point of
    comparison (never on the path).  The library takes one E8M0 scale per 32-wide K block,
    so each 128-wide block's scale is repeated four times: the same products exactly.
    Returns (launch, output) or (None, reason)."""
    try:
        a8 = torch.from_numpy(qa).to(device).view(torch.float8_e4m3fn)
        b8 = torch.from_numpy(qb).to(device).view(torch.float8_e4m3fn)
        s_a = torch.from_numpy(block_scale_tiles(np.repeat(sa, 4, axis=1))).to(device).view(torch.float8_e8m0fnu)
        s_b = torch.from_numpy(block_scale_tiles(np.repeat(sb, 4, axis=1))).to(device).view(torch.float8_e8m0fnu)
        out = torch.empty((qa.shape[0], qb.shape[0]), dtype=torch.bfloat16, device=device)

        def launch():
            torch._scaled_mm(a8, b8.t(), s_a, s_b, out_dtype=torch.bfloat16, out=out)
        launch()
        torch.cuda.synchronize()
        return launch, out
    except Exception as e:  # an older torch or a GPU without the block-scaled path
        return None, f"{type(e).__name__}: {str(e)[:200]}"


def link_bandwidth(torch, h_in, d_in, h_out, d_out, streams) -> dict:
    """Host link bandwidth with pinned buffers: H2D alone, D2H alone, and both at once on two
    streams (GB/s, best of 3).  The copy engines and kernels that load or store host memory
    directly reach the same figures on this machine, so this is the e2e roofline."""
    def timed(fn, nbytes):
        best = 0.0
        for _ in range(3):
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            best = max(best, nbytes / (a.elapsed_time(b) * 1e-3) / 1e9)
        return best

    n_in = h_in.numel() * h_in.element_size()
    n_out = h_out.numel() * h_out.element_size()

    def both():
        ev = torch.cuda.Event()
        ev.record()
        for st in streams:
            st.wait_event(ev)
        with torch.cuda.stream(streams[0]):
            d_in.copy_(h_in, non_blocking=True)
        with torch.cuda.stream(streams[1]):
            h_out.copy_(d_out, non_blocking=True)
        for st in streams:
            torch.cuda.current_stream().wait_stream(st)

    return {"h2d_gbs": timed(lambda: d_in.copy_(h_in, non_blocking=True), n_in),
            "d2h_gbs": timed(lambda: h_out.copy_(d_out, non_blocking=True), n_out),
            "both_gbs": timed(both, n_in + n_out)}


BF16_CFGS = ((0, "auto"), (1, "1cta_128x128"), (2, "1cta_128x256"), (3, "2cta_256x128"), (4, "2cta_256x256"))
RAGGED = [(4864, 4096, 2048), (128, 16384, 16384), (3000, 5000, 1024)]


def graph_us(torch, fn, reps: int = 50) -> float:
    """Device time per call of `fn` replayed from a CUDA graph of `reps` calls (us)."""
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(reps):
            fn()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(5):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return 1e3 * e0.elapsed_time(e1) / (5 * reps)


def small_256(torch, pgt, ctx, device):
    """bf16 256^3 (U[-1,1], seed 0): per scheduler on 128 x 128 tiles (4 tiles, 4 workers),
    and per kernel configuration (swizzled, group 2) incl. AUTO; latency in microseconds,
    eager and replayed from a CUDA graph.  Launch-bound: no roofline fraction is claimed."""
    import synthetic
    a, b = synthetic.gemm_bf16_inputs(256, 256, 256, seed=0, dist="uniform")
    ta = torch.from_numpy(a.view(np.int16)).to(device)
    tb_ = torch.from_numpy(b.view(np.int16)).to(device)
    tc = torch.empty((256, 256), dtype=torch.int16, device=device)
    res = {}
    for mode, name in ((pgt.BLOCKED, "blocked"), (pgt.INTERLEAVED, "interleaved"), (pgt.SWIZZLED, "swizzled"),
                       (pgt.WORK_STEALING, "work_stealing"), (pgt.LAUNCH_CONTROL, "launch_control")):
        d = pgt.make_desc(256, 256, 256, sched_mode=mode, group_size=2, kernel_cfg=pgt.CFG_1CTA_128x128)
        _, per = time_launches(torch, lambda: ctx.gemm_ex(d, ta, tb_, tc), 50, 5)
        res[name] = {"us_eager": 1e3 * float(np.median(per)), "us_graph": graph_us(torch, lambda: ctx.gemm_ex(d, ta, tb_, tc))}
    per_cfg = {}
    for cfg, cname in BF16_CFGS:
        d = pgt.make_desc(256, 256, 256, sched_mode=pgt.SWIZZLED, group_size=2, kernel_cfg=cfg)
        per_cfg[cname] = {"us_graph": graph_us(torch, lambda: ctx.gemm_ex(d, ta, tb_, tc)),
                          "kernel_cfg": ctx.gemm_plan(d)["kernel_cfg"]}
    res["per_cfg"] = per_cfg
    return res


def ragged_set(torch, pgt, ctx, device):
    """The ragged-tail set (tile counts not a multiple of the SM count), every kernel
    configuration (AUTO included) and every scheduler: TFLOP/s and tail idle
    (1 - busy / (workers * span)) from a traced launch."""
    import synthetic
    res = {}
    names = {pgt.BLOCKED: "blocked", pgt.INTERLEAVED: "interleaved", pgt.SWIZZLED: "swizzled",
             pgt.WORK_STEALING: "work_stealing", pgt.BLOCKED_GROUPED_M: "blocked_grouped_m",
             pgt.LAUNCH_CONTROL: "launch_control"}
    for (m, n, k), (a, b) in zip(RAGGED, synthetic.gemm_bf16_sequence(RAGGED, seed=3, dist="uniform")):
        ta = torch.from_numpy(a.view(np.int16)).to(device)
        tb_ = torch.from_numpy(b.view(np.int16)).to(device)
        tc = torch.empty((m, n), dtype=torch.int16, device=device)
        key = f"{m}x{n}x{k}"
        res[key] = {}
        variants = [(mode, name, pgt.WS_RANGES) for mode, name in names.items()]
        variants.append((pgt.WORK_STEALING, "work_stealing_striped", pgt.WS_STRIPED))
        for cfg, cname in BF16_CFGS:
            for mode, name, layout in variants:
                d = pgt.make_desc(m, n, k, b_layout=pgt.B_KN, sched_mode=mode, group_size=16, ws_groups=8,
                                  kernel_cfg=cfg, ws_layout=layout)
                _, per = time_launches(torch, lambda: ctx.gemm_ex(d, ta, tb_, tc), 20, 3)
                ms = float(np.median(per))
                plan = ctx.gemm_plan(d)
                tr = pgt.TraceBuffers(plan["ctas"], plan["tiles"], device=device)
                ctx.gemm_ex(d, ta, tb_, tc, trace=tr.struct)
                torch.cuda.synchronize()
                times = tr.times.cpu().numpy()
                res[key][f"{cname}_{name}"] = {"tflops": 2.0 * m * n * k / (ms * 1e-3) / 1e12, "ms": ms,
                                               "tail_idle": tail_idle(times),
                                               "tail_idle_all_sms": tail_idle(times, ctx.num_sms),
                                               "tiles": plan["tiles"], "workers": plan["workers"],
                                               "kernel_cfg": plan["kernel_cfg"]}
        # AUTO against the fastest configuration under the swizzled order
        sw = {c: res[key][f"{c}_swizzled"]["tflops"] for _, c in BF16_CFGS if c != "auto"}
        best = max(sw, key=sw.get)
        res[key]["auto_vs_best"] = {"best": best, "auto_frac_of_best": res[key]["auto_swizzled"]["tflops"] / sw[best]}
        del ta, tb_, tc
    return res


def run_ragged_launches(args, pgt, ctx, device):
    """--kernel ragged: one untraced launch per (shape, configuration, scheduler) of the
    ragged set, in a fixed order, for a profiler to capture (e.g. SM-active against elapsed
    cycles per launch); prints the launch order as one JSON line."""
    import torch

    import synthetic
    order = []
    modes = ((pgt.BLOCKED, "blocked", pgt.WS_RANGES), (pgt.INTERLEAVED, "interleaved", pgt.WS_RANGES),
             (pgt.SWIZZLED, "swizzled", pgt.WS_RANGES), (pgt.WORK_STEALING, "work_stealing", pgt.WS_RANGES),
             (pgt.WORK_STEALING, "work_stealing_striped", pgt.WS_STRIPED),
             (pgt.BLOCKED_GROUPED_M, "blocked_grouped_m", pgt.WS_RANGES),
             (pgt.LAUNCH_CONTROL, "launch_control", pgt.WS_RANGES))
    for (m, n, k), (a, b) in zip(RAGGED, synthetic.gemm_bf16_sequence(RAGGED, seed=3, dist="uniform")):
        ta = torch.from_numpy(a.view(np.int16)).to(device)
        tb_ = torch.from_numpy(b.view(np.int16)).to(device)
        tc = torch.empty((m, n), dtype=torch.int16, device=device)
        for cfg, cname in ((0, "auto"), (2, "1cta_128x256"), (3, "2cta_256x128")):
            for mode, name, layout in modes:
                d = pgt.make_desc(m, n, k, sched_mode=mode, group_size=16, ws_groups=8, kernel_cfg=cfg,
                                  ws_layout=layout)
                ctx.gemm_ex(d, ta, tb_, tc)
                plan = ctx.gemm_plan(d)
                order.append({"shape": f"{m}x{n}x{k}", "cfg": cname, "kernel_cfg": plan["kernel_cfg"],
                              "sched": name, "tiles": plan["tiles"], "workers": plan["workers"],
                              "ctas": plan["ctas"]})
        torch.cuda.synchronize()
        del ta, tb_, tc
    rc, detail = ctx.last_error()
    if rc != 0:
        raise RuntimeError(f"device-side timeout: {detail}")
    print(json.dumps({"metric": "ragged-set launches (profiling)", "launches": order}), flush=True)
    ctx.close()


def main():
    global M, N, K, FLOP, WORKLOAD
    args = parse()
    if args.size != 8192:
        if args.size < 256 or args.size % 256:
            raise SystemExit("--size must be a positive multiple of 256")
        M = N = K = args.size
        FLOP = 2.0 * M * N * K
        WORKLOAD = WORKLOAD.replace("M=N=K=8192", f"M=N=K={args.size}")
    if args.sched != "swizzled" or args.group != 16:
        sched = args.sched
        if sched == "work_stealing":
            sched += f" ({args.ws_groups} counter groups, {args.ws_layout})"
        WORKLOAD = WORKLOAD.replace("swizzled group_size=16", f"{sched} group_size={args.group}")
    world, rank, local, pg = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local, pg)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
