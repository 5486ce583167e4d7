// Allocation-free form of the work-stealing bf16 GEMM.
//
// The regular entry points need a context from pgt_preamble, which cudaMallocs the tile
// counters.  Some callers cannot allocate device memory at all: code that runs inside
// another runtime's memory-pool or allocator hook (where a cudaMalloc would re-enter or
// bypass the pool), plugins of inference servers whose device memory is budgeted up front
// and must not grow, and real-time paths that forbid allocation after start-up.  This
// file serves them: the scratch the kernel needs (work-stealing counters, done counter,
// error word) lives in a fixed-size file-scope __device__ array that every GPU loading
// the library holds until the process exits.
#include <mutex>

#include "pgt_internal.h"
#include "pgt_sched.cuh"

namespace {

constexpr int kNoallocMaxDevices = 64;
// counters for PGT_NOALLOC_MAX_GROUPS groups (one 128-byte line each), the done counter's
// line and the error word's line: 18 lines = 2304 bytes
constexpr int kScratchInts = pgt::kCounterStride * (PGT_NOALLOC_MAX_GROUPS + 2);

static __device__ __align__(256) int g_noalloc_scratch[kScratchInts];

struct DeviceScratch {
    bool ready;
    int* scratch;  // device address of g_noalloc_scratch on this device
    int num_sms;
};

DeviceScratch g_devices[kNoallocMaxDevices];
std::mutex g_mutex;

// Once per device, with that device current: resolve the array's device address (the
// host-side symbol is only a stand-in and must never be handed to a kernel) and the SM
// count.  The lookup may load the module, so it is refused while `stream` is capturing.
int device_setup(int device, cudaStream_t stream, DeviceScratch* out) {
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceScratch& s = g_devices[device];
    if (!s.ready) {
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return PGT_ERR_CUDA;
        if (cap != cudaStreamCaptureStatusNone) return PGT_ERR_ARG;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return PGT_ERR_CUDA;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || sms < 1)
            return PGT_ERR_CUDA;
        s.scratch = static_cast<int*>(p);
        s.num_sms = sms;
        s.ready = true;
    }
    *out = s;
    return PGT_OK;
}

}  // namespace

extern "C" int pgt_gemm_noalloc(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                                int b_layout, int group_size, int ws_groups, int32_t* d_err, void* stream) {
    if (A == nullptr || B == nullptr || C == nullptr) return PGT_ERR_ARG;
    if (ws_groups == 0) ws_groups = 8;
    if (ws_groups < 1 || ws_groups > PGT_NOALLOC_MAX_GROUPS) return PGT_ERR_GROUPS;
    int device = -1;
    if (cudaGetDevice(&device) != cudaSuccess) return PGT_ERR_CUDA;
    if (device < 0 || device >= kNoallocMaxDevices) return PGT_ERR_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    DeviceScratch ds;
    int rc = device_setup(device, st, &ds);
    if (rc) return rc;

    // a context that only points into the static scratch; nothing here is allocated
    pgt_ctx c;
    c.device = device;
    c.num_sms = ds.num_sms;
    c.max_groups = PGT_NOALLOC_MAX_GROUPS;
    c.flags = 0;
    c.d_counters = ds.scratch;
    c.d_done = ds.scratch + pgt::kCounterStride * PGT_NOALLOC_MAX_GROUPS;
    // without a caller error word the kernel writes timeouts into a sink line of the array
    // (never through a null pointer); nothing reads it
    c.d_err = d_err != nullptr ? d_err : c.d_done + pgt::kCounterStride;
    c.d_release = nullptr;
    c.d_block = nullptr;
    c.release_armed = false;

    pgt_gemm_desc in = {};
    in.M = M;
    in.N = N;
    in.K = K;
    in.dtype = PGT_BF16;
    in.b_layout = b_layout;
    in.sched_mode = PGT_WORK_STEALING;
    in.group_size = group_size;
    in.ws_groups = ws_groups;
    in.kernel_cfg = PGT_CFG_AUTO;
    pgt_gemm_desc d;
    pgt_gemm_plan_info plan;
    rc = pgt::gemm_plan(&c, &in, &d, &plan);
    if (rc) return rc;
    // the array keeps the previous call's contents: counters, done counter (and the error
    // word when the caller passed none) must start at zero
    const size_t clear_ints = pgt::kCounterStride * (PGT_NOALLOC_MAX_GROUPS + (d_err != nullptr ? 1 : 2));
    if (cudaMemsetAsync(ds.scratch, 0, sizeof(int) * clear_ints, st) != cudaSuccess) return PGT_ERR_CUDA;
    return pgt::gemm_launch(&c, d, plan, A, B, nullptr, nullptr, C, nullptr, 0, nullptr, st);
}
