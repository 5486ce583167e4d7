// The C ABI (pgt.h): context creation, argument checks, the schedule-log kernel, error
// reporting, and the flat / end-to-end GEMM forms.
#include <stdlib.h>
#include <string.h>

#include "pgt_device.cuh"
#include "pgt_internal.h"
#include "pgt_sched.cuh"

namespace pgt {

// One thread per worker runs the device scheduler and records its visits (no GEMM work).
// Launch control: one block per tile; a running block takes its own tile, then the tiles
// of blocks it cancels before they start.
__global__ void schedule_log_kernel(const SchedParams sp, int32_t* visits, int64_t max_visits, int32_t* counts,
                                    int64_t* times, int* err) {
    __shared__ __align__(16) uint8_t clc_resp[16];
    __shared__ __align__(8) uint64_t clc_bar_word;
    if (threadIdx.x != 0) return;
    const int w = blockIdx.x;
    if (times != nullptr) times[2 * w] = (int64_t)globaltimer();
    Scheduler sch;
    sch.init(sp, w);
    const bool clc = sp.mode == kLaunchControl;
    const uint32_t clc_bar = smem_u32(&clc_bar_word), resp = smem_u32(clc_resp);
    if (clc) {
        mbar_init(clc_bar, 1);
        fence_mbar_init();
    }
    volatile int abort_local = 0;
    uint32_t phase = 0;
    int next = w;
    int n = 0;
    for (;;) {
        int t;
        if (clc) {
            t = next;
            if (t < 0) break;
            mbar_arrive_expect_tx(clc_bar, 16);
            clc_try_cancel(resp, clc_bar);
            next = -1;
            volatile int no_abort = 0;
            if (mbar_wait(clc_bar, phase & 1u, &no_abort, err, kRoleScheduler, 11) && !abort_local) {
                const int x = clc_query(resp);
                next = (x < 0 || x >= sp.tiles) ? -1 : x;
            }
            ++phase;
        } else {
            t = sch.fetch();
        }
        if (t < 0) break;
        int m, nn;
        decode_tile(sp, t, m, nn);
        if (n < max_visits) {
            int32_t* r = visits + ((int64_t)w * max_visits + n) * PGT_VISIT_FIELDS;
            r[0] = t;
            r[1] = m;
            r[2] = nn;
            r[3] = (int32_t)smid();
        }
        ++n;
    }
    sch.finish();
    counts[w] = n;
    if (times != nullptr) times[2 * w + 1] = (int64_t)globaltimer();
}

// Self-test of the bounded waits: one thread waits on an mbarrier that only `arrive` makes
// complete.  Without it the wait gives up after the kernels' time limit, records the
// timeout in the error word and the kernel returns.
__global__ void wait_probe_kernel(int arrive, int* err) {
    __shared__ __align__(8) uint64_t bar_word;
    const uint32_t bar = smem_u32(&bar_word);
    mbar_init(bar, 1);
    fence_mbar_init();
    if (arrive) mbar_arrive(bar);
    volatile int abort_flag = 0;
    mbar_wait(bar, 0, &abort_flag, err, kRoleScheduler, 12);
}

int schedule_log_launch(pgt_ctx* ctx, int64_t m_blocks, int64_t n_blocks, int cluster_size, int sched_mode,
                        int group_size, int ws_groups, int ws_layout, int num_workers, const pgt_trace* trace,
                        cudaStream_t stream) {
    if (ctx == nullptr || trace == nullptr || trace->visits == nullptr || trace->counts == nullptr ||
        trace->max_visits < 1)
        return PGT_ERR_ARG;
    if (m_blocks < 1 || n_blocks < 1 || (cluster_size != 1 && cluster_size != 2)) return PGT_ERR_ARG;
    if (sched_mode < PGT_BLOCKED || sched_mode > PGT_LAUNCH_CONTROL || group_size < 1 || num_workers < 1)
        return PGT_ERR_ARG;
    if (ws_groups < 1 || ws_groups > ctx->max_groups) return PGT_ERR_GROUPS;
    if (ws_layout != PGT_WS_RANGES && ws_layout != PGT_WS_STRIPED) return PGT_ERR_ARG;
    const int64_t m_tiles = (m_blocks + cluster_size - 1) / cluster_size;
    const int64_t tiles = m_tiles * n_blocks;
    if (m_blocks >= ((int64_t)1 << 31) || n_blocks >= ((int64_t)1 << 31) || tiles >= ((int64_t)1 << 31))
        return PGT_ERR_ARG;
    if (sched_mode == PGT_LAUNCH_CONTROL && num_workers != tiles) return PGT_ERR_ARG;  // one per tile
    if (sched_mode == PGT_WORK_STEALING && num_workers > kMaxWsWorkers) return PGT_ERR_ARG;
    SchedParams sp;
    sp.tiles = (int)tiles;
    sp.m_tiles = (int)m_tiles;
    sp.n_tiles = (int)n_blocks;
    sp.mode = sched_mode;
    int g = group_size;
    if (sched_mode == PGT_BLOCKED_GROUPED_M) {
        if (g > sp.m_tiles) g = sp.m_tiles;
    } else if (g > sp.n_tiles) {
        g = sp.n_tiles;
    }
    sp.group = g;
    sp.ws_groups = ws_groups < num_workers ? ws_groups : num_workers;  // every group has a home worker
    sp.ws_layout = ws_layout;
    sp.workers = num_workers;
    sp.counters = ctx->d_counters;
    sp.done = ctx->d_done;
    sp.release = ctx->release_armed ? ctx->d_release : nullptr;
    if (sched_mode == PGT_WORK_STEALING && (ctx->flags & PGT_FLAG_HOST_RESET)) {
        if (cudaMemsetAsync(ctx->d_counters, 0, sizeof(int) * kCounterStride * (ctx->max_groups + 1), stream) !=
            cudaSuccess)
            return PGT_ERR_CUDA;
    }
    schedule_log_kernel<<<num_workers, 32, 0, stream>>>(sp, trace->visits, trace->max_visits, trace->counts,
                                                       trace->times_ns, ctx->d_err);
    return cuda_status(cudaGetLastError());
}

}  // namespace pgt

using namespace pgt;

extern "C" {

int pgt_preamble(int device, int max_groups, int flags, pgt_ctx** out) {
    if (out == nullptr) return PGT_ERR_ARG;
    *out = nullptr;
    if (max_groups < 1 || max_groups > kMaxGroups || (flags & ~PGT_FLAG_HOST_RESET) != 0) return PGT_ERR_ARG;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess) return PGT_ERR_CUDA;
    if (device < 0 || device >= ndev) return PGT_ERR_ARG;
    if (cudaSetDevice(device) != cudaSuccess) return PGT_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || sms < 1)
        return PGT_ERR_CUDA;
    // counters: max_groups lines, then the done counter's line, the error word's line and
    // two lines of release flags
    const size_t bytes = sizeof(int) * kCounterStride * (max_groups + 4);
    void* blk = nullptr;
    if (cudaMalloc(&blk, bytes) != cudaSuccess) return PGT_ERR_CUDA;
    if (cudaMemset(blk, 0, bytes) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
        cudaFree(blk);
        return PGT_ERR_CUDA;
    }
    pgt_ctx* c = static_cast<pgt_ctx*>(calloc(1, sizeof(pgt_ctx)));
    if (c == nullptr) {
        cudaFree(blk);
        return PGT_ERR_ARG;
    }
    c->device = device;
    c->num_sms = sms;
    c->max_groups = max_groups;
    c->flags = flags;
    c->d_block = blk;
    c->d_counters = static_cast<int*>(blk);
    c->d_done = c->d_counters + kCounterStride * max_groups;
    c->d_err = c->d_done + kCounterStride;
    c->d_release = c->d_err + kCounterStride;
    *out = c;
    return PGT_OK;
}

int pgt_destroy(pgt_ctx* ctx) {
    if (ctx == nullptr) return PGT_OK;
    int rc = PGT_OK;
    int prev = -1;
    cudaGetDevice(&prev);
    if (cudaSetDevice(ctx->device) != cudaSuccess) rc = PGT_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) rc = PGT_ERR_CUDA;
    if (cudaFree(ctx->d_block) != cudaSuccess) rc = PGT_ERR_CUDA;
    if (prev >= 0) cudaSetDevice(prev);
    free(ctx);
    return rc;
}

int pgt_set_release(pgt_ctx* ctx, const int32_t* h_flags, int n, void* stream) {
    if (ctx == nullptr || h_flags == nullptr || n < 1 || n > ctx->max_groups) return PGT_ERR_ARG;
    if (cudaSetDevice(ctx->device) != cudaSuccess) return PGT_ERR_CUDA;
    // from now on work-stealing launches read the flags (until then they skip the reads)
    ctx->release_armed = true;
    return cuda_status(cudaMemcpyAsync(ctx->d_release, h_flags, sizeof(int32_t) * n, cudaMemcpyHostToDevice,
                                       static_cast<cudaStream_t>(stream)));
}

int pgt_wait_probe(pgt_ctx* ctx, int arrive, void* stream) {
    if (ctx == nullptr) return PGT_ERR_ARG;
    if (cudaSetDevice(ctx->device) != cudaSuccess) return PGT_ERR_CUDA;
    wait_probe_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(arrive != 0, ctx->d_err);
    return cuda_status(cudaGetLastError());
}

int pgt_num_sms(const pgt_ctx* ctx) { return ctx ? ctx->num_sms : PGT_ERR_ARG; }

int pgt_max_groups(const pgt_ctx* ctx) { return ctx ? ctx->max_groups : PGT_ERR_ARG; }

int pgt_last_error(pgt_ctx* ctx, void* stream, int32_t* detail) {
    if (ctx == nullptr) return PGT_ERR_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return PGT_ERR_CUDA;
    int32_t w[4] = {0, 0, 0, 0};
    if (cudaMemcpy(w, ctx->d_err, sizeof(w), cudaMemcpyDeviceToHost) != cudaSuccess) return PGT_ERR_CUDA;
    if (detail != nullptr) memcpy(detail, w, sizeof(w));
    if (w[0] != 0) {
        if (cudaMemset(ctx->d_err, 0, sizeof(w)) != cudaSuccess) return PGT_ERR_CUDA;
        // a launch that gave up may have left work-stealing counters mid-way
        if (cudaMemset(ctx->d_counters, 0, sizeof(int) * kCounterStride * (ctx->max_groups + 1)) != cudaSuccess)
            return PGT_ERR_CUDA;
        if (cudaDeviceSynchronize() != cudaSuccess) return PGT_ERR_CUDA;
        return PGT_ERR_TIMEOUT;
    }
    return PGT_OK;
}

const char* pgt_strerror(int status) {
    switch (status) {
        case PGT_OK: return "ok";
        case PGT_ERR_ARG: return "invalid argument";
        case PGT_ERR_ALIGN: return "pointer or row stride not 16-byte aligned";
        case PGT_ERR_UNSUPPORTED: return "no kernel for this configuration";
        case PGT_ERR_CUDA: return "CUDA call failed";
        case PGT_ERR_TIMEOUT: return "device wait timed out";
        case PGT_ERR_GROUPS: return "ws_groups outside [1, max_groups]";
        case PGT_ERR_WORKSPACE: return "workspace missing or too small";
        case PGT_ERR_CAPACITY: return "trace buffer too small";
        default: return "unknown status";
    }
}

size_t pgt_gemm_workspace_bytes(const pgt_gemm_desc* desc) {
    if (desc == nullptr) return 0;
    return gemm_workspace_bytes(*desc);
}

int pgt_gemm_plan(const pgt_ctx* ctx, const pgt_gemm_desc* desc, pgt_gemm_plan_info* out) {
    pgt_gemm_desc d;
    if (ctx == nullptr) return PGT_ERR_ARG;
    if (cudaSetDevice(ctx->device) != cudaSuccess) return PGT_ERR_CUDA;
    return gemm_plan(ctx, desc, &d, out);
}

int pgt_gemm_ex(pgt_ctx* ctx, const pgt_gemm_desc* desc, const void* A, const void* B, const uint8_t* sfa,
                const uint8_t* sfb, void* C, void* workspace, size_t workspace_bytes, const pgt_trace* trace,
                void* stream) {
    pgt_gemm_desc d;
    pgt_gemm_plan_info plan;
    if (ctx == nullptr) return PGT_ERR_ARG;
    if (cudaSetDevice(ctx->device) != cudaSuccess) return PGT_ERR_CUDA;
    int rc = gemm_plan(ctx, desc, &d, &plan);
    if (rc) return rc;
    return gemm_launch(ctx, d, plan, A, B, sfa, sfb, C, workspace, workspace_bytes, trace,
                       static_cast<cudaStream_t>(stream));
}

int pgt_gemm(pgt_ctx* ctx, const void* A, const void* B, const uint8_t* sfa, const uint8_t* sfb, void* C, int64_t M,
             int64_t N, int64_t K, int dtype, int b_layout, int sched_mode, int group_size, int ws_groups,
             void* workspace, size_t workspace_bytes, void* stream) {
    if (ws_groups < 0 || ws_groups > kMaxGroups) return PGT_ERR_GROUPS;  // no context can hold that many
    pgt_gemm_desc d;
    memset(&d, 0, sizeof(d));
    d.ws_groups = ws_groups;
    d.M = M;
    d.N = N;
    d.K = K;
    d.dtype = dtype;
    d.b_layout = b_layout;
    d.sched_mode = sched_mode;
    d.group_size = group_size;
    return pgt_gemm_ex(ctx, &d, A, B, sfa, sfb, C, workspace, workspace_bytes, nullptr, stream);
}

int pgt_gemm_host(pgt_ctx* ctx, const pgt_gemm_desc* desc, const void* h_A, const void* h_B, const uint8_t* h_sfa,
                  const uint8_t* h_sfb, void* h_C, void* d_A, void* d_B, uint8_t* d_sfa, uint8_t* d_sfb, void* d_C,
                  void* workspace, size_t workspace_bytes, void* stream) {
    pgt_gemm_desc d;
    pgt_gemm_plan_info plan;
    if (ctx == nullptr) return PGT_ERR_ARG;
    if (cudaSetDevice(ctx->device) != cudaSuccess) return PGT_ERR_CUDA;
    int rc = gemm_plan(ctx, desc, &d, &plan);
    if (rc) return rc;
    if (h_A == nullptr || h_B == nullptr || h_C == nullptr || d_A == nullptr || d_B == nullptr || d_C == nullptr)
        return PGT_ERR_ARG;
    const bool mx = d.dtype == PGT_MXFP8;
    if (mx && (h_sfa == nullptr || h_sfb == nullptr || d_sfa == nullptr || d_sfb == nullptr)) return PGT_ERR_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t es = mx ? 1 : 2;
    const size_t b_rows = d.b_layout == PGT_B_KN ? (size_t)d.K : (size_t)d.N;
    const size_t b_inner = d.b_layout == PGT_B_KN ? (size_t)d.N : (size_t)d.K;
    if (cudaMemcpy2DAsync(d_A, d.lda * es, h_A, d.K * es, d.K * es, d.M, cudaMemcpyHostToDevice, st) != cudaSuccess)
        return PGT_ERR_CUDA;
    if (cudaMemcpy2DAsync(d_B, d.ldb * es, h_B, b_inner * es, b_inner * es, b_rows, cudaMemcpyHostToDevice, st) !=
        cudaSuccess)
        return PGT_ERR_CUDA;
    if (mx) {
        if (cudaMemcpyAsync(d_sfa, h_sfa, (size_t)d.M * (d.K / 128), cudaMemcpyHostToDevice, st) != cudaSuccess ||
            cudaMemcpyAsync(d_sfb, h_sfb, (size_t)d.N * (d.K / 128), cudaMemcpyHostToDevice, st) != cudaSuccess)
            return PGT_ERR_CUDA;
    }
    rc = gemm_launch(ctx, d, plan, d_A, d_B, mx ? d_sfa : nullptr, mx ? d_sfb : nullptr, d_C, workspace,
                     workspace_bytes, nullptr, st);
    if (rc) return rc;
    if (cudaMemcpy2DAsync(h_C, d.N * 2, d_C, d.ldc * 2, d.N * 2, d.M, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return PGT_ERR_CUDA;
    return PGT_OK;
}

int pgt_add(pgt_ctx* ctx, const float* x, const float* y, float* out, int64_t rows, int64_t cols, int64_t ldx,
            int64_t ldy, int64_t ldo, int sched_mode, int tile_r, int tile_c, int num_workers,
            const pgt_trace* trace, void* stream) {
    if (ctx == nullptr) return PGT_ERR_ARG;
    if (cudaSetDevice(ctx->device) != cudaSuccess) return PGT_ERR_CUDA;
    return add_launch(ctx, x, y, out, rows, cols, ldx, ldy, ldo, sched_mode, tile_r, tile_c, num_workers, trace,
                      static_cast<cudaStream_t>(stream));
}

int pgt_add_workers(const pgt_ctx* ctx, int64_t rows, int64_t cols, int tile_r, int tile_c, int sched_mode,
                    int num_workers) {
    return add_workers(ctx, rows, cols, tile_r, tile_c, sched_mode, num_workers);
}

int pgt_schedule_log(pgt_ctx* ctx, int64_t m_blocks, int64_t n_blocks, int cluster_size, int sched_mode,
                     int group_size, int ws_groups, int ws_layout, int num_workers, const pgt_trace* trace,
                     void* stream) {
    if (ctx == nullptr) return PGT_ERR_ARG;
    if (cudaSetDevice(ctx->device) != cudaSuccess) return PGT_ERR_CUDA;
    return schedule_log_launch(ctx, m_blocks, n_blocks, cluster_size, sched_mode, group_size, ws_groups, ws_layout,
                               num_workers, trace, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
