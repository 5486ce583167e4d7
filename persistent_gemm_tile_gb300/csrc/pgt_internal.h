// Host-side internals shared by the library's translation units (not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pgt.h"

struct pgt_ctx {
    int device;
    int num_sms;
    int max_groups;
    int flags;
    int* d_counters;  // max_groups counters, kCounterStride ints apart, zero between launches
    int* d_done;      // work-stealing done counter (own 128-byte line)
    int* d_err;       // device error word: code, role, block, site
    int* d_release;   // work-stealing release flags, one int per group (two 128-byte lines)
    void* d_block;    // the single allocation holding the three above
    bool release_armed;  // pgt_set_release was called: kernels read the flags (else they skip them)
};

namespace pgt {

constexpr int kMaxGroups = 64;
constexpr int kMaxWsWorkers = 65535;  // work stealing's 32-bit group arithmetic (pgt_sched.cuh)

// Status from a CUDA runtime result.
inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? PGT_OK : PGT_ERR_CUDA; }

// 2-D tiled tensor map over a row-major matrix: `inner` elements per row (contiguous),
// `outer` rows, `row_bytes` between rows; box of box_inner x box_outer elements.
int encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner,
                   uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                   CUtensorMapSwizzle swizzle);

// Validates `desc`, applies defaults and fills the launch plan (no device work).
int gemm_plan(const pgt_ctx* ctx, const pgt_gemm_desc* desc, pgt_gemm_desc* resolved,
              pgt_gemm_plan_info* plan);

int gemm_launch(pgt_ctx* ctx, const pgt_gemm_desc& d, const pgt_gemm_plan_info& plan, const void* A,
                const void* B, const uint8_t* sfa, const uint8_t* sfb, void* C, void* workspace,
                size_t workspace_bytes, const pgt_trace* trace, cudaStream_t stream);

size_t gemm_workspace_bytes(const pgt_gemm_desc& d);

int add_launch(pgt_ctx* ctx, const float* x, const float* y, float* out, int64_t rows, int64_t cols,
               int64_t ldx, int64_t ldy, int64_t ldo, int sched_mode, int tile_r, int tile_c,
               int num_workers, const pgt_trace* trace, cudaStream_t stream);

int add_workers(const pgt_ctx* ctx, int64_t rows, int64_t cols, int tile_r, int tile_c, int sched_mode,
                int num_workers);

int schedule_log_launch(pgt_ctx* ctx, int64_t m_blocks, int64_t n_blocks, int cluster_size,
                        int sched_mode, int group_size, int ws_groups, int ws_layout, int num_workers,
                        const pgt_trace* trace, cudaStream_t stream);

}  // namespace pgt
