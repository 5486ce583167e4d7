// Persistent tiled GEMM C = A . B for sm_103a: TMA producer warp, tcgen05 MMA warp issuing
// into double-buffered tensor-memory accumulators, four epilogue warps, an mbarrier
// stage ring, and a tile-id ring that carries the scheduler's choices to every role.
//
// Design source: the warp-specialised persistent kernel of "[Feature] Introduce tile
// scheduler" (tilelang PR #2441, gemm_mxfp8_blockscaled_1d1d.py): TMA warp, MMA warp,
// epilogue warpgroup (threads 128..255), loaded/consumed barriers indexed by
// phase = iter * k_iters + k with stage = phase % stages and parity = (phase / stages) & 1,
// tmem_full / tmem_empty between MMA and epilogue.  Differences: the accumulator is double
// buffered in tensor memory so the epilogue of one tile overlaps the next tile's
// mainloop; the producer runs the scheduler and publishes each tile through a small
// shared-memory ring (needed for work stealing, where roles cannot recompute the tile).
#include <cuda_bf16.h>
#include <stdio.h>

#include "pgt_device.cuh"
#include "pgt_internal.h"
#include "pgt_sched.cuh"

namespace pgt {

struct GemmParams {
    int M, N, K;
    int k_iters;
    SchedParams sp;
    int* err;
    int32_t* tr_visits;
    int64_t tr_max;
    int32_t* tr_counts;
    int64_t* tr_times;
};

constexpr int kThreads = 256;     // warp 0 producer, warp 1 MMA, warps 4-7 epilogue
constexpr int kTileRing = 4;      // tile-id ring depth
constexpr int kEpiWarps = 4;
constexpr int kEpiBufBytes = 32 * 128;  // 32 rows x 64 bf16, 128B-swizzled, per buffer

// Shared-memory layout of the 1-CTA bf16 kernel (offsets from a 1024-aligned base).
template <int BN, int STAGES>
struct Bf16Layout {
    static constexpr int BM = 128, BK = 64;
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int EPI_OFF = STAGES * STAGE_BYTES;
    static constexpr int BAR_OFF = EPI_OFF + kEpiWarps * 2 * kEpiBufBytes;
    // barriers: full[S], empty[S], tfull[2], tempty[2], sfull[Q], sempty[Q], mma_done
    static constexpr int NUM_BARS = 2 * STAGES + 4 + 2 * kTileRing + 1;
    // the ring holds int4 entries: 16-byte aligned
    static constexpr int RING_OFF = BAR_OFF + (NUM_BARS * 8 + 15) / 16 * 16;
    static constexpr int MISC_OFF = RING_OFF + kTileRing * 16;  // tmem slot, abort flag
    static constexpr int BYTES = MISC_OFF + 16;
    static constexpr int SMEM = BYTES + 1024;  // alignment slack
    static constexpr int TMEM_COLS = 2 * BN;
    static_assert(STAGE_BYTES % 1024 == 0 && A_BYTES % 1024 == 0, "stages must keep 1024-byte swizzle alignment");
    static_assert(EPI_OFF % 1024 == 0 && BAR_OFF % 1024 == 0, "epilogue buffers need 1024-byte alignment");
    static_assert(RING_OFF % 16 == 0 && MISC_OFF % 16 == 0, "ring entries are 16-byte vectors");
    static_assert(SMEM <= 232448, "dynamic shared memory above the 227 KB per-CTA limit");
};

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo, uint32_t hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(lo), __uint_as_float(hi));
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// bf16 GEMM, one CTA per worker, 128 x BN output tiles, K step 64 per stage.
// B_MN: B stored K x N (N contiguous); otherwise N x K (K contiguous).
template <int BN, int STAGES, bool B_MN, bool TRACE>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_bf16_1cta_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                          const __grid_constant__ CUtensorMap tmC, const GemmParams gp) {
    using L = Bf16Layout<BN, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);

    const int warp = threadIdx.x >> 5;
    const uint32_t lane = lane_id();

    const uint32_t bar0 = base + L::BAR_OFF;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
    auto tempty = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
    auto sfull = [&](int q) { return bar0 + 8u * (2 * STAGES + 4 + q); };
    auto sempty = [&](int q) { return bar0 + 8u * (2 * STAGES + 4 + kTileRing + q); };
    const uint32_t mma_done = bar0 + 8u * (2 * STAGES + 4 + 2 * kTileRing);
    int4* ring = reinterpret_cast<int4*>(gbase + L::RING_OFF);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gbase + L::MISC_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + L::MISC_OFF + 4);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull(a), 1);
            mbar_init(tempty(a), kEpiWarps);
        }
        for (int q = 0; q < kTileRing; ++q) {
            mbar_init(sfull(q), 1);
            mbar_init(sempty(q), 1 + kEpiWarps);
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc<1>(base + L::MISC_OFF, L::TMEM_COLS);
        tmem_relinquish<1>();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (TRACE && threadIdx.x == 0 && gp.tr_times != nullptr) gp.tr_times[2 * blockIdx.x] = (int64_t)globaltimer();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tensormap(&tmA);
            prefetch_tensormap(&tmB);
            Scheduler sch;
            sch.init(gp.sp, blockIdx.x);
            uint32_t it = 0, qc = 0;
            int nvis = 0;
            bool ok = true;
            while (ok) {
                int t = *abort_flag ? -1 : sch.fetch();
                int m = 0, n = 0;
                if (t >= 0) decode_tile(gp.sp, t, m, n);
                const int q = qc % kTileRing;
                if (!mbar_wait(sempty(q), ((qc / kTileRing) & 1u) ^ 1u, abort_flag, gp.err, kRoleProducer, 0)) break;
                ring[q] = make_int4(t, m, n, 0);
                mbar_arrive(sfull(q));
                ++qc;
                if (t < 0) break;
                if (TRACE && gp.tr_visits != nullptr) {
                    if (nvis < gp.tr_max) {
                        int32_t* r = gp.tr_visits + ((int64_t)blockIdx.x * gp.tr_max + nvis) * PGT_VISIT_FIELDS;
                        r[0] = t;
                        r[1] = m;
                        r[2] = n;
                        r[3] = (int32_t)smid();
                    }
                    ++nvis;
                }
                const int m0 = m * L::BM;
                const int n0 = n * BN;
                for (int k = 0; k < gp.k_iters; ++k, ++it) {
                    const int s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1u;
                    if (!mbar_wait(empty(s), ph ^ 1u, abort_flag, gp.err, kRoleProducer, 1)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = base + s * L::STAGE_BYTES;
                    const uint32_t sb = sa + L::A_BYTES;
                    mbar_arrive_expect_tx(full(s), L::STAGE_BYTES);
                    tma_load_2d(sa, &tmA, full(s), k * L::BK, m0);
                    if constexpr (B_MN) {
#pragma unroll
                        for (int j = 0; j < BN / 64; ++j) tma_load_2d(sb + j * 8192, &tmB, full(s), n0 + 64 * j, k * L::BK);
                    } else {
                        tma_load_2d(sb, &tmB, full(s), k * L::BK, n0);
                    }
                }
            }
            sch.finish();
            if (TRACE && gp.tr_counts != nullptr) gp.tr_counts[blockIdx.x] = nvis;
        }
        __syncwarp();
    } else if (warp == 1) {
        // ----------------------------------------------------------------- MMA
        if (lane == 0) {
            constexpr uint32_t idesc = make_idesc_bf16(128, BN, false, B_MN);
            uint32_t it = 0, qc = 0, tc = 0;
            bool ok = true;
            while (ok) {
                const int q = qc % kTileRing;
                if (!mbar_wait(sfull(q), (qc / kTileRing) & 1u, abort_flag, gp.err, kRoleMma, 2)) break;
                const int t = ring[q].x;
                mbar_arrive(sempty(q));
                ++qc;
                if (t < 0) break;
                const int acc = tc & 1;
                if (!mbar_wait(tempty(acc), ((tc >> 1) & 1u) ^ 1u, abort_flag, gp.err, kRoleMma, 3)) break;
                tc_fence_after();
                const uint32_t d = tmem_base + acc * BN;
                for (int k = 0; k < gp.k_iters; ++k, ++it) {
                    const int s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1u;
                    if (!mbar_wait(full(s), ph, abort_flag, gp.err, kRoleMma, 4)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = base + s * L::STAGE_BYTES;
                    const uint32_t sb = sa + L::A_BYTES;
                    const uint64_t adesc = make_smem_desc(sa, 16, 1024, kLayoutSw128);
                    const uint64_t bdesc = B_MN ? make_smem_desc(sb, 8192, 1024, kLayoutSw128)
                                                : make_smem_desc(sb, 16, 1024, kLayoutSw128);
#pragma unroll
                    for (int kk = 0; kk < L::BK / 16; ++kk) {
                        // K-major operands advance 16 elements = 32 bytes inside the
                        // 128-byte swizzle row; the MN-major B advances 16 rows of 128 bytes.
                        const uint64_t a_k = adesc + (uint64_t)(2 * kk);
                        const uint64_t b_k = bdesc + (uint64_t)(B_MN ? 128 * kk : 2 * kk);
                        mma_bf16<1>(d, a_k, b_k, idesc, (k | kk) != 0 ? 1u : 0u);
                    }
                    mma_commit(empty(s));
                }
                if (!ok) break;
                mma_commit(tfull(acc));
                ++tc;
            }
            // every MMA issued above has completed once this barrier flips
            mma_commit(mma_done);
            volatile int no_abort = 0;
            mbar_wait(mma_done, 0, &no_abort, gp.err, kRoleMma, 5);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------------------ epilogue
        const int qw = warp - 4;  // TMEM lane quarter this warp may access
        const uint32_t epi = base + L::EPI_OFF + qw * 2 * kEpiBufBytes;
        uint32_t qc = 0, tc = 0, chunk = 0;
        while (true) {
            const int q = qc % kTileRing;
            if (!mbar_wait(sfull(q), (qc / kTileRing) & 1u, abort_flag, gp.err, kRoleEpilogue, 6)) break;
            const int4 e = ring[q];
            __syncwarp();
            if (lane == 0) mbar_arrive(sempty(q));
            ++qc;
            if (e.x < 0) break;
            const int acc = tc & 1;
            if (!mbar_wait(tfull(acc), (tc >> 1) & 1u, abort_flag, gp.err, kRoleEpilogue, 7)) break;
            tc_fence_after();
            const int row0 = e.y * L::BM + 32 * qw;
            const int col0 = e.z * BN;
            const uint32_t tacc = tmem_base + ((uint32_t)(32 * qw) << 16) + acc * BN;
#pragma unroll 1
            for (int c = 0; c < BN / 64; ++c, ++chunk) {
                uint32_t r0[32], r1[32];
                tmem_ld_32x32b_x32(tacc + c * 64, r0);
                tmem_ld_32x32b_x32(tacc + c * 64 + 32, r1);
                tmem_ld_wait();
                if (c == BN / 64 - 1) {
                    // accumulator fully read: hand it back to the MMA warp
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(tempty(acc));
                }
                const uint32_t buf = epi + (chunk & 1u) * kEpiBufBytes;
                if (lane == 0) bulk_wait_read<1>();
                __syncwarp();
                const uint32_t rowaddr = buf + lane * 128u;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    st_shared_v4(rowaddr + ((j ^ (lane & 7u)) << 4), pack_bf16x2(r0[8 * j], r0[8 * j + 1]),
                                 pack_bf16x2(r0[8 * j + 2], r0[8 * j + 3]), pack_bf16x2(r0[8 * j + 4], r0[8 * j + 5]),
                                 pack_bf16x2(r0[8 * j + 6], r0[8 * j + 7]));
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    st_shared_v4(rowaddr + (((j + 4) ^ (lane & 7u)) << 4), pack_bf16x2(r1[8 * j], r1[8 * j + 1]),
                                 pack_bf16x2(r1[8 * j + 2], r1[8 * j + 3]), pack_bf16x2(r1[8 * j + 4], r1[8 * j + 5]),
                                 pack_bf16x2(r1[8 * j + 6], r1[8 * j + 7]));
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    const int x = col0 + 64 * c;
                    if (row0 < gp.M && x < gp.N) tma_store_2d(&tmC, buf, x, row0);
                    bulk_commit();
                }
            }
            ++tc;
        }
        if (lane == 0) bulk_wait<0>();
        __syncwarp();
    }

    __syncthreads();
    if (TRACE && threadIdx.x == 0 && gp.tr_times != nullptr) gp.tr_times[2 * blockIdx.x + 1] = (int64_t)globaltimer();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<1>(tmem_base, L::TMEM_COLS);
    }
}

// ============================================================================ host side
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (fn == nullptr) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

inline int64_t cdiv64(int64_t a, int64_t b) { return (a + b - 1) / b; }

struct CfgShape {
    int bm, bn, bk, cs, stages, smem;
};

bool cfg_shape(int cfg, int dtype, CfgShape* s) {
    if (dtype == PGT_BF16) {
        switch (cfg) {
            case PGT_CFG_1CTA_128x128:
                *s = {128, 128, 64, 1, 6, Bf16Layout<128, 6>::SMEM};
                return true;
            case PGT_CFG_1CTA_128x256:
                *s = {128, 256, 64, 1, 4, Bf16Layout<256, 4>::SMEM};
                return true;
            default:
                return false;
        }
    }
    return false;
}

template <int BN, int S, bool BMN, bool TR>
int launch_bf16_1cta(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc, const GemmParams& gp,
                     int ctas, int device, cudaStream_t st) {
    auto kern = gemm_bf16_1cta_kernel<BN, S, BMN, TR>;
    constexpr int smem = Bf16Layout<BN, S>::SMEM;
    static bool attr_done[64] = {};
    if (device < 0 || device >= 64) return PGT_ERR_ARG;
    if (!attr_done[device]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
            return PGT_ERR_CUDA;
        attr_done[device] = true;
    }
    kern<<<ctas, kThreads, smem, st>>>(ta, tb, tc, gp);
    return cuda_status(cudaGetLastError());
}

template <int BN, int S>
int dispatch_bf16_1cta(bool bmn, bool trace, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                       const GemmParams& gp, int ctas, int device, cudaStream_t st) {
    if (bmn) {
        return trace ? launch_bf16_1cta<BN, S, true, true>(ta, tb, tc, gp, ctas, device, st)
                     : launch_bf16_1cta<BN, S, true, false>(ta, tb, tc, gp, ctas, device, st);
    }
    return trace ? launch_bf16_1cta<BN, S, false, true>(ta, tb, tc, gp, ctas, device, st)
                 : launch_bf16_1cta<BN, S, false, false>(ta, tb, tc, gp, ctas, device, st);
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

int encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                   uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return PGT_ERR_CUDA;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PGT_OK : PGT_ERR_CUDA;
}

size_t gemm_workspace_bytes(const pgt_gemm_desc& d) {
    (void)d;
    return 0;
}

int gemm_plan(const pgt_ctx* ctx, const pgt_gemm_desc* in, pgt_gemm_desc* d, pgt_gemm_plan_info* p) {
    if (ctx == nullptr || in == nullptr || p == nullptr || d == nullptr) return PGT_ERR_ARG;
    *d = *in;
    const int64_t lim = (int64_t)1 << 31;
    if (d->M < 1 || d->N < 1 || d->K < 1 || d->M >= lim || d->N >= lim || d->K >= lim) return PGT_ERR_ARG;
    if (d->dtype != PGT_BF16 && d->dtype != PGT_MXFP8) return PGT_ERR_ARG;
    if (d->b_layout != PGT_B_KN && d->b_layout != PGT_B_NK) return PGT_ERR_ARG;
    if (d->sched_mode < PGT_BLOCKED || d->sched_mode > PGT_BLOCKED_GROUPED_M) return PGT_ERR_ARG;
    if (d->group_size < 1) return PGT_ERR_ARG;
    if (d->num_workers < 0) return PGT_ERR_ARG;
    if (d->ws_groups == 0) d->ws_groups = ctx->max_groups < 8 ? ctx->max_groups : 8;
    if (d->ws_groups < 1 || d->ws_groups > ctx->max_groups) return PGT_ERR_GROUPS;
    const int64_t es = d->dtype == PGT_BF16 ? 2 : 1;
    const int64_t b_inner = d->b_layout == PGT_B_KN ? d->N : d->K;
    if (d->lda == 0) d->lda = d->K;
    if (d->ldb == 0) d->ldb = b_inner;
    if (d->ldc == 0) d->ldc = d->N;
    if (d->lda < d->K || d->ldb < b_inner || d->ldc < d->N) return PGT_ERR_ARG;
    if (d->lda >= lim || d->ldb >= lim || d->ldc >= lim) return PGT_ERR_ARG;
    if ((d->lda * es) % 16 || (d->ldb * es) % 16 || (d->ldc * 2) % 16) return PGT_ERR_ALIGN;
    if (d->dtype == PGT_MXFP8) {
        if (d->K % 128 != 0 || d->b_layout != PGT_B_NK) return PGT_ERR_ARG;
    }
    if (d->kernel_cfg == PGT_CFG_AUTO) d->kernel_cfg = d->dtype == PGT_BF16 ? PGT_CFG_1CTA_128x256 : PGT_CFG_AUTO;
    CfgShape s;
    if (!cfg_shape(d->kernel_cfg, d->dtype, &s)) return PGT_ERR_UNSUPPORTED;
    const int64_t m_blocks = cdiv64(d->M, s.bm);
    const int64_t n_blocks = cdiv64(d->N, s.bn);
    const int64_t m_tiles = cdiv64(m_blocks, s.cs);
    const int64_t tiles = m_tiles * n_blocks;
    if (tiles >= lim) return PGT_ERR_ARG;
    int64_t workers = d->num_workers;
    if (workers == 0) {
        workers = ctx->num_sms / s.cs;
        if (workers > tiles) workers = tiles;
        if (workers < 1) workers = 1;
    }
    if (workers * s.cs >= lim) return PGT_ERR_ARG;
    p->kernel_cfg = d->kernel_cfg;
    p->bm = s.bm;
    p->bn = s.bn;
    p->bk = s.bk;
    p->cluster_size = s.cs;
    p->stages = s.stages;
    p->m_blocks = (int32_t)m_blocks;
    p->n_blocks = (int32_t)n_blocks;
    p->m_tiles = (int32_t)m_tiles;
    p->tiles = (int32_t)tiles;
    p->workers = (int32_t)workers;
    p->ctas = (int32_t)(workers * s.cs);
    p->k_iters = (int32_t)cdiv64(d->K, s.bk);
    p->smem_bytes = s.smem;
    return PGT_OK;
}

int gemm_launch(pgt_ctx* ctx, const pgt_gemm_desc& d, const pgt_gemm_plan_info& plan, const void* A, const void* B,
                const uint8_t* sfa, const uint8_t* sfb, void* C, void* workspace, size_t workspace_bytes,
                const pgt_trace* trace, cudaStream_t stream) {
    if (A == nullptr || B == nullptr || C == nullptr) return PGT_ERR_ARG;
    if (!aligned16(A) || !aligned16(B) || !aligned16(C)) return PGT_ERR_ALIGN;
    if (d.dtype == PGT_BF16 && (sfa != nullptr || sfb != nullptr)) return PGT_ERR_ARG;
    const size_t ws_need = gemm_workspace_bytes(d);
    if (ws_need > 0 && (workspace == nullptr || workspace_bytes < ws_need)) return PGT_ERR_WORKSPACE;
    if (trace != nullptr) {
        if (trace->visits == nullptr || trace->counts == nullptr || trace->max_visits < 1) return PGT_ERR_ARG;
    }
    if (d.dtype != PGT_BF16 || plan.cluster_size != 1) return PGT_ERR_UNSUPPORTED;

    GemmParams gp;
    gp.M = (int)d.M;
    gp.N = (int)d.N;
    gp.K = (int)d.K;
    gp.k_iters = plan.k_iters;
    gp.sp.tiles = plan.tiles;
    gp.sp.m_tiles = plan.m_tiles;
    gp.sp.n_tiles = plan.n_blocks;
    gp.sp.mode = d.sched_mode;
    int g = d.group_size;
    if (d.sched_mode == PGT_BLOCKED_GROUPED_M) {
        if (g > plan.m_tiles) g = plan.m_tiles;
    } else if (g > plan.n_blocks) {
        g = plan.n_blocks;
    }
    gp.sp.group = g;
    gp.sp.ws_groups = d.ws_groups;
    gp.sp.workers = plan.workers;
    gp.sp.counters = ctx->d_counters;
    gp.sp.done = ctx->d_done;
    gp.err = ctx->d_err;
    gp.tr_visits = trace ? trace->visits : nullptr;
    gp.tr_max = trace ? trace->max_visits : 0;
    gp.tr_counts = trace ? trace->counts : nullptr;
    gp.tr_times = trace ? trace->times_ns : nullptr;

    if (d.sched_mode == PGT_WORK_STEALING && (ctx->flags & PGT_FLAG_HOST_RESET)) {
        if (cudaMemsetAsync(ctx->d_counters, 0, sizeof(int) * 32 * (ctx->max_groups + 1), stream) != cudaSuccess)
            return PGT_ERR_CUDA;
    }

    const bool bmn = d.b_layout == PGT_B_KN;
    CUtensorMap ta, tb, tc;
    int rc = encode_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, A, d.K, d.M, d.lda * 2, 64, 128,
                            CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
    if (bmn)
        rc = encode_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, B, d.N, d.K, d.ldb * 2, 64, 64,
                            CU_TENSOR_MAP_SWIZZLE_128B);
    else
        rc = encode_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, B, d.K, d.N, d.ldb * 2, 64, plan.bn,
                            CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
    rc = encode_tmap_2d(&tc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, C, d.N, d.M, d.ldc * 2, 64, 32,
                        CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;

    const bool tr = trace != nullptr;
    if (plan.kernel_cfg == PGT_CFG_1CTA_128x256)
        return dispatch_bf16_1cta<256, 4>(bmn, tr, ta, tb, tc, gp, plan.ctas, ctx->device, stream);
    if (plan.kernel_cfg == PGT_CFG_1CTA_128x128)
        return dispatch_bf16_1cta<128, 6>(bmn, tr, ta, tb, tc, gp, plan.ctas, ctx->device, stream);
    return PGT_ERR_UNSUPPORTED;
}

}  // namespace pgt
