// Host side of the persistent tiled GEMM: configuration table, launch plan, tensor maps,
// scale repack and cluster launch.  The kernels are in pgt_gemm_kernel.cuh.
#include <mutex>

#include "pgt_gemm_kernel.cuh"
#include "pgt_internal.h"

namespace pgt {

// ============================================================================ host side
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::mutex mu;
    static EncodeTiledFn fn = nullptr;
    std::lock_guard<std::mutex> lock(mu);
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
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Stage counts per configuration (the Layout static_asserts check they fit).
template <int CS, int BN, bool MX>
struct Stages;
template <> struct Stages<1, 128, false> { static constexpr int value = 6; };
template <> struct Stages<1, 256, false> { static constexpr int value = 4; };
template <> struct Stages<2, 128, false> { static constexpr int value = 8; };
template <> struct Stages<2, 256, false> { static constexpr int value = 6; };
template <> struct Stages<1, 128, true> { static constexpr int value = 5; };
template <> struct Stages<1, 256, true> { static constexpr int value = 4; };
template <> struct Stages<2, 128, true> { static constexpr int value = 7; };
template <> struct Stages<2, 256, true> { static constexpr int value = 6; };
template <> struct Stages<2, 224, true> { static constexpr int value = 6; };

struct CfgShape {
    int cs, bn, stages, smem, bk;
};

template <int CS, int BN, bool MX>
CfgShape shape_of() {
    using L = Layout<CS, BN, Stages<CS, BN, MX>::value, MX>;
    return {CS, BN, Stages<CS, BN, MX>::value, L::SMEM, L::BK};
}

bool cfg_shape(int cfg, int dtype, CfgShape* s) {
    const bool mx = dtype == PGT_MXFP8;
    switch (cfg) {
        case PGT_CFG_1CTA_128x128: *s = mx ? shape_of<1, 128, true>() : shape_of<1, 128, false>(); return true;
        case PGT_CFG_1CTA_128x256: *s = mx ? shape_of<1, 256, true>() : shape_of<1, 256, false>(); return true;
        case PGT_CFG_2CTA_256x128: *s = mx ? shape_of<2, 128, true>() : shape_of<2, 128, false>(); return true;
        case PGT_CFG_2CTA_256x256: *s = mx ? shape_of<2, 256, true>() : shape_of<2, 256, false>(); return true;
        case PGT_CFG_2CTA_256x224:
            if (!mx) return false;  // MXFP8 only: bf16 keeps two 256-column accumulators already
            *s = shape_of<2, 224, true>();
            return true;
        default: return false;
    }
}

using KernelFn = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, GemmParams);

template <int CS, int BN, bool BMN, bool MX, bool TR>
KernelFn kernel_ptr() {
    return reinterpret_cast<KernelFn>(&gemm_kernel<CS, BN, Stages<CS, BN, MX>::value, BMN, MX, TR>);
}

template <int CS, int BN, bool MX>
KernelFn pick_layout_trace(bool bmn, bool tr) {
    if constexpr (MX) {
        return tr ? kernel_ptr<CS, BN, false, true, true>() : kernel_ptr<CS, BN, false, true, false>();
    } else {
        if (bmn) return tr ? kernel_ptr<CS, BN, true, false, true>() : kernel_ptr<CS, BN, true, false, false>();
        return tr ? kernel_ptr<CS, BN, false, false, true>() : kernel_ptr<CS, BN, false, false, false>();
    }
}

KernelFn pick_kernel(int cfg, bool mx, bool bmn, bool tr) {
    switch (cfg) {
        case PGT_CFG_1CTA_128x128: return mx ? pick_layout_trace<1, 128, true>(bmn, tr) : pick_layout_trace<1, 128, false>(bmn, tr);
        case PGT_CFG_1CTA_128x256: return mx ? pick_layout_trace<1, 256, true>(bmn, tr) : pick_layout_trace<1, 256, false>(bmn, tr);
        case PGT_CFG_2CTA_256x128: return mx ? pick_layout_trace<2, 128, true>(bmn, tr) : pick_layout_trace<2, 128, false>(bmn, tr);
        case PGT_CFG_2CTA_256x256: return mx ? pick_layout_trace<2, 256, true>(bmn, tr) : pick_layout_trace<2, 256, false>(bmn, tr);
        case PGT_CFG_2CTA_256x224: return mx ? pick_layout_trace<2, 224, true>(bmn, tr) : nullptr;
        default: return nullptr;
    }
}

constexpr int kMaxDevices = 64;
constexpr int kNumCfgSlots = (PGT_CFG_2CTA_256x224 + 1) * 2 * 2 * 2;  // cfg x mx x bmn x trace

// Per device and kernel: dynamic shared memory attribute set, and how many workers
// (CTAs or CTA pairs) fit on the GPU at once.
struct KernelInfo {
    bool ready;
    int max_workers;
};
KernelInfo g_kinfo[kMaxDevices][kNumCfgSlots];
std::mutex g_kinfo_mutex;

int kernel_info(int device, int cfg, bool mx, bool bmn, bool tr, const CfgShape& s, KernelInfo* out) {
    if (device < 0 || device >= kMaxDevices) return PGT_ERR_ARG;
    const int slot = ((cfg * 2 + (int)mx) * 2 + (int)bmn) * 2 + (int)tr;
    std::lock_guard<std::mutex> lock(g_kinfo_mutex);
    KernelInfo& ki = g_kinfo[device][slot];
    if (!ki.ready) {
        KernelFn k = pick_kernel(cfg, mx, bmn, tr);
        if (k == nullptr) return PGT_ERR_UNSUPPORTED;
        if (cudaFuncSetAttribute(reinterpret_cast<const void*>(k), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 s.smem) != cudaSuccess)
            return PGT_ERR_CUDA;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return PGT_ERR_CUDA;
        int workers = sms / s.cs;
        if (s.cs > 1) {
            cudaLaunchConfig_t lc = {};
            cudaLaunchAttribute at[1];
            at[0].id = cudaLaunchAttributeClusterDimension;
            at[0].val.clusterDim.x = s.cs;
            at[0].val.clusterDim.y = 1;
            at[0].val.clusterDim.z = 1;
            lc.gridDim = dim3(s.cs * workers, 1, 1);
            lc.blockDim = dim3(kThreads, 1, 1);
            lc.dynamicSmemBytes = s.smem;
            lc.attrs = at;
            lc.numAttrs = 1;
            int clusters = 0;
            if (cudaOccupancyMaxActiveClusters(&clusters, reinterpret_cast<const void*>(k), &lc) == cudaSuccess &&
                clusters > 0)
                workers = clusters;
            cudaGetLastError();
        }
        ki.max_workers = workers > 0 ? workers : 1;
        ki.ready = true;
    }
    *out = ki;
    return PGT_OK;
}

// Packed-scale workspace geometry: k groups of four 128-wide K blocks, 128-row blocks of
// A and B rounded up to even counts (pairs of CTAs).  When the tile width `bn` is not a
// multiple of 128, B's blocks are cut per tile instead: ceil(bn / 128) blocks per tile of
// bn rows, so every tile's scales start on a block.
struct SfGeometry {
    int kb, kgroups, ma, nb;
    int tile_n, nbt;  // B rows per tile and 128-row blocks per tile (128 and 1: plain blocks)
    size_t bytes_a, bytes_b;
};

SfGeometry sf_geometry(int64_t M, int64_t N, int64_t K, int bn) {
    SfGeometry g;
    g.kb = (int)(K / 128);
    g.kgroups = (g.kb + 3) / 4;
    g.ma = (int)((cdiv64(M, 128) + 1) / 2 * 2);
    if (bn % 128 == 0) {
        g.tile_n = 128;
        g.nbt = 1;
        g.nb = (int)((cdiv64(N, 128) + 1) / 2 * 2);
    } else {
        g.tile_n = bn;
        g.nbt = (bn + 127) / 128;
        g.nb = (int)(cdiv64(N, bn) * g.nbt);
    }
    g.bytes_a = (size_t)g.kgroups * g.ma * 512;
    g.bytes_b = (size_t)g.kgroups * g.nb * 512;
    return g;
}

// ------------------------------------------------------------- automatic configuration
// PGT_CFG_AUTO picks, per problem, the configuration with the least predicted launch time
//     t = a + W * (b + r * K + s * MB)  (microseconds)
// where W = ceil(T / P) is the number of waves of tiles (T tiles on P resident workers), K
// the reduction length, and MB the operand bytes one CTA loads per tile (its 128 rows of A
// and its rows or columns of B over K, in millions), counted twice for an operand whose row
// pitch is not a multiple of 128 bytes (every TMA box row then straddles two L2 lines).
// a is the launch and pipeline fill/drain cost, b the per-tile switch, r and s the
// mainloop.  The coefficients are fitted to launches of each configuration timed on a GB300
// (bf16: 18 shapes, square 256 .. 8192, the ragged set, skinny M or N, short and long K; the
// fit then picked the fastest configuration on 27 further shapes; MXFP8: 18 shapes),
// weighting relative error.  Candidates: bf16 1-CTA 128x128, 1-CTA 128x256 and pair
// 256x256 (the pair 256x128 is never more than a percent faster than 1-CTA 128x128, and
// usually slower); MXFP8 the same three (the 256x224 tile repacks B's scales per tile, so it
// would change the workspace size, and it is slower wherever measured).
struct CostModel {
    int cfg;
    double a, b, r, s;
};
constexpr CostModel kBf16Cost[] = {
    {PGT_CFG_1CTA_128x128, 4.4861, 0.204532, 0.00281482, 3.14444},
    {PGT_CFG_1CTA_128x256, 4.96696, 0.562448, 0.00141099, 5.56054},
    {PGT_CFG_2CTA_256x256, 6.78523, 1.13483, 0.00126101, 7.12013},
};
// MXFP8 rows are K bytes with K a multiple of 128, so the operand bytes are proportional to
// K and fold into r (s = 0); times include the per-call scale repack.
constexpr CostModel kMxCost[] = {
    {PGT_CFG_1CTA_128x128, 5.98816, 0.328656, 0.00265461, 0.0},
    {PGT_CFG_1CTA_128x256, 5.88766, 0.390631, 0.00332382, 0.0},
    {PGT_CFG_2CTA_256x256, 6.66304, 1.33953, 0.00307062, 0.0},
};

// The configuration a workspace is sized for: AUTO only ever picks tiles whose widths are
// multiples of 128, and those share one packed-scale layout.
int workspace_cfg(int cfg) { return cfg == PGT_CFG_AUTO ? PGT_CFG_2CTA_256x256 : cfg; }

// Resolve PGT_CFG_AUTO for `d` (leading dimensions already defaulted) on the context's device.
int resolve_cfg(const pgt_ctx* ctx, const pgt_gemm_desc& d, int* out) {
    if (d.kernel_cfg != PGT_CFG_AUTO) {
        *out = d.kernel_cfg;
        return PGT_OK;
    }
    const bool mx = d.dtype == PGT_MXFP8;
    const int64_t es = mx ? 1 : 2;
    const bool mis_a = (d.lda * es) % 128 != 0;
    const bool mis_b = (d.ldb * es) % 128 != 0;
    const CostModel* table = mx ? kMxCost : kBf16Cost;
    const int n_cand = mx ? (int)(sizeof(kMxCost) / sizeof(kMxCost[0])) : (int)(sizeof(kBf16Cost) / sizeof(kBf16Cost[0]));
    double best_t = 0.0;
    int best = -1;
    for (int i = 0; i < n_cand; ++i) {
        const CostModel& cm = table[i];
        CfgShape s;
        if (!cfg_shape(cm.cfg, d.dtype, &s)) continue;
        KernelInfo ki;
        const int rc = kernel_info(ctx->device, cm.cfg, mx, d.b_layout == PGT_B_KN, false, s, &ki);
        if (rc) return rc;
        const int64_t tiles = cdiv64(cdiv64(d.M, 128), s.cs) * cdiv64(d.N, s.bn);
        const int64_t workers = ki.max_workers < tiles ? ki.max_workers : tiles;
        const double waves = (double)cdiv64(tiles, workers > 0 ? workers : 1);
        const double mb = ((double)128 * d.K * es * (mis_a ? 2 : 1) + (double)(s.bn / s.cs) * d.K * es * (mis_b ? 2 : 1)) *
                          1e-6;
        const double t = cm.a + waves * (cm.b + cm.r * (double)d.K + cm.s * mb);
        if (best < 0 || t < best_t) {
            best_t = t;
            best = cm.cfg;
        }
    }
    if (best < 0) return PGT_ERR_UNSUPPORTED;
    *out = best;
    return PGT_OK;
}

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
    if (d.dtype != PGT_MXFP8 || d.M < 1 || d.N < 1 || d.K < 128 || d.K % 128) return 0;
    CfgShape s;
    if (!cfg_shape(workspace_cfg(d.kernel_cfg), d.dtype, &s)) return 0;
    const SfGeometry g = sf_geometry(d.M, d.N, d.K, s.bn);
    return g.bytes_a + g.bytes_b;
}

int gemm_plan(const pgt_ctx* ctx, const pgt_gemm_desc* in, pgt_gemm_desc* d, pgt_gemm_plan_info* p) {
    if (ctx == nullptr || in == nullptr || p == nullptr || d == nullptr) return PGT_ERR_ARG;
    *d = *in;
    const int64_t lim = (int64_t)1 << 31;
    if (d->M < 1 || d->N < 1 || d->K < 1 || d->M >= lim || d->N >= lim || d->K >= lim) return PGT_ERR_ARG;
    if (d->dtype != PGT_BF16 && d->dtype != PGT_MXFP8) return PGT_ERR_ARG;
    if (d->b_layout != PGT_B_KN && d->b_layout != PGT_B_NK) return PGT_ERR_ARG;
    if (d->sched_mode < PGT_BLOCKED || d->sched_mode > PGT_LAUNCH_CONTROL) return PGT_ERR_ARG;
    if (d->group_size < 1) return PGT_ERR_ARG;
    if (d->num_workers < 0) return PGT_ERR_ARG;
    if (d->ws_groups == 0) d->ws_groups = ctx->max_groups < 8 ? ctx->max_groups : 8;
    if (d->ws_groups < 1 || d->ws_groups > ctx->max_groups) return PGT_ERR_GROUPS;
    if (d->ws_layout != PGT_WS_RANGES && d->ws_layout != PGT_WS_STRIPED) return PGT_ERR_ARG;
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
    int cfg = 0;
    int rc0 = resolve_cfg(ctx, *d, &cfg);
    if (rc0) return rc0;
    d->kernel_cfg = cfg;
    CfgShape s;
    if (!cfg_shape(d->kernel_cfg, d->dtype, &s)) return PGT_ERR_UNSUPPORTED;
    const int64_t m_blocks = cdiv64(d->M, 128);
    const int64_t n_blocks = cdiv64(d->N, s.bn);
    const int64_t m_tiles = cdiv64(m_blocks, s.cs);
    const int64_t tiles = m_tiles * n_blocks;
    if (tiles >= lim) return PGT_ERR_ARG;
    int64_t workers = d->num_workers;
    if (d->sched_mode == PGT_LAUNCH_CONTROL) {
        // one worker (CTA or pair) per tile; the hardware cancels the ones not yet started
        if (workers != 0 && workers != tiles) return PGT_ERR_ARG;
        workers = tiles;
    } else if (workers == 0) {
        KernelInfo ki;
        int rc = kernel_info(ctx->device, d->kernel_cfg, d->dtype == PGT_MXFP8, d->b_layout == PGT_B_KN, false, s,
                             &ki);
        if (rc) return rc;
        workers = ki.max_workers;
        if (workers > tiles) workers = tiles;
        if (workers < 1) workers = 1;
    }
    if (workers * s.cs >= lim) return PGT_ERR_ARG;
    if (d->sched_mode == PGT_WORK_STEALING && workers > kMaxWsWorkers) return PGT_ERR_ARG;
    // every counter group gets a home worker (a group without one would only be stolen from)
    if (d->ws_groups > workers) d->ws_groups = (int32_t)workers;
    p->kernel_cfg = d->kernel_cfg;
    p->bm = 128;
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
    p->ws_groups = d->ws_groups;
    return PGT_OK;
}

int gemm_launch(pgt_ctx* ctx, const pgt_gemm_desc& d, const pgt_gemm_plan_info& plan, const void* A, const void* B,
                const uint8_t* sfa, const uint8_t* sfb, void* C, void* workspace, size_t workspace_bytes,
                const pgt_trace* trace, cudaStream_t stream) {
    const bool mx = d.dtype == PGT_MXFP8;
    if (A == nullptr || B == nullptr || C == nullptr) return PGT_ERR_ARG;
    if (!aligned16(A) || !aligned16(B) || !aligned16(C)) return PGT_ERR_ALIGN;
    if (!mx && (sfa != nullptr || sfb != nullptr)) return PGT_ERR_ARG;
    if (mx && (sfa == nullptr || sfb == nullptr)) return PGT_ERR_ARG;
    const size_t ws_need = gemm_workspace_bytes(d);
    if (ws_need > 0 && (workspace == nullptr || workspace_bytes < ws_need || !aligned16(workspace)))
        return PGT_ERR_WORKSPACE;
    if (trace != nullptr) {
        if (trace->visits == nullptr || trace->counts == nullptr || trace->max_visits < 1) return PGT_ERR_ARG;
    }
    if (d.epilogue & ~(PGT_EPI_ALPHA | PGT_EPI_BIAS)) return PGT_ERR_ARG;
    if ((d.epilogue & PGT_EPI_BIAS) && (d.bias == nullptr || (reinterpret_cast<uintptr_t>(d.bias) & 3u)))
        return PGT_ERR_ARG;
    CfgShape s;
    if (!cfg_shape(plan.kernel_cfg, d.dtype, &s)) return PGT_ERR_UNSUPPORTED;
    const bool bmn = d.b_layout == PGT_B_KN;
    const bool tr = trace != nullptr;
    KernelInfo ki;
    int rc = kernel_info(ctx->device, plan.kernel_cfg, mx, bmn, tr, s, &ki);
    if (rc) return rc;

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
    gp.sp.ws_layout = d.ws_layout;
    gp.sp.workers = plan.workers;
    gp.sp.counters = ctx->d_counters;
    gp.sp.done = ctx->d_done;
    gp.sp.release = ctx->release_armed ? ctx->d_release : nullptr;  // no reads until release is used
    gp.err = ctx->d_err;
    gp.sfa_rows = 0;
    gp.sfb_rows = 0;
    gp.epi = d.epilogue != 0;
    gp.alpha = (d.epilogue & PGT_EPI_ALPHA) ? d.alpha : 1.0f;
    gp.bias = (d.epilogue & PGT_EPI_BIAS) ? d.bias : nullptr;
    gp.C = static_cast<uint16_t*>(C);
    gp.ldc = d.ldc;
    // K-direction period: the workers this configuration keeps resident at once (capped at
    // T), whatever the scheduler or the requested worker count, so every scheduler gives a
    // tile the same K order.  bf16 only: MXFP8 loads its scales in forward groups of four K
    // blocks, and walking K backwards measured 4-8% slower for it.
    gp.kdir_period = 0;
    if (!mx) {
        KernelInfo k0;
        rc = kernel_info(ctx->device, plan.kernel_cfg, mx, bmn, false, s, &k0);
        if (rc) return rc;
        gp.kdir_period = k0.max_workers < plan.tiles ? k0.max_workers : plan.tiles;
    }
    gp.tr_visits = trace ? trace->visits : nullptr;
    gp.tr_max = trace ? trace->max_visits : 0;
    gp.tr_counts = trace ? trace->counts : nullptr;
    gp.tr_times = trace ? trace->times_ns : nullptr;

    if (d.sched_mode == PGT_WORK_STEALING && (ctx->flags & PGT_FLAG_HOST_RESET)) {
        if (cudaMemsetAsync(ctx->d_counters, 0, sizeof(int) * kCounterStride * (ctx->max_groups + 1), stream) !=
            cudaSuccess)
            return PGT_ERR_CUDA;
    }

    const CUtensorMapDataType op_type = mx ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const int64_t es = mx ? 1 : 2;
    const uint32_t bk = (uint32_t)s.bk;
    const uint32_t bn_cta = (uint32_t)(s.bn / s.cs);
    CUtensorMap ta, tb, tc, tsa, tsb;
    rc = encode_tmap_2d(&ta, op_type, A, d.K, d.M, d.lda * es, bk, 128, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
    if (bmn)
        rc = encode_tmap_2d(&tb, op_type, B, d.N, d.K, d.ldb * es, 64, bk, CU_TENSOR_MAP_SWIZZLE_128B);
    else
        rc = encode_tmap_2d(&tb, op_type, B, d.K, d.N, d.ldb * es, bk, bn_cta, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
    rc = encode_tmap_2d(&tc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, C, d.N, d.M, d.ldc * 2, 64, 32,
                        CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
    tsa = ta;
    tsb = ta;
    if (mx) {
        const SfGeometry sg = sf_geometry(d.M, d.N, d.K, s.bn);
        uint32_t* wa = static_cast<uint32_t*>(workspace);
        uint32_t* wb = wa + sg.bytes_a / 4;
        const int64_t words = (int64_t)(sg.bytes_a + sg.bytes_b) / 4;
        int blocks = (int)((words + 255) / 256);
        if (blocks > 4 * ctx->num_sms) blocks = 4 * ctx->num_sms;
        sf_repack_kernel<<<blocks, 256, 0, stream>>>(sfa, sfb, (int)d.M, (int)d.N, sg.kb, sg.kgroups, sg.ma, sg.nb,
                                                     sg.tile_n, sg.nbt, wa, wb);
        if (cudaGetLastError() != cudaSuccess) return PGT_ERR_CUDA;
        rc = encode_tmap_2d(&tsa, CU_TENSOR_MAP_DATA_TYPE_UINT32, wa, 128, (uint64_t)sg.kgroups * sg.ma, 512, 128, 1,
                            CU_TENSOR_MAP_SWIZZLE_NONE);
        if (rc) return rc;
        rc = encode_tmap_2d(&tsb, CU_TENSOR_MAP_DATA_TYPE_UINT32, wb, 128, (uint64_t)sg.kgroups * sg.nb, 512, 128,
                            (uint32_t)((s.bn + 127) / 128), CU_TENSOR_MAP_SWIZZLE_NONE);
        if (rc) return rc;
        gp.sfa_rows = sg.ma;
        gp.sfb_rows = sg.nb;
    }

    KernelFn k = pick_kernel(plan.kernel_cfg, mx, bmn, tr);
    if (k == nullptr) return PGT_ERR_UNSUPPORTED;
    cudaLaunchConfig_t lc = {};
    cudaLaunchAttribute at[1];
    lc.gridDim = dim3(plan.ctas, 1, 1);
    lc.blockDim = dim3(kThreads, 1, 1);
    lc.dynamicSmemBytes = s.smem;
    lc.stream = stream;
    if (s.cs > 1) {
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = s.cs;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        lc.attrs = at;
        lc.numAttrs = 1;
    }
    if (cudaLaunchKernelEx(&lc, k, ta, tb, tc, tsa, tsb, gp) != cudaSuccess) {
        cudaGetLastError();
        return PGT_ERR_CUDA;
    }
    return PGT_OK;
}

}  // namespace pgt
