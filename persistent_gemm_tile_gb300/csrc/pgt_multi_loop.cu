// Fused persistent loop over several independent elementwise tile spaces: out_s = scale_s * x_s.
//
// Source: "Implement persistent kernels" (helion PR #238), the two multi-loop listings: the
// tile ids of every space are laid end to end (total_pids = sum of the spaces' tile
// counts), one SM-count grid walks them in persistent_blocked or persistent_interleaved
// order, and each id is handled by the first space whose range holds it, decoded with tile
// rows varying fastest inside that space (the listing computes result1 = 2 * x and
// result2 = 3 * y).  One launch keeps every SM busy across both spaces instead of two
// launches each with its own tail.  Each tile streams with 128-bit accesses when its
// space's rows allow it, else with scalar accesses; one IEEE multiply per element.
#include "pgt_device.cuh"
#include "pgt_internal.h"
#include "pgt_sched.cuh"

namespace pgt {

struct SpaceParams {
    const float* x;
    float* out;
    int64_t rows, cols, ldx, ldo;
    float scale;
    int first;    // first global tile id of this space
    int m_tiles;  // tile rows
    int vec;      // 128-bit accesses allowed
};

struct MultiParams {
    SpaceParams sp[PGT_MAX_SPACES];
    int n_spaces;
    int tile_r, tile_c;
    SchedParams sched;
    int32_t* tr_visits;
    int64_t tr_max;
    int32_t* tr_counts;
    int64_t* tr_times;
};

__global__ void __launch_bounds__(256) multi_loop_kernel(const MultiParams p) {
    const int tid = threadIdx.x;
    const int T = blockDim.x;
    Scheduler sch;
    sch.init(p.sched, blockIdx.x);
    if (p.tr_times != nullptr && tid == 0) p.tr_times[2 * blockIdx.x] = (int64_t)globaltimer();
    int nvis = 0;
    for (;;) {
        const int t = sch.fetch();
        if (t < 0) break;
        int s = 0;
        while (s + 1 < p.n_spaces && t >= p.sp[s + 1].first) ++s;
        const SpaceParams& q = p.sp[s];
        const int local = t - q.first;
        const int n = local / q.m_tiles;
        const int m = local - n * q.m_tiles;
        if (p.tr_visits != nullptr && tid == 0 && nvis < p.tr_max) {
            // records: tile id, m, n, and the space in the high byte of the SM id field
            int32_t* r = p.tr_visits + ((int64_t)blockIdx.x * p.tr_max + nvis) * PGT_VISIT_FIELDS;
            r[0] = t;
            r[1] = m;
            r[2] = n;
            r[3] = (int32_t)((uint32_t)s << 24 | smid());
        }
        ++nvis;
        const int64_t r0 = (int64_t)m * p.tile_r;
        const int64_t c0 = (int64_t)n * p.tile_c;
        const int rh = (int)min((int64_t)p.tile_r, q.rows - r0);
        const int ch = (int)min((int64_t)p.tile_c, q.cols - c0);
        if (q.vec) {
            constexpr int kUnroll = 4;  // 128-bit loads in flight per thread before the stores
            const int u = (ch + 3) >> 2;
            const int total = rh * u;
            for (int i0 = tid; i0 < total; i0 += T * kUnroll) {
                float4 a[kUnroll];
                int rr[kUnroll], cc[kUnroll];
#pragma unroll
                for (int j = 0; j < kUnroll; ++j) {
                    const int i = i0 + j * T;
                    rr[j] = -1;
                    if (i < total) {
                        rr[j] = i / u;
                        cc[j] = (i - rr[j] * u) << 2;
                        if (cc[j] + 4 <= ch)
                            a[j] = __ldcs(reinterpret_cast<const float4*>(q.x + (r0 + rr[j]) * q.ldx + c0 + cc[j]));
                    }
                }
#pragma unroll
                for (int j = 0; j < kUnroll; ++j) {
                    if (rr[j] < 0) continue;
                    const int64_t row = r0 + rr[j], col = c0 + cc[j];
                    if (cc[j] + 4 <= ch) {
                        float4 o;
                        o.x = __fmul_rn(q.scale, a[j].x);
                        o.y = __fmul_rn(q.scale, a[j].y);
                        o.z = __fmul_rn(q.scale, a[j].z);
                        o.w = __fmul_rn(q.scale, a[j].w);
                        __stcs(reinterpret_cast<float4*>(q.out + row * q.ldo + col), o);
                    } else {
                        for (int64_t c = col; c < c0 + ch; ++c)
                            q.out[row * q.ldo + c] = __fmul_rn(q.scale, q.x[row * q.ldx + c]);
                    }
                }
            }
        } else {
            const int total = rh * ch;
            for (int i = tid; i < total; i += T) {
                const int rr = i / ch;
                const int cc = i - rr * ch;
                const int64_t row = r0 + rr, col = c0 + cc;
                q.out[row * q.ldo + col] = __fmul_rn(q.scale, q.x[row * q.ldx + col]);
            }
        }
    }
    if (tid == 0) {
        if (p.tr_counts != nullptr) p.tr_counts[blockIdx.x] = nvis;
        if (p.tr_times != nullptr) p.tr_times[2 * blockIdx.x + 1] = (int64_t)globaltimer();
    }
}

}  // namespace pgt

using namespace pgt;

extern "C" int pgt_multi_loop(pgt_ctx* ctx, const pgt_scale_space* spaces, int n_spaces, int sched_mode, int tile_r,
                              int tile_c, int num_workers, const pgt_trace* trace, void* stream) {
    if (ctx == nullptr || spaces == nullptr || n_spaces < 1 || n_spaces > PGT_MAX_SPACES) return PGT_ERR_ARG;
    if (sched_mode != PGT_BLOCKED && sched_mode != PGT_INTERLEAVED) return PGT_ERR_ARG;
    if (tile_r == 0 && tile_c == 0) {
        tile_r = 8;
        tile_c = 1024;
    }
    if (tile_r < 1 || tile_r > 1024 || tile_c < 1 || tile_c > 4096 || (int64_t)tile_r * tile_c > 65536)
        return PGT_ERR_ARG;
    if (num_workers < 0) return PGT_ERR_ARG;
    if (trace != nullptr && (trace->visits == nullptr || trace->counts == nullptr || trace->max_visits < 1))
        return PGT_ERR_ARG;
    MultiParams p;
    int64_t total = 0;
    for (int s = 0; s < n_spaces; ++s) {
        const pgt_scale_space& in = spaces[s];
        SpaceParams& q = p.sp[s];
        if (in.x == nullptr || in.out == nullptr || in.rows < 1 || in.cols < 1) return PGT_ERR_ARG;
        const int64_t ldx = in.ldx ? in.ldx : in.cols, ldo = in.ldo ? in.ldo : in.cols;
        if (ldx < in.cols || ldo < in.cols) return PGT_ERR_ARG;
        const int64_t mt = (in.rows + tile_r - 1) / tile_r, nt = (in.cols + tile_c - 1) / tile_c;
        if (mt >= ((int64_t)1 << 31) || mt * nt >= ((int64_t)1 << 31)) return PGT_ERR_ARG;
        q.x = in.x;
        q.out = in.out;
        q.rows = in.rows;
        q.cols = in.cols;
        q.ldx = ldx;
        q.ldo = ldo;
        q.scale = in.scale;
        q.first = (int)total;
        q.m_tiles = (int)mt;
        q.vec = ((reinterpret_cast<uintptr_t>(in.x) | reinterpret_cast<uintptr_t>(in.out)) & 15u) == 0 &&
                ldx % 4 == 0 && ldo % 4 == 0 && tile_c % 4 == 0;
        total += mt * nt;
        if (total >= ((int64_t)1 << 31)) return PGT_ERR_ARG;
    }
    if (cudaSetDevice(ctx->device) != cudaSuccess) return PGT_ERR_CUDA;
    const int64_t units = (int64_t)tile_r * ((tile_c + 3) / 4);
    int T = (int)((units + 31) / 32 * 32);
    if (T > 256) T = 256;
    if (T < 32) T = 32;
    int workers = num_workers;
    if (workers == 0) {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, multi_loop_kernel, T, 0) != cudaSuccess)
            return PGT_ERR_CUDA;
        int64_t w = (int64_t)(per_sm > 0 ? per_sm : 1) * ctx->num_sms;
        workers = (int)(w < total ? w : total);
    }
    p.n_spaces = n_spaces;
    p.tile_r = tile_r;
    p.tile_c = tile_c;
    p.sched.tiles = (int)total;
    p.sched.m_tiles = 1;
    p.sched.n_tiles = (int)total;
    p.sched.mode = sched_mode;
    p.sched.group = 1;
    p.sched.ws_groups = 1;
    p.sched.ws_layout = 0;
    p.sched.workers = workers;
    p.sched.counters = nullptr;
    p.sched.done = nullptr;
    p.sched.release = nullptr;
    p.tr_visits = trace ? trace->visits : nullptr;
    p.tr_max = trace ? trace->max_visits : 0;
    p.tr_counts = trace ? trace->counts : nullptr;
    p.tr_times = trace ? trace->times_ns : nullptr;
    multi_loop_kernel<<<workers, T, 0, static_cast<cudaStream_t>(stream)>>>(p);
    return cuda_status(cudaGetLastError());
}
