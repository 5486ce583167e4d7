// Persistent elementwise add out = x + y (fp32) for sm_103a.
//
// Source: "Implement persistent kernels" (helion PR #238), the _simple_add_kernel listings:
// a grid of SM-count programs loops over 2-D tiles (32 x 16 there) in persistent_blocked
// or persistent_interleaved order, decodes each virtual program id with tile rows varying
// fastest, and does a masked load / add / store.  Here a worker is one CTA; the grid holds
// every CTA that fits on the GPU at once.  Each tile is streamed with 128-bit loads and
// stores (cache-streaming hints, data is touched once) when the rows allow it; ragged
// tile edges fall back to scalar accesses.  The add is __fadd_rn: IEEE binary32, round to
// nearest even, subnormals kept (the library is built without flush-to-zero).
#include <mutex>

#include "pgt_device.cuh"
#include "pgt_internal.h"
#include "pgt_sched.cuh"

namespace pgt {

struct AddParams {
    const float* x;
    const float* y;
    float* out;
    int64_t rows, cols, ldx, ldy, ldo;
    int tile_r, tile_c;
    SchedParams sp;
    int32_t* tr_visits;
    int64_t tr_max;
    int32_t* tr_counts;
    int64_t* tr_times;
};

constexpr int kAddUnroll = 4;

// VEC: pointers 16-byte aligned, leading dimensions and tile_c multiples of 4.
template <bool VEC>
__global__ void __launch_bounds__(256) add_kernel(const AddParams p) {
    const int tid = threadIdx.x;
    const int T = blockDim.x;
    Scheduler sch;
    sch.init(p.sp, blockIdx.x);
    if (p.tr_times != nullptr && tid == 0) p.tr_times[2 * blockIdx.x] = (int64_t)globaltimer();
    int nvis = 0;
    for (;;) {
        const int t = sch.fetch();
        if (t < 0) break;
        int m, n;
        decode_tile(p.sp, t, m, n);
        if (p.tr_visits != nullptr && tid == 0) {
            if (nvis < p.tr_max) {
                int32_t* r = p.tr_visits + ((int64_t)blockIdx.x * p.tr_max + nvis) * PGT_VISIT_FIELDS;
                r[0] = t;
                r[1] = m;
                r[2] = n;
                r[3] = (int32_t)smid();
            }
        }
        ++nvis;
        const int64_t r0 = (int64_t)m * p.tile_r;
        const int64_t c0 = (int64_t)n * p.tile_c;
        const int rh = (int)min((int64_t)p.tile_r, p.rows - r0);
        const int ch = (int)min((int64_t)p.tile_c, p.cols - c0);
        if constexpr (VEC) {
            const int u = (ch + 3) >> 2;  // 4-wide units per row (last may be partial)
            const int total = rh * u;
            for (int i0 = tid; i0 < total; i0 += T * kAddUnroll) {
                float4 a[kAddUnroll], b[kAddUnroll];
                int64_t off[kAddUnroll];
                bool full[kAddUnroll];
#pragma unroll
                for (int j = 0; j < kAddUnroll; ++j) {
                    const int i = i0 + j * T;
                    full[j] = false;
                    off[j] = -1;
                    if (i < total) {
                        const int rr = i / u;
                        const int cc = (i - rr * u) << 2;
                        off[j] = ((int64_t)rr << 32) | (uint32_t)cc;  // row, column inside the tile
                        full[j] = cc + 4 <= ch;
                        if (full[j]) {
                            const int64_t row = r0 + rr, col = c0 + cc;
                            a[j] = __ldcs(reinterpret_cast<const float4*>(p.x + row * p.ldx + col));
                            b[j] = __ldcs(reinterpret_cast<const float4*>(p.y + row * p.ldy + col));
                        }
                    }
                }
#pragma unroll
                for (int j = 0; j < kAddUnroll; ++j) {
                    if (off[j] < 0) continue;
                    const int64_t row = r0 + (off[j] >> 32);
                    const int64_t col = c0 + (int64_t)(uint32_t)(off[j] & 0xFFFFFFFF);
                    if (full[j]) {
                        float4 o;
                        o.x = __fadd_rn(a[j].x, b[j].x);
                        o.y = __fadd_rn(a[j].y, b[j].y);
                        o.z = __fadd_rn(a[j].z, b[j].z);
                        o.w = __fadd_rn(a[j].w, b[j].w);
                        __stcs(reinterpret_cast<float4*>(p.out + row * p.ldo + col), o);
                    } else {
                        for (int64_t c = col; c < c0 + ch; ++c)
                            p.out[row * p.ldo + c] = __fadd_rn(p.x[row * p.ldx + c], p.y[row * p.ldy + c]);
                    }
                }
            }
        } else {
            const int total = rh * ch;
            for (int i = tid; i < total; i += T) {
                const int rr = i / ch;
                const int cc = i - rr * ch;
                const int64_t row = r0 + rr, col = c0 + cc;
                p.out[row * p.ldo + col] = __fadd_rn(p.x[row * p.ldx + col], p.y[row * p.ldy + col]);
            }
        }
    }
    if (tid == 0) {
        if (p.tr_counts != nullptr) p.tr_counts[blockIdx.x] = nvis;
        if (p.tr_times != nullptr) p.tr_times[2 * blockIdx.x + 1] = (int64_t)globaltimer();
    }
}

namespace {

constexpr int kWideTileR = 8, kWideTileC = 1024;

int add_threads(int tile_r, int tile_c) {
    const int64_t units = (int64_t)tile_r * ((tile_c + 3) / 4);
    int64_t t = (units + 31) / 32 * 32;
    if (t > 256) t = 256;
    if (t < 32) t = 32;
    return (int)t;
}

int resolve_tile(int* tile_r, int* tile_c) {
    if (*tile_r == 0 && *tile_c == 0) {
        *tile_r = kWideTileR;
        *tile_c = kWideTileC;
    }
    if (*tile_r < 1 || *tile_r > 1024 || *tile_c < 1 || *tile_c > 4096) return PGT_ERR_ARG;
    if ((int64_t)*tile_r * *tile_c > 65536) return PGT_ERR_ARG;
    return PGT_OK;
}

}  // namespace

int add_workers(const pgt_ctx* ctx, int64_t rows, int64_t cols, int tile_r, int tile_c, int num_workers) {
    if (ctx == nullptr || rows < 1 || cols < 1 || num_workers < 0) return PGT_ERR_ARG;
    int rc = resolve_tile(&tile_r, &tile_c);
    if (rc) return rc;
    const int64_t m_tiles = (rows + tile_r - 1) / tile_r;
    const int64_t n_tiles = (cols + tile_c - 1) / tile_c;
    const int64_t tiles = m_tiles * n_tiles;
    if (tiles >= ((int64_t)1 << 31)) return PGT_ERR_ARG;
    if (num_workers > 0) return num_workers;
    // resident CTAs per SM for this block size, cached per device
    static std::mutex mu;
    static int cache[64][8];  // [device][threads / 32 - 1], 0 = not queried yet
    const int T = add_threads(tile_r, tile_c);  // a multiple of 32 in [32, 256]
    const int slot = T / 32 - 1;
    if (ctx->device < 0 || ctx->device >= 64) return PGT_ERR_ARG;
    int per_sm = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        per_sm = cache[ctx->device][slot];
        if (per_sm == 0) {
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, add_kernel<true>, T, 0) != cudaSuccess)
                return PGT_ERR_CUDA;
            if (per_sm < 1) per_sm = 1;
            cache[ctx->device][slot] = per_sm;
        }
    }
    int64_t w = (int64_t)per_sm * ctx->num_sms;
    if (w > tiles) w = tiles;
    return (int)w;
}

int add_launch(pgt_ctx* ctx, const float* x, const float* y, float* out, int64_t rows, int64_t cols, int64_t ldx,
               int64_t ldy, int64_t ldo, int sched_mode, int tile_r, int tile_c, int num_workers,
               const pgt_trace* trace, cudaStream_t stream) {
    if (ctx == nullptr || x == nullptr || y == nullptr || out == nullptr) return PGT_ERR_ARG;
    if (rows < 1 || cols < 1 || rows >= ((int64_t)1 << 40) || cols >= ((int64_t)1 << 31)) return PGT_ERR_ARG;
    if (sched_mode != PGT_BLOCKED && sched_mode != PGT_INTERLEAVED) return PGT_ERR_ARG;
    if (ldx == 0) ldx = cols;
    if (ldy == 0) ldy = cols;
    if (ldo == 0) ldo = cols;
    if (ldx < cols || ldy < cols || ldo < cols) return PGT_ERR_ARG;
    int rc = resolve_tile(&tile_r, &tile_c);
    if (rc) return rc;
    if (trace != nullptr && (trace->visits == nullptr || trace->counts == nullptr || trace->max_visits < 1))
        return PGT_ERR_ARG;
    const int workers = add_workers(ctx, rows, cols, tile_r, tile_c, num_workers);
    if (workers < 0) return workers;
    AddParams p;
    p.x = x;
    p.y = y;
    p.out = out;
    p.rows = rows;
    p.cols = cols;
    p.ldx = ldx;
    p.ldy = ldy;
    p.ldo = ldo;
    p.tile_r = tile_r;
    p.tile_c = tile_c;
    p.sp.m_tiles = (int)((rows + tile_r - 1) / tile_r);
    p.sp.n_tiles = (int)((cols + tile_c - 1) / tile_c);
    p.sp.tiles = p.sp.m_tiles * p.sp.n_tiles;
    p.sp.mode = sched_mode;
    p.sp.group = 1;
    p.sp.ws_groups = 1;
    p.sp.ws_layout = 0;
    p.sp.workers = workers;
    p.sp.counters = nullptr;
    p.sp.done = nullptr;
    p.sp.release = nullptr;
    p.tr_visits = trace ? trace->visits : nullptr;
    p.tr_max = trace ? trace->max_visits : 0;
    p.tr_counts = trace ? trace->counts : nullptr;
    p.tr_times = trace ? trace->times_ns : nullptr;
    const bool vec = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y) |
                       reinterpret_cast<uintptr_t>(out)) & 15u) == 0 &&
                     ldx % 4 == 0 && ldy % 4 == 0 && ldo % 4 == 0 && tile_c % 4 == 0;
    const int T = add_threads(tile_r, tile_c);
    if (vec)
        add_kernel<true><<<workers, T, 0, stream>>>(p);
    else
        add_kernel<false><<<workers, T, 0, stream>>>(p);
    return cuda_status(cudaGetLastError());
}

}  // namespace pgt
