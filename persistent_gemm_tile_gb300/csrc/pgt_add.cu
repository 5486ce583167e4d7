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
    int batch;  // tiles of the worker's order streamed together (1 .. kAddMaxBatch)
    SchedParams sp;
    int32_t* tr_visits;
    int64_t tr_max;
    int32_t* tr_counts;
    int64_t* tr_times;
};

constexpr int kAddUnroll = 4;    // units (float4, or one float) in flight per thread
constexpr int kAddMaxBatch = 8;  // most tiles streamed together

// A worker takes the next `batch` tiles of its scheduler order at a time and treats their
// units as one index space: thread i of the CTA moves units i, i + T, ..., kAddUnroll of them
// per step, all loads issued before the adds and stores.  The grid holds at most the CTAs
// that fit on the GPU at once; when there are more workers than CTAs, CTA b runs workers b,
// b + grid, b + 2 grid, ... one after the other.  A unit is 4 consecutive floats of a
// tile row (VEC: pointers 16-byte aligned, leading dimensions and tile_c multiples of 4) or
// one float.  Small tiles (the page's 32 x 16 holds 128 float4 units) thus keep several
// tiles' loads in flight per thread; a wide tile is one batch of its own.  Ragged edge tiles
// mask the units past their rows and columns.
// 72 registers: seven 128-thread CTAs (the page's 32 x 16 tile) or three 256-thread CTAs fit
// on an SM, with nothing spilled.
template <bool VEC>
__global__ void __maxnreg__(72) add_kernel(const AddParams p) {
    const int tid = threadIdx.x;
    const int T = blockDim.x;
    const int upr = VEC ? (p.tile_c + 3) >> 2 : p.tile_c;  // units per tile row
    const int U = p.tile_r * upr;                         // units per tile
    for (int w = blockIdx.x; w < p.sp.workers; w += gridDim.x) {
    Scheduler sch;
    sch.init(p.sp, w);
    if (p.tr_times != nullptr && tid == 0) p.tr_times[2 * w] = (int64_t)globaltimer();
    int nvis = 0;
    for (;;) {
        int first, step;
        const int cnt = sch.fetch_run(p.batch, first, step);
        if (cnt == 0) break;
        if (p.tr_visits != nullptr && tid == 0) {
            for (int b = 0; b < cnt; ++b, ++nvis) {
                if (nvis >= p.tr_max) continue;
                const int t = first + b * step;
                int m, n;
                decode_tile(p.sp, t, m, n);
                int32_t* r = p.tr_visits + ((int64_t)w * p.tr_max + nvis) * PGT_VISIT_FIELDS;
                r[0] = t;
                r[1] = m;
                r[2] = n;
                r[3] = (int32_t)smid();
            }
        } else {
            nvis += cnt;
        }
        const int total = cnt * U;
        for (int i0 = tid; i0 < total; i0 += T * kAddUnroll) {
            // where each of this thread's units lies: its row and first column (row -1: no
            // unit), and the columns left in its tile row from there
            int64_t row[kAddUnroll];
            int col[kAddUnroll], left[kAddUnroll];
#pragma unroll
            for (int j = 0; j < kAddUnroll; ++j) {
                const int g = i0 + j * T;
                left[j] = 0;
                row[j] = -1;
                col[j] = 0;
                if (g < total) {
                    const int b = g / U;
                    const int l = g - b * U;
                    const int rr = l / upr;
                    const int cc = (l - rr * upr) * (VEC ? 4 : 1);
                    int m, n;
                    decode_tile(p.sp, first + b * step, m, n);
                    const int64_t r = (int64_t)m * p.tile_r + rr;
                    const int64_t c = (int64_t)n * p.tile_c + cc;
                    const int64_t c_end = min((int64_t)(n + 1) * p.tile_c, p.cols);
                    if (r < p.rows && c < c_end) {
                        row[j] = r;
                        col[j] = (int)c;
                        left[j] = (int)(c_end - c);
                    }
                }
            }
            if constexpr (VEC) {
                float4 a[kAddUnroll], c[kAddUnroll];
#pragma unroll
                for (int j = 0; j < kAddUnroll; ++j) {
                    if (left[j] >= 4) {
                        a[j] = __ldcs(reinterpret_cast<const float4*>(p.x + row[j] * p.ldx + col[j]));
                        c[j] = __ldcs(reinterpret_cast<const float4*>(p.y + row[j] * p.ldy + col[j]));
                    }
                }
#pragma unroll
                for (int j = 0; j < kAddUnroll; ++j) {
                    float* o = p.out + row[j] * p.ldo + col[j];
                    if (left[j] >= 4) {
                        float4 v;
                        v.x = __fadd_rn(a[j].x, c[j].x);
                        v.y = __fadd_rn(a[j].y, c[j].y);
                        v.z = __fadd_rn(a[j].z, c[j].z);
                        v.w = __fadd_rn(a[j].w, c[j].w);
                        __stcs(reinterpret_cast<float4*>(o), v);
                    } else {
                        // the last 1-3 columns of a ragged row
                        const float* xs = p.x + row[j] * p.ldx + col[j];
                        const float* ys = p.y + row[j] * p.ldy + col[j];
                        for (int e = 0; e < left[j]; ++e) o[e] = __fadd_rn(xs[e], ys[e]);
                    }
                }
            } else {
                float a[kAddUnroll], c[kAddUnroll];
#pragma unroll
                for (int j = 0; j < kAddUnroll; ++j) {
                    if (left[j] > 0) {
                        a[j] = p.x[row[j] * p.ldx + col[j]];
                        c[j] = p.y[row[j] * p.ldy + col[j]];
                    }
                }
#pragma unroll
                for (int j = 0; j < kAddUnroll; ++j)
                    if (left[j] > 0) p.out[row[j] * p.ldo + col[j]] = __fadd_rn(a[j], c[j]);
            }
        }
    }
    if (tid == 0) {
        if (p.tr_counts != nullptr) p.tr_counts[w] = nvis;
        if (p.tr_times != nullptr) p.tr_times[2 * w + 1] = (int64_t)globaltimer();
    }
    }
}

namespace {

constexpr int kWideTileR = 8, kWideTileC = 1024;

// Threads per CTA: enough for two rounds of kAddUnroll float4 units per thread over a full
// batch of tiles, a multiple of 32 in [32, 256] (the page's 32 x 16 tile: 128, so more
// CTAs, i.e. workers, fit on an SM).
int add_threads(int tile_r, int tile_c) {
    const int64_t units = (int64_t)tile_r * ((tile_c + 3) / 4);
    int64_t t = (units * kAddMaxBatch / (2 * kAddUnroll) + 31) / 32 * 32;
    if (t > 256) t = 256;
    if (t < 32) t = 32;
    return (int)t;
}

// Tiles per batch: as many as fill every thread's kAddUnroll slots once, 1 .. kAddMaxBatch.
// In the blocked order a worker's tiles are consecutive rows of one tile column, and twice
// that (two rounds per batch) measured faster; in the interleaved order a batch spans tiles
// P apart, and longer batches measured slower.
int add_batch(int tile_r, int tile_c, bool vec, int threads, int sched_mode) {
    const int64_t units = (int64_t)tile_r * (vec ? (tile_c + 3) / 4 : tile_c);
    int64_t b = (int64_t)threads * kAddUnroll / units * (sched_mode == PGT_BLOCKED ? 2 : 1);
    if (b > kAddMaxBatch) b = kAddMaxBatch;
    if (b < 1) b = 1;
    return (int)b;
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

// Default worker count.  Every CTA that fits on the GPU at once, except for tiles narrower
// than a 128-byte line: with rows varying fastest, a worker walks down a column of tiles,
// and the rest of each line it reads belongs to the next tile column(s).  The L2 fetches
// whole lines, so unless the worker on the neighbouring column reads the same rows at about
// the same time, every line is fetched from DRAM once per tile column (twice for the page's
// 16-float tiles, measured).  Worker counts that keep line partners in flight together:
//   blocked:     P = n_tiles * j with j dividing m_tiles (each worker covers an equal part
//                of one tile column, all workers at the same rows of their columns), the
//                largest that fits on the GPU at once;
//   interleaved: P a multiple of m_tiles * (tile columns per line) (each wave of P tiles
//                covers whole groups of line-sharing columns), the largest up to twice what
//                fits, each CTA then running two workers in turn (measured faster than one
//                resident wave: 0.83 against 0.75 of HBM at 8192 x 8192).
// Returns 0 when no such count applies.
int64_t line_friendly_workers(int sched_mode, int64_t m_tiles, int64_t n_tiles, int tile_c, int64_t cap) {
    const int tile_bytes = 4 * tile_c;
    if (tile_bytes >= 128 || 128 % tile_bytes != 0) return 0;
    const int64_t per_line = 128 / tile_bytes;
    if (sched_mode == PGT_BLOCKED) {
        for (int64_t j = cap / n_tiles; j >= 1; --j)
            if (m_tiles % j == 0) return n_tiles * j;
        return 0;
    }
    const int64_t q = m_tiles * per_line;
    return q <= 2 * cap ? 2 * cap / q * q : 0;
}

// CTAs of the add kernel with T threads that fit on the context's GPU at once (cached).
int add_capacity(const pgt_ctx* ctx, int T, int64_t* cap) {
    static std::mutex mu;
    static int cache[64][8];  // [device][threads / 32 - 1], 0 = not queried yet
    const int slot = T / 32 - 1;
    if (ctx->device < 0 || ctx->device >= 64 || slot < 0 || slot >= 8) return PGT_ERR_ARG;
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
    *cap = (int64_t)per_sm * ctx->num_sms;
    return PGT_OK;
}

int add_workers(const pgt_ctx* ctx, int64_t rows, int64_t cols, int tile_r, int tile_c, int sched_mode,
                int num_workers) {
    if (ctx == nullptr || rows < 1 || cols < 1 || num_workers < 0) return PGT_ERR_ARG;
    if (sched_mode != PGT_BLOCKED && sched_mode != PGT_INTERLEAVED) return PGT_ERR_ARG;
    int rc = resolve_tile(&tile_r, &tile_c);
    if (rc) return rc;
    const int64_t m_tiles = (rows + tile_r - 1) / tile_r;
    const int64_t n_tiles = (cols + tile_c - 1) / tile_c;
    const int64_t tiles = m_tiles * n_tiles;
    if (tiles >= ((int64_t)1 << 31)) return PGT_ERR_ARG;
    if (num_workers > 0) return num_workers;
    int64_t cap = 0;
    rc = add_capacity(ctx, add_threads(tile_r, tile_c), &cap);
    if (rc) return rc;
    int64_t w = line_friendly_workers(sched_mode, m_tiles, n_tiles, tile_c, cap);
    if (w == 0) w = cap;
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
    const int workers = add_workers(ctx, rows, cols, tile_r, tile_c, sched_mode, num_workers);
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
    p.batch = add_batch(tile_r, tile_c, vec, T, sched_mode);
    int64_t cap = 0;
    rc = add_capacity(ctx, T, &cap);
    if (rc) return rc;
    const int grid = workers < cap ? workers : (int)cap;  // CTAs host workers in turn beyond that
    if (vec)
        add_kernel<true><<<grid, T, 0, stream>>>(p);
    else
        add_kernel<false><<<grid, T, 0, stream>>>(p);
    return cuda_status(cudaGetLastError());
}

}  // namespace pgt
