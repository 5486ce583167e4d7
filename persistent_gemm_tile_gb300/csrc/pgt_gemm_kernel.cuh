// Device code of the persistent tiled GEMM (the host side is pgt_gemm.cu).
//
// Persistent tiled GEMM C = A . B for sm_103a: TMA producer warp, tcgen05 MMA warp issuing
// into tensor-memory accumulators, a scheduler thread, four epilogue warps, an mbarrier
// stage ring, and a tile-id ring that carries the scheduler's choices to every role.
//
// Design source: the warp-specialised persistent kernel of "[Feature] Introduce tile
// scheduler" (tilelang PR #2441, gemm_mxfp8_blockscaled_1d1d.py): TMA warp, MMA warp,
// epilogue warpgroup (threads 128..255), loaded/consumed barriers indexed by
// phase = iter * k_iters + k with stage = phase % stages and parity = (phase / stages) & 1,
// tmem_full / tmem_empty between MMA and epilogue, 2-CTA clusters where CTA cta_id of a
// pair owns tile row bx = m_idx * 2 + cta_id and loads half of B's tile, and MXFP8 scales
// (one E8M0 byte per row and 128-wide K block) copied to tensor memory for block-scaled
// MMAs.  Differences: the accumulator is double buffered whenever tensor memory allows, so
// the epilogue of one tile overlaps the next tile's mainloop; a scheduler thread of its own
// publishes each tile ahead through a small shared-memory ring (needed for work stealing,
// where roles cannot recompute the tile, and keeping every decision out of the producer's
// instruction stream); scales are repacked once per call into the tensor-memory copy
// layout, so no transpose warp is needed.
//
// Template parameters: CS = CTAs per worker (1, or 2 for a cluster pair issuing
// cta_group::2 MMAs with M = 256); BN = output columns per worker tile; B_MN = B stored
// K x N (N contiguous) instead of N x K; MX = MXFP8 operands (E4M3 + E8M0 scales) instead
// of bf16; TRACE = record every visit.
#pragma once

#include <cuda_bf16.h>

#include "pgt.h"
#include "pgt_device.cuh"
#include "pgt_sched.cuh"

namespace pgt {

struct GemmParams {
    int M, N, K;
    int k_iters;
    SchedParams sp;
    int* err;
    int sfa_rows;  // MXFP8: rows of 128-row scale blocks per k group in the packed SFA
    int sfb_rows;  // MXFP8: same for SFB
    int epi;       // nonzero: C = alpha * acc + bias[n] before rounding
    float alpha;
    const float* bias;  // fp32[N] or nullptr
    uint16_t* C;        // bf16 output (the last, narrower store chunk of a tile is written directly)
    int64_t ldc;        // elements
    int kdir_period;    // bf16: tiles t with odd t / kdir_period run K backwards (0: all forward)
    int32_t* tr_visits;
    int64_t tr_max;
    int32_t* tr_counts;
    int64_t* tr_times;
};

constexpr int kThreads = 256;           // warp 0 producer, warp 1 MMA, warp 2 scheduler, warps 4-7 epilogue
constexpr int kTileRing = 4;            // tile-id ring depth
constexpr int kEpiWarps = 4;
constexpr int kEpiBufBytes = 32 * 128;  // 32 rows x 64 bf16, 128B-swizzled, per buffer
constexpr int kMaxSmem = 232448;        // 227 KB dynamic shared memory per CTA
constexpr int kTicketLead = 8;          // work stealing: the next tile is asked for this many
                                        // stages before the current tile's last load
constexpr int kSchedPatience = 8;       // bounded waits the scheduler thread may chain for a
                                        // free ring entry while every other role progresses

constexpr int pow2_at_least(int v) {
    int p = 32;
    while (p < v) p *= 2;
    return p;
}

// Shared-memory and tensor-memory layout (offsets from a 1024-aligned base).  Every stage
// holds this CTA's 128 x 128-byte A slice, its BN/CS rows (or columns) of B, and for MXFP8
// a scale area refilled every fourth stage.
template <int CS, int BN, int STAGES, bool MX>
struct Layout {
    static constexpr int BM = 128;                 // rows per CTA
    static constexpr int BK = MX ? 128 : 64;       // K elements per stage (128 bytes per row)
    static constexpr int BN_CTA = BN / CS;         // B rows (or columns) held by one CTA
    static constexpr int A_BYTES = BM * 128;
    static constexpr int B_BYTES = BN_CTA * 128;
    static constexpr int NB128 = (BN + 127) / 128;  // 128-row scale blocks of B per tile
    static constexpr int SF_BYTES = MX ? ((512 + 512 * NB128 + 1023) / 1024 * 1024) : 0;
    static constexpr int SFB_OFF = A_BYTES + B_BYTES + 512;  // SFA at A+B, SFB after it
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SF_BYTES;
    static constexpr int TX_BYTES = A_BYTES + B_BYTES;             // per CTA, every stage
    static constexpr int SF_TX_BYTES = MX ? 512 + 512 * NB128 : 0;  // per CTA, every 4th stage
    // accumulators: double buffered unless tensor memory cannot hold two plus the scales.
    // Accumulator a starts at column a * ACC_STRIDE (BN rounded up to 128).  The scales
    // (two buffers of 4 SFA columns and two of 4 * NB128 SFB columns) follow the last
    // accumulator, or, when the tile leaves a gap of at least 8 columns before the second
    // accumulator, SFA sits in that gap and SFB follows the second accumulator.
    static constexpr int ACC_STRIDE = (BN + 127) / 128 * 128;
    static constexpr int SFA_COLS = MX ? 8 : 0;
    static constexpr int SFB_COLS = MX ? 8 * NB128 : 0;
    static constexpr bool SF_IN_GAP = MX && ACC_STRIDE - BN >= SFA_COLS && ACC_STRIDE + BN + SFB_COLS <= 512;
    static constexpr int ACC_BUFS = (SF_IN_GAP || 2 * ACC_STRIDE + SFA_COLS + SFB_COLS <= 512) ? 2 : 1;
    static constexpr int SFA_COL = SF_IN_GAP ? BN : ACC_BUFS * ACC_STRIDE;
    static constexpr int SFB_COL = SF_IN_GAP ? ACC_STRIDE + BN : SFA_COL + SFA_COLS;
    static constexpr int TMEM_COLS =
        pow2_at_least(SF_IN_GAP ? SFB_COL + SFB_COLS : ACC_BUFS * ACC_STRIDE + SFA_COLS + SFB_COLS);
    static constexpr int EPI_BUFS = (STAGES * STAGE_BYTES + kEpiWarps * 2 * kEpiBufBytes + 2048 <= kMaxSmem) ? 2 : 1;
    static constexpr int EPI_OFF = STAGES * STAGE_BYTES;
    static constexpr int BAR_OFF = EPI_OFF + kEpiWarps * EPI_BUFS * kEpiBufBytes;
    // barriers: full[S], empty[S], tfull[2], tempty[2], sfull[Q], sempty[Q], mma_done, clc,
    // ticket request
    static constexpr int NUM_BARS = 2 * STAGES + 4 + 2 * kTileRing + 3;
    static constexpr int RING_OFF = BAR_OFF + (NUM_BARS * 8 + 15) / 16 * 16;  // int4 entries
    static constexpr int MISC_OFF = RING_OFF + kTileRing * 16;                // tmem slot, abort flag
    static constexpr int CLC_OFF = MISC_OFF + 16;                             // launch-control answer
    static constexpr int BYTES = CLC_OFF + 16;
    static constexpr int SMEM = BYTES + 1024;  // alignment slack
    static_assert(STAGE_BYTES % 1024 == 0 && A_BYTES % 1024 == 0 && (A_BYTES + B_BYTES) % 1024 == 0,
                  "stages must keep 1024-byte swizzle alignment");
    static_assert(EPI_OFF % 1024 == 0 && BAR_OFF % 1024 == 0, "epilogue buffers need 1024-byte alignment");
    static_assert(RING_OFF % 16 == 0 && MISC_OFF % 16 == 0, "ring entries are 16-byte vectors");
    static_assert(SMEM <= kMaxSmem, "dynamic shared memory above the 227 KB per-CTA limit");
    static_assert(TMEM_COLS <= 512, "tensor memory holds 512 columns");
    static_assert(BN_CTA % 8 == 0, "B rows per CTA must fill whole 8-row swizzle atoms");
    static_assert(MX || BN % 64 == 0, "bf16 tiles are whole 64-column store chunks");
};

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo, uint32_t hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(lo), __uint_as_float(hi));
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void st_global_v4(uint16_t* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// TMA load whose completion goes to `bar`: plain form for one CTA, pair form (the barrier
// may be the leader's) for a cluster pair.
template <int CS>
__device__ __forceinline__ void tma_load(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t x, int32_t y) {
    if constexpr (CS == 1)
        tma_load_2d(dst, map, bar, x, y);
    else
        tma_load_2d_pair(dst, map, bar, x, y);
}

// Arrive on a barrier of this CTA, or on the same barrier of the pair's leader.
__device__ __forceinline__ void arrive_local_or_leader(uint32_t local_bar, bool remote) {
    if (remote)
        mbar_arrive_remote(mapa_shared(local_bar, 0));
    else
        mbar_arrive(local_bar);
}

// The same for an arrival that needs no release: the pair's other CTA then arrives relaxed.
__device__ __forceinline__ void arrive_local_or_leader_relaxed(uint32_t local_bar, bool remote) {
    if (remote)
        mbar_arrive_remote_relaxed(mapa_shared(local_bar, 0));
    else
        mbar_arrive(local_bar);
}

template <int CS, int BN, int STAGES, bool B_MN, bool MX, bool TRACE>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmSFA,
                const __grid_constant__ CUtensorMap tmSFB, const GemmParams gp) {
    using L = Layout<CS, BN, STAGES, MX>;
    constexpr bool kPair = CS == 2;
    static_assert(!B_MN || L::BN_CTA % 64 == 0, "B stored K x N is loaded in 64-column boxes");
    static_assert(BN % 64 == 0 || L::ACC_BUFS == 2, "a ragged last store chunk needs the double-buffered epilogue");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);

    const int warp = threadIdx.x >> 5;
    const uint32_t lane = lane_id();
    const uint32_t rank = kPair ? cluster_ctarank() : 0u;  // CTA index inside the pair
    const bool leader = rank == 0;
    const int worker = blockIdx.x / CS;

    // The scheduler runs on a thread of its own in the worker's leader CTA (warp 2, lane 0)
    // and posts each decision into the tile ring ahead of the roles that read it, so no
    // decision (a decode, a counter round trip, the writes into the pair's other CTA) sits
    // in the producer's instruction stream at a tile boundary.  The static orders run up to
    // a ring's depth ahead; work stealing takes each later ticket only when the producer
    // asks for it, a few stages before its current tile's last load.  Launch control stays
    // in the producer, which cancels a cluster once it has taken a tile.  Work stealing
    // starts reading its release flag here, so the read overlaps the set-up.
    const bool ws = gp.sp.mode == kWorkStealing;
    const bool clc = gp.sp.mode == kLaunchControl;
    const bool sched_thread = !clc;  // the ring is written by warp 2 (else by the producer)
    Scheduler sch;
    if (leader && sched_thread && threadIdx.x == 64) sch.init(gp.sp, worker);

    const uint32_t bar0 = base + L::BAR_OFF;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
    auto tempty = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
    auto sfull = [&](int q) { return bar0 + 8u * (2 * STAGES + 4 + q); };
    auto sempty = [&](int q) { return bar0 + 8u * (2 * STAGES + 4 + kTileRing + q); };
    const uint32_t mma_done = bar0 + 8u * (2 * STAGES + 4 + 2 * kTileRing);
    const uint32_t clc_bar = mma_done + 8u;
    const uint32_t tk_req = clc_bar + 8u;  // work stealing: the producer asks for its next tile
    const uint32_t clc_resp = base + L::CLC_OFF;
    int4* ring = reinterpret_cast<int4*>(gbase + L::RING_OFF);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gbase + L::MISC_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + L::MISC_OFF + 4);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full(s), 1);   // the leader's expect_tx; bytes of both CTAs of a pair
            mbar_init(empty(s), 1);  // one MMA commit
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull(a), 1);
            mbar_init(tempty(a), kEpiWarps * CS);
        }
        for (int q = 0; q < kTileRing; ++q) {
            mbar_init(sfull(q), 1);
            // consumers of a ring entry: the MMA thread, the epilogue warps, in a pair also the
            // peer's producer and epilogue warps (all counted on the leader), and this CTA's
            // producer when the scheduler thread writes the ring
            mbar_init(sempty(q), (kPair ? 2 + 2 * kEpiWarps : 1 + kEpiWarps) + (sched_thread ? 1 : 0));
        }
        mbar_init(mma_done, 1);
        mbar_init(clc_bar, 1);
        mbar_init(tk_req, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc<CS>(base + L::MISC_OFF, L::TMEM_COLS);
        tmem_relinquish<CS>();
    }
    tc_fence_before();
    if constexpr (kPair)
        cluster_sync();
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (TRACE && threadIdx.x == 0 && gp.tr_times != nullptr) gp.tr_times[2 * blockIdx.x] = (int64_t)globaltimer();

    // K direction of a tile (bf16): tiles of alternate waves walk K backwards, so a wave starts
    // on the K slices of the panels the previous wave read last, which are still in L2.  A
    // tile's wave is its position in the 16-column-group order (the swizzled order with group
    // 16) divided by kdir_period, the number of workers the GPU holds at once.  It depends on
    // (m, n) alone, so each output tile has one K order whatever the scheduler, group size or
    // worker count.
    auto k_reversed = [&](int m, int n) -> bool {
        if (MX || gp.kdir_period <= 0) return false;
        const int g16 = min(16, gp.sp.n_tiles);
        const int grp = n / g16;
        const int gw = min(g16, gp.sp.n_tiles - grp * g16);
        const int pos = grp * g16 * gp.sp.m_tiles + m * gw + (n - grp * g16);
        return ((pos / gp.kdir_period) & 1) != 0;
    };
    // Post tile t (-1: no more tiles) as ring entry qc for every role of the worker, decoded
    // and with its K direction, in this CTA and, in a pair, in the other CTA as well.  The
    // scheduler thread runs up to a ring's depth ahead of the slowest reader (the epilogue),
    // so its wait for a free entry may span more than a tile: it keeps waiting, one bounded
    // wait after another, while no other role has given up (at most kSchedPatience rounds).
    auto post_tile = [&](uint32_t qc, int t, int role, int site, bool patient) -> bool {
        const int q = qc % kTileRing;
        const uint32_t par = ((qc / kTileRing) & 1u) ^ 1u;
        int m = 0, n = 0, rev = 0;
        if (t >= 0) {
            decode_tile(gp.sp, t, m, n);
            rev = k_reversed(m, n) ? 1 : 0;
        }
        bool got = false;
        for (int r = 0; patient && !got && r < kSchedPatience && !*abort_flag; ++r) {
            volatile int quiet = 0;  // a round that runs out reports nothing
            got = mbar_wait<kPair>(sempty(q), par, &quiet, nullptr, role, site);
        }
        if (!got && !mbar_wait<kPair>(sempty(q), par, abort_flag, gp.err, role, site)) return false;
        ring[q] = make_int4(t, m, n, rev);
        if constexpr (kPair) {
            // the other CTA's copy: an asynchronous store whose 16 bytes that CTA's barrier
            // counts, armed by a relaxed arrive (a cluster-scope release arrive would hold
            // this thread up for about a microsecond)
            const uint32_t peer_full = mapa_shared(sfull(q), 1);
            mbar_arrive_expect_tx_remote_relaxed(peer_full, 16);
            st_async_v4(mapa_shared(smem_u32(ring + q), 1), t, m, n, rev, peer_full);
        }
        mbar_arrive(sfull(q));
        return true;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tensormap(&tmA);
            prefetch_tensormap(&tmB);
            if constexpr (MX) {
                prefetch_tensormap(&tmSFA);
                prefetch_tensormap(&tmSFB);
            }
            // work stealing: the scheduler thread takes the next ticket when asked, this many
            // stages before the current tile's last load; with no more tiles than workers
            // every ticket is a launch ticket and there is nothing to ask for
            const int lead_k = gp.k_iters > kTicketLead ? gp.k_iters - kTicketLead : 0;
            const bool ws_ask = ws && leader && gp.sp.tiles > gp.sp.workers;
            bool clc_first = true, clc_pending = false;
            uint32_t clc_phase = 0;
            // launch control: the worker's own tile first, then tiles of clusters it cancels
            // before they start; one request in flight, issued as soon as a tile is taken
            auto clc_fetch = [&]() -> int {
                int t = -1;
                if (clc_first) {
                    clc_first = false;
                    t = worker;
                } else if (clc_pending) {
                    clc_pending = false;
                    if (mbar_wait(clc_bar, clc_phase & 1u, abort_flag, gp.err, kRoleScheduler, 9)) {
                        const int x = clc_query(clc_resp);
                        t = (x < 0 || x / CS >= gp.sp.tiles) ? -1 : x / CS;
                    }
                    ++clc_phase;
                }
                if (t >= 0 && !*abort_flag) {
                    mbar_arrive_expect_tx(clc_bar, 16);
                    clc_try_cancel(clc_resp, clc_bar);
                    clc_pending = true;
                }
                return t;
            };
            uint32_t it = 0, qc = 0;
            int nvis = 0;
            bool ok = true;
            while (ok) {
                const int q = qc % kTileRing;
                if (leader && !sched_thread) {
                    // launch control: this thread takes the tile and writes the ring itself
                    if (!post_tile(qc, *abort_flag ? -1 : clc_fetch(), kRoleProducer, 0, false)) break;
                } else {
                    // read the entry the scheduler thread (or, for the pair's other CTA, the
                    // leader) posted, then hand the entry back
                    if (!mbar_wait<kPair>(sfull(q), (qc / kTileRing) & 1u, abort_flag, gp.err, kRoleProducer, 8)) break;
                }
                const int4 e = ring[q];
                // The leader hands the entry back at once (a CTA-scope arrive).  The pair's
                // other CTA does so after the tile's first loads, whose coordinates consume
                // the entry, so its arrive can be relaxed (a cluster-scope release would hold
                // up those loads).
                if (sched_thread && leader) mbar_arrive(sempty(q));
                bool held = !leader;
                ++qc;
                const int t = e.x, m = e.y, n = e.z;
                const bool rev = e.w != 0;
                if (t < 0) {
                    if (held) mbar_arrive_remote_relaxed(mapa_shared(sempty(q), 0));
                    break;
                }
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
                const int row0 = (m * CS + (int)rank) * L::BM;  // this CTA's rows of A
                const int col0 = n * BN + (int)rank * L::BN_CTA;  // this CTA's slice of B
                for (int k = 0; k < gp.k_iters; ++k, ++it) {
                    const int kc = rev ? gp.k_iters - 1 - k : k;  // K slice loaded at iteration k
                    const int s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1u;
                    if (!mbar_wait(empty(s), ph ^ 1u, abort_flag, gp.err, kRoleProducer, 1)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = base + s * L::STAGE_BYTES;
                    const uint32_t sb = sa + L::A_BYTES;
                    const bool sf_now = MX && (k & 3) == 0;
                    if (leader) mbar_arrive_expect_tx(full(s), CS * (L::TX_BYTES + (sf_now ? L::SF_TX_BYTES : 0)));
                    const uint32_t fb = kPair ? mapa_shared(full(s), 0) : full(s);
                    tma_load<CS>(sa, &tmA, fb, kc * L::BK, row0);
                    if constexpr (B_MN) {
#pragma unroll
                        for (int j = 0; j < L::BN_CTA / 64; ++j)
                            tma_load<CS>(sb + j * 8192, &tmB, fb, col0 + 64 * j, kc * L::BK);
                    } else {
                        tma_load<CS>(sb, &tmB, fb, kc * L::BK, col0);
                    }
                    if constexpr (MX) {
                        if (sf_now) {
                            const int kg = k >> 2;
                            tma_load<CS>(sb + L::B_BYTES, &tmSFA, fb, 0, kg * gp.sfa_rows + m * CS + (int)rank);
                            tma_load<CS>(sa + L::SFB_OFF, &tmSFB, fb, 0, kg * gp.sfb_rows + n * L::NB128);
                        }
                    }
                    if (held) {
                        mbar_arrive_remote_relaxed(mapa_shared(sempty(q), 0));
                        held = false;
                    }
                    if (ws_ask && k == lead_k) mbar_arrive(tk_req);  // ask for the next tile
                }
                if (held) mbar_arrive_remote_relaxed(mapa_shared(sempty(q), 0));  // no load issued
            }
            if (clc_pending) {
                // never leave with an answer still to land in this CTA's shared memory
                volatile int no_abort = 0;
                mbar_wait(clc_bar, clc_phase & 1u, &no_abort, gp.err, kRoleScheduler, 10);
            }
            if (TRACE && gp.tr_counts != nullptr) gp.tr_counts[blockIdx.x] = nvis;
        }
        __syncwarp();
    } else if (warp == 1) {
        // ----------------------------------------------------------------- MMA
        if (leader && lane == 0) {
            uint32_t it = 0, qc = 0, tc = 0;
            bool ok = true;
            while (ok) {
                const int q = qc % kTileRing;
                if (!mbar_wait(sfull(q), (qc / kTileRing) & 1u, abort_flag, gp.err, kRoleMma, 2)) break;
                const int t = ring[q].x;
                mbar_arrive(sempty(q));
                ++qc;
                if (t < 0) break;
                const int acc = tc % L::ACC_BUFS;
                if (!mbar_wait<kPair>(tempty(acc), ((tc / L::ACC_BUFS) & 1u) ^ 1u, abort_flag, gp.err, kRoleMma, 3))
                    break;
                tc_fence_after();
                const uint32_t d = tmem_base + acc * L::ACC_STRIDE;
                // two stages per loop body (MXFP8: 5-7% faster than one stage per body,
                // measured): this single thread runs only about a stage ahead of the pipe
#pragma unroll 2
                for (int k = 0; k < gp.k_iters; ++k, ++it) {
                    const int s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1u;
                    if (!mbar_wait<kPair>(full(s), ph, abort_flag, gp.err, kRoleMma, 4)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = base + s * L::STAGE_BYTES;
                    const uint32_t sb = sa + L::A_BYTES;
                    const uint64_t adesc = make_smem_desc(sa, 16, 1024, kLayoutSw128);
                    const uint64_t bdesc = B_MN ? make_smem_desc(sb, 8192, 1024, kLayoutSw128)
                                                : make_smem_desc(sb, 16, 1024, kLayoutSw128);
                    if constexpr (MX) {
                        const uint32_t buf = (k >> 2) & 1;
                        const uint32_t sfa_t = tmem_base + L::SFA_COL + 4 * buf;
                        const uint32_t sfb_t = tmem_base + L::SFB_COL + 4 * L::NB128 * buf;
                        if ((k & 3) == 0) {
                            // scales of the next four K blocks: smem -> tensor memory
                            tmem_cp_32x128b_x4<CS>(sfa_t, make_smem_desc(sb + L::B_BYTES, 0, 128, kLayoutNone));
#pragma unroll
                            for (int b = 0; b < L::NB128; ++b)
                                tmem_cp_32x128b_x4<CS>(sfb_t + 4 * b,
                                                       make_smem_desc(sa + L::SFB_OFF + 512 * b, 0, 128, kLayoutNone));
                        }
                        // every 32-wide MMA of this 128-wide K block uses the block's scale byte
                        const uint32_t idesc = make_idesc_mxf8(128 * CS, BN, k & 3, k & 3);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_mxf8<CS>(d, adesc + (uint64_t)(2 * kk), bdesc + (uint64_t)(2 * kk), idesc, sfa_t, sfb_t,
                                         (k | kk) != 0 ? 1u : 0u);
                    } else {
                        constexpr uint32_t idesc = make_idesc_bf16(128 * CS, BN, false, B_MN);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            // K-major operands advance 16 elements = 32 bytes inside the
                            // 128-byte swizzle row; the MN-major B advances 16 rows of 128 bytes.
                            const uint64_t a_k = adesc + (uint64_t)(2 * kk);
                            const uint64_t b_k = bdesc + (uint64_t)(B_MN ? 128 * kk : 2 * kk);
                            mma_bf16<CS>(d, a_k, b_k, idesc, (k | kk) != 0 ? 1u : 0u);
                        }
                    }
                    if constexpr (kPair)
                        mma_commit_pair(empty(s), 3);
                    else
                        mma_commit(empty(s));
                }
                if (!ok) break;
                if constexpr (kPair)
                    mma_commit_pair(tfull(acc), 3);
                else
                    mma_commit(tfull(acc));
                ++tc;
            }
            // every MMA issued above has completed once this barrier flips
            if constexpr (kPair)
                mma_commit_pair(mma_done, 1);
            else
                mma_commit(mma_done);
            volatile int no_abort = 0;
            mbar_wait(mma_done, 0, &no_abort, gp.err, kRoleMma, 5);
        }
        __syncwarp();
    } else if (warp == 2) {
        // ---------------------------------------------------------- scheduler
        // Posts the worker's tiles into the ring.  Static orders: as fast as entries free up.
        // Work stealing: the launch ticket at once (no counter round trip), every later
        // ticket when the producer asks for it; then the last worker resets the counters.
        if (leader && lane == 0 && sched_thread) {
            uint32_t qc = 0, ph = 0;
            for (;;) {
                if (ws && qc > 0 && !sch.solo) {
                    if (!mbar_wait(tk_req, ph & 1u, abort_flag, gp.err, kRoleScheduler, 13)) break;
                    ++ph;
                }
                const int t = *abort_flag ? -1 : sch.fetch();
                if (!post_tile(qc, t, kRoleScheduler, 11, true)) break;
                ++qc;
                if (t < 0) break;
            }
            if (ws) sch.finish();
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------------------ epilogue
        const int qw = warp - 4;  // TMEM lane quarter this warp may access
        const uint32_t epi = base + L::EPI_OFF + qw * L::EPI_BUFS * kEpiBufBytes;
        uint32_t qc = 0, tc = 0, chunk = 0;
        while (true) {
            const int q = qc % kTileRing;
            if (!mbar_wait<kPair>(sfull(q), (qc / kTileRing) & 1u, abort_flag, gp.err, kRoleEpilogue, 6)) break;
            const int4 e = ring[q];
            __syncwarp();
            if (lane == 0) arrive_local_or_leader(sempty(q), !leader);
            ++qc;
            if (e.x < 0) break;
            const int acc = tc % L::ACC_BUFS;
            if (!mbar_wait<kPair>(tfull(acc), (tc / L::ACC_BUFS) & 1u, abort_flag, gp.err, kRoleEpilogue, 7)) break;
            tc_fence_after();
            const int row0 = (e.y * CS + (int)rank) * L::BM + 32 * qw;
            const int col0 = e.z * BN;
            const uint32_t tacc = tmem_base + ((uint32_t)(32 * qw) << 16) + acc * L::ACC_STRIDE;
            // fp32 accumulator pair -> bf16x2, with the optional scale and bias fused in
            // (one fma per element; columns past N read no bias)
            auto cvt = [&](uint32_t lo, uint32_t hi, int col) __attribute__((always_inline)) -> uint32_t {
                if (!gp.epi) return pack_bf16x2(lo, hi);
                float b0 = 0.f, b1 = 0.f;
                if (gp.bias != nullptr) {
                    if (col < gp.N) b0 = __ldg(gp.bias + col);
                    if (col + 1 < gp.N) b1 = __ldg(gp.bias + col + 1);
                }
                const float v0 = __fmaf_rn(gp.alpha, __uint_as_float(lo), b0);
                const float v1 = __fmaf_rn(gp.alpha, __uint_as_float(hi), b1);
                return pack_bf16x2(__float_as_uint(v0), __float_as_uint(v1));
            };
            // Stage 64 columns (32 packed bf16 pairs per row) in this warp's 128B-swizzled
            // buffer and store them with one TMA box; edges are clipped by the tensor map.
            auto store_chunk = [&](int c, const uint32_t* w) __attribute__((always_inline)) {
                const uint32_t buf = epi + (chunk % L::EPI_BUFS) * kEpiBufBytes;
                if (lane == 0) {
                    if constexpr (L::EPI_BUFS == 2)
                        bulk_wait_read<1>();
                    else
                        bulk_wait_read<0>();
                }
                __syncwarp();
                const uint32_t rowaddr = buf + lane * 128u;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    st_shared_v4(rowaddr + ((j ^ (lane & 7u)) << 4), w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    const int x = col0 + 64 * c;
                    if (row0 < gp.M && x < gp.N) tma_store_2d(&tmC, buf, x, row0);
                    bulk_commit();
                }
                ++chunk;
            };
            if constexpr (L::ACC_BUFS == 1) {
                // a single accumulator: read all of it into registers (as bf16 pairs), hand
                // it back to the MMA warp at once, then stage and store.  pk[j] holds columns
                // 2j and 2j + 1; the accumulator is read 128 columns per wait, and handed back
                // as soon as the last load has landed, before its columns are converted
                static_assert(BN % 128 == 0, "single-accumulator tiles are read 128 columns at a time");
                uint32_t pk[BN / 2];
#pragma unroll
                for (int h = 0; h < BN / 128; ++h) {
                    uint32_t r[4][32];
#pragma unroll
                    for (int q = 0; q < 4; ++q) tmem_ld_32x32b_x32(tacc + h * 128 + 32 * q, r[q]);
                    tmem_ld_wait();
                    if (h == BN / 128 - 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) arrive_local_or_leader_relaxed(tempty(acc), !leader);
                    }
                    if (!gp.epi) {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
#pragma unroll
                            for (int i = 0; i < 16; ++i) pk[64 * h + 16 * q + i] = pack_bf16x2(r[q][2 * i], r[q][2 * i + 1]);
                    } else {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                pk[64 * h + 16 * q + i] =
                                    cvt(r[q][2 * i], r[q][2 * i + 1], col0 + 128 * h + 32 * q + 2 * i);
                    }
                }
#pragma unroll
                for (int c = 0; c < BN / 64; ++c) store_chunk(c, pk + 32 * c);
            } else {
                constexpr int kFull = BN / 64;  // whole 64-column chunks, stored through TMA
                constexpr int kTail = BN % 64;  // columns of a narrower last chunk (MXFP8 256 x 224)
#pragma unroll 1
                for (int c = 0; c < kFull; ++c) {
                    uint32_t r0[32], r1[32], w[32];
                    tmem_ld_32x32b_x32(tacc + c * 64, r0);
                    tmem_ld_32x32b_x32(tacc + c * 64 + 32, r1);
                    tmem_ld_wait();
                    if (kTail == 0 && c == kFull - 1) {
                        // accumulator fully read: hand it back to the MMA warp
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) arrive_local_or_leader_relaxed(tempty(acc), !leader);
                    }
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        w[i] = cvt(r0[2 * i], r0[2 * i + 1], col0 + 64 * c + 2 * i);
                        w[16 + i] = cvt(r1[2 * i], r1[2 * i + 1], col0 + 64 * c + 32 + 2 * i);
                    }
                    store_chunk(c, w);
                }
                if constexpr (kTail > 0) {
                    // The last kTail columns: read them, hand the accumulator back, and store
                    // each thread's row segment with 16-byte global stores.  A TMA box of 64
                    // columns would overwrite the next tile's first columns.  Rows past M and
                    // columns past N are not written.
                    static_assert(kTail == 16 || kTail == 32 || kTail == 48, "tail is 16, 32 or 48 columns");
                    uint32_t ta[32], tb[16];
                    const uint32_t tcol = tacc + kFull * 64;
                    if constexpr (kTail == 16) {
                        tmem_ld_32x32b_x16(tcol, tb);
                    } else {
                        tmem_ld_32x32b_x32(tcol, ta);
                        if constexpr (kTail == 48) tmem_ld_32x32b_x16(tcol + 32, tb);
                    }
                    tmem_ld_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) arrive_local_or_leader_relaxed(tempty(acc), !leader);
                    auto tv = [&](int i) __attribute__((always_inline)) -> uint32_t {
                        if constexpr (kTail == 16)
                            return tb[i];
                        else if constexpr (kTail == 32)
                            return ta[i];
                        else
                            return i < 32 ? ta[i] : tb[i - 32];
                    };
                    const int row = row0 + (int)lane;
                    const int cb = col0 + kFull * 64;
                    if (row < gp.M) {
                        uint16_t* dst = gp.C + (int64_t)row * gp.ldc + cb;
#pragma unroll
                        for (int j = 0; j < kTail / 8; ++j) {
                            uint32_t q[4];
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                q[i] = cvt(tv(8 * j + 2 * i), tv(8 * j + 2 * i + 1), cb + 8 * j + 2 * i);
                            const int c8 = cb + 8 * j;
                            if (c8 + 8 <= gp.N) {
                                st_global_v4(dst + 8 * j, q[0], q[1], q[2], q[3]);
                            } else {
                                for (int e = 0; e < 8 && c8 + e < gp.N; ++e)
                                    dst[8 * j + e] = (uint16_t)(q[e >> 1] >> (16 * (e & 1)));
                            }
                        }
                    }
                }
            }
            ++tc;
        }
        if (lane == 0) bulk_wait<0>();
        __syncwarp();
    }

    if constexpr (kPair)
        cluster_sync();
    else
        __syncthreads();
    if (TRACE && threadIdx.x == 0 && gp.tr_times != nullptr) gp.tr_times[2 * blockIdx.x + 1] = (int64_t)globaltimer();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<CS>(tmem_base, L::TMEM_COLS);
    }
}

// MXFP8 scales: plain [rows][K/128] bytes -> for each group of four 128-wide K blocks and
// each block of 128 rows, 512 bytes in the tensor-memory copy layout (byte
// lane*16 + c*4 + j holds row c*32 + lane of the block, K block 4*group + j; zero past the
// edges).  Output row (group * blocks + block) is one 128-word line: group-major, block
// minor.  A's blocks are plain 128-row blocks.  B's blocks are cut per tile of `tile_n` rows,
// `nbt` blocks per tile (tile_n = 128, nbt = 1 gives plain blocks): block b of tile t covers
// rows t*tile_n + b*128 ... up to the tile's end.
__global__ void sf_repack_kernel(const uint8_t* __restrict__ sfa, const uint8_t* __restrict__ sfb, int M, int N,
                                 int kb, int kgroups, int ma, int nb, int tile_n, int nbt,
                                 uint32_t* __restrict__ outa, uint32_t* __restrict__ outb) {
    const int64_t words_a = (int64_t)kgroups * ma * 128;
    const int64_t words_b = (int64_t)kgroups * nb * 128;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < words_a + words_b;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const bool is_a = idx < words_a;
        const int64_t i = is_a ? idx : idx - words_a;
        const int blocks = is_a ? ma : nb;
        const int rows = is_a ? M : N;
        const uint8_t* src = is_a ? sfa : sfb;
        const int w = (int)(i & 127);
        const int64_t line = i >> 7;
        const int blk = (int)(line % blocks);
        const int kg = (int)(line / blocks);
        const int in_block = (w & 3) * 32 + (w >> 2);
        const int per_tile = is_a ? 1 : nbt;
        const int span = is_a ? 128 : tile_n;
        const int b = blk % per_tile;
        const int64_t r = (int64_t)(blk / per_tile) * span + b * 128 + in_block;
        uint32_t v = 0;
        if (b * 128 + in_block < span && r < rows) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int kbi = kg * 4 + j;
                if (kbi < kb) v |= (uint32_t)src[r * kb + kbi] << (8 * j);
            }
        }
        (is_a ? outa : outb)[i] = v;
    }
}

}  // namespace pgt
