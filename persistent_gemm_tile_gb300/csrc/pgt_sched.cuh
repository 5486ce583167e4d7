// Device tile scheduler: the order in which a persistent worker (a CTA, or a CTA pair)
// visits output tiles, and the tile id -> (m_idx, n_idx) decodes.
//
// Orders follow "Implement persistent kernels" (helion PR #238): persistent_blocked gives
// worker p the contiguous range [p*B, min((p+1)*B, T)) with B = ceil(T/P);
// persistent_interleaved gives p, p+P, p+2P, ...  The swizzled mode walks the same waves
// as the 2-CTA kernel of "[Feature] Introduce tile scheduler" (tilelang PR #2441):
// tile_id = num_clusters * wave + cluster_id.  Work stealing follows "Work Stealing
// Scheduler Kernel" (tritonBLAS PR #65): int32 tile counters, one per group of workers,
// worker p homed on counter p mod G, all counters zero at launch.
#pragma once

#include "pgt_device.cuh"

namespace pgt {

enum : int { kBlocked = 0, kInterleaved = 1, kSwizzled = 2, kWorkStealing = 3, kBlockedGroupedM = 4,
             kLaunchControl = 5 };

// One counter per 128-byte line so counters of different groups never share a line
// ("8-way spread contention" in the tritonBLAS PR).
constexpr int kCounterStride = 32;

struct SchedParams {
    int tiles;      // T = m_tiles * n_tiles
    int m_tiles;    // worker-tile rows (cluster rows)
    int n_tiles;    // tile columns
    int mode;       // kBlocked .. kBlockedGroupedM
    int group;      // group width, already clamped to the grid (>= 1)
    int ws_groups;  // counter groups (>= 1)
    int ws_layout;  // tile ownership of the counter groups: 0 ranges, 1 striped
    int workers;    // P
    int* counters;  // ws_groups * kCounterStride ints, zero at launch
    int* done;      // workers that have finished fetching
    const int* release;  // work stealing: per-group release flags (may be null)
};

// Linear decode: tile rows vary fastest (helion pid_0 = vpid % num_blocks_0).
__device__ __forceinline__ void decode_linear(int t, int m_tiles, int& m, int& n) {
    n = t / m_tiles;
    m = t - n * m_tiles;
}

// Column-group swizzle (tilelang): groups of `G` tile columns; inside a group the column
// cycles fastest over the group's width, then the cluster row advances.  The last group
// may be narrower than G.  Equal to the page's bx_cluster / by formulas when
// n_tiles % G == 0.
__device__ __forceinline__ void decode_swizzled(int t, int G, int m_tiles, int n_tiles, int& m, int& n) {
    const int span = G * m_tiles;
    const int g = t / span;
    const int r = t - g * span;
    const int gw = min(G, n_tiles - g * G);
    const int q = r / gw;
    m = q;
    n = g * G + (r - q * gw);
}

// L2 grouping (helion "PERSISTENT BLOCKED WITH L2 GROUPING"): bands of G tile rows, rows
// fastest inside a band.
__device__ __forceinline__ void decode_grouped_m(int t, int G, int m_tiles, int n_tiles, int& m, int& n) {
    const int per_group = G * n_tiles;
    const int group_id = t / per_group;
    const int first_m = group_id * G;
    const int gsm = min(m_tiles - first_m, G);
    const int local = t - group_id * per_group;
    const int q = local / gsm;
    m = first_m + (local - q * gsm);
    n = q;
}

__device__ __forceinline__ void decode_tile(const SchedParams& p, int t, int& m, int& n) {
    if (p.mode == kBlockedGroupedM) {
        // the L2-grouping formula for every group width (width 1 gives columns fastest)
        decode_grouped_m(t, p.group, p.m_tiles, p.n_tiles, m, n);
    } else if (p.mode == kBlocked || p.mode == kInterleaved || p.group <= 1) {
        decode_linear(t, p.m_tiles, m, n);
    } else {
        decode_swizzled(t, p.group, p.m_tiles, p.n_tiles, m, n);
    }
}

// Work-stealing counter groups.  Worker c of P is homed on group c mod G, so n_g = P div G +
// (g < P mod G) workers are homed on g and S_g = g (P div G) + min(g, P mod G) on the groups
// before it.  Group g owns a share of the T tiles in proportion to n_g (with P a multiple of
// G, as on the tritonBLAS PR's GPU with its equal XCDs, the even split):
//   ranges:  the contiguous [floor(T S_g / P), floor(T S_{g+1} / P)), ticket j = start + j
//            (one region per group, as the per-XCD counters);
//   striped: the tiles t with (t mod P) mod G = g in increasing order, i.e. those the
//            workers homed on g would visit in the interleaved order (every group on the
//            same front of the decode order: one shared L2); ticket j is
//            (j div n_g) P + g + (j mod n_g) G.
// With T = a P + b, floor(T S / P) = a S + floor(b S / P), and b S < P^2 fits 32 unsigned
// bits for P <= 65535 (the host's limit), so a lookup costs one 32-bit division.  (Host
// callable too, for a test against the oracle.)
struct WsGroups {
    int G, layout, P, a, b, wq, wr;
    __host__ __device__ __forceinline__ void init(int T, int workers, int groups, int lay) {
        G = groups;
        layout = lay;
        P = workers;
        a = T / workers;
        b = T - a * workers;
        wq = workers / groups;
        wr = workers - wq * groups;
    }
    __host__ __device__ __forceinline__ int homed(int g) const { return wq + (g < wr ? 1 : 0); }
    __host__ __device__ __forceinline__ int start(int g) const {
        const unsigned s = (unsigned)(g * wq + (g < wr ? g : wr));
        return (int)(s * (unsigned)a + s * (unsigned)b / (unsigned)P);
    }
    __host__ __device__ __forceinline__ int size(int g) const {
        if (layout == 1) return a * homed(g) + (b > g ? (b - g - 1) / G + 1 : 0);
        return start(g + 1) - start(g);
    }
    __host__ __device__ __forceinline__ int tile(int g, int ticket) const {
        if (layout == 1) {
            const int n = homed(g);
            const int round = ticket / n;
            return round * P + g + (ticket - round * n) * G;
        }
        return start(g) + ticket;
    }
};

// Per-worker scheduler.  Static modes are pure functions of (worker, iteration); work
// stealing draws tickets from the counters.
//
// Work stealing keeps the protocol's round trips off the tile pipeline:
//  * a worker's first ticket of its home group is implied: worker w, homed on g = w mod G,
//    takes ticket w div G at launch, and the counter of g hands out tickets from n_g (the
//    number of workers homed on g) on, so counters still start every launch at zero;
//  * later tickets are taken by a thread of their own (the GEMM kernel's scheduler thread), a
//    few stages before the producer needs the next tile, so the counter round trips never
//    sit in the producer's instruction stream (an early ticket taken by the producer itself
//    measured slower than a late one);
//  * the home group's release flag is read one decision ahead and its value used at the
//    next one, so no decision waits for it.  A worker released before launch still runs
//    its implied first tile; a release raised later lands within a tile;
//  * with no more tiles than workers (T <= P) every ticket of every group is implied, so a
//    worker runs its launch tile, if it has one, and stops without touching a counter.
// Every tile is still handed out exactly once, and a worker's tickets in a group still
// increase (the validator's invariants).
struct Scheduler {
    SchedParams p;
    int next;    // static: next tile id
    int end;     // static: one past the last tile id
    int stride;  // static: step between tile ids
    int home;    // work stealing: home group
    int cursor;  // work stealing: groups found exhausted, counted from home
    int first;   // work stealing: the implied first ticket of the home group (-1 once used)
    bool stopped;  // work stealing: the home group's release flag was seen
    int rel;       // work stealing: the release flag as last read (used at the next decision)
    WsGroups wg;   // work stealing: the groups' tiles
    bool solo;     // work stealing: T <= P, every ticket implied (no counter is touched)
    static constexpr int kScan = 8;  // counters read at once by a steal scan

    __device__ __forceinline__ void init(const SchedParams& params, int worker) {
        p = params;
        home = 0;
        cursor = 0;
        first = -1;
        stopped = false;
        rel = 0;
        solo = false;
        if (p.mode == kBlocked || p.mode == kBlockedGroupedM) {
            const int B = (p.tiles + p.workers - 1) / p.workers;
            const long long s = static_cast<long long>(worker) * B;
            next = static_cast<int>(s < p.tiles ? s : p.tiles);
            end = static_cast<int>(s + B < p.tiles ? s + B : p.tiles);
            stride = 1;
        } else if (p.mode == kWorkStealing) {
            wg.init(p.tiles, p.workers, p.ws_groups, p.ws_layout);
            solo = p.tiles <= p.workers;
            home = worker % p.ws_groups;
            first = worker / p.ws_groups;
            next = end = 0;
            stride = 0;
            read_release();
        } else {
            next = worker;
            end = p.tiles;
            stride = p.workers;
        }
    }

    // Work stealing: the tile of this worker's launch ticket, or -1 when its home group holds
    // no such ticket (the worker then starts by stealing).  No side effect: a second thread
    // of the worker may run the scheduler and drop the ticket (drop_launch_ticket) after the
    // first has taken the tile itself.
    __device__ __forceinline__ int launch_tile() const {
        return (p.mode == kWorkStealing && first >= 0 && first < wg.size(home)) ? wg.tile(home, first) : -1;
    }
    __device__ __forceinline__ void drop_launch_ticket() {
        if (launch_tile() >= 0) first = -1;
    }

    // Work stealing: workers homed on group g (G <= P, so at least one): the implied tickets
    // 0 .. n_g - 1 of g belong to them, and the counter's value c stands for ticket c + n_g.
    __device__ __forceinline__ int homed(int g) const { return wg.homed(g); }

    // Work stealing: the counter of the group `offset` places after home (0 past the last).
    __device__ __forceinline__ int read_counter(int offset) const {
        if (offset >= p.ws_groups) return 0;
        int g = home + offset;
        if (g >= p.ws_groups) g -= p.ws_groups;
        return *reinterpret_cast<const volatile int*>(p.counters + g * kCounterStride);
    }

    // Work stealing: cooperative release.  Start reading the home group's flag (never group
    // 0's: its workers finish whatever is left); the value is used by the next decision.
    __device__ __forceinline__ void read_release() {
        rel = (p.release != nullptr && home != 0) ? *reinterpret_cast<const volatile int*>(p.release + home) : 0;
    }

    // Next tile id, or -1 when this worker is done.
    __device__ __forceinline__ int fetch() {
        if (p.mode == kWorkStealing) {
            // home group first; once it is exhausted, steal from the following groups.  Counters
            // only grow during a launch, so a group whose counter already reads at its size is
            // exhausted: the steal scan reads up to kScan counters at once (independent loads)
            // and takes an atomic ticket only where one may be left.
            const int size_home = wg.size(home);
            if (first >= 0) {
                const int t = first;
                first = -1;
                if (t < size_home) return wg.tile(home, t);
                if (solo) return -1;  // every other ticket is some other worker's launch tile
                cursor = 1;  // an implied ticket past the group's size: every ticket of it is taken
                if (rel != 0) {  // and stealing takes atomics, which a release forbids
                    stopped = true;
                    return -1;
                }
                read_release();
            } else if (solo) {
                return -1;
            } else {
                if (stopped || rel != 0) {
                    stopped = true;
                    return -1;
                }
                read_release();
                if (cursor == 0) {
                    const int ticket = atomicAdd(p.counters + home * kCounterStride, 1) + homed(home);
                    if (ticket < size_home) return wg.tile(home, ticket);
                    cursor = 1;
                }
            }
            while (cursor < p.ws_groups) {
                // A value that already reaches the group's size means exhausted; one below it
                // is only a hint (the atomic decides).
                int seen[kScan];
#pragma unroll
                for (int j = 0; j < kScan; ++j) seen[j] = read_counter(cursor + j);
                // invariant: seen[j] belongs to the group `cursor` points at in step j
#pragma unroll
                for (int j = 0; j < kScan; ++j) {
                    if (cursor >= p.ws_groups) break;
                    int g = home + cursor;
                    while (g >= p.ws_groups) g -= p.ws_groups;
                    const int size = wg.size(g);
                    const int n = homed(g);
                    if (seen[j] + n < size) {
                        const int ticket = atomicAdd(p.counters + g * kCounterStride, 1) + n;
                        if (ticket < size) return wg.tile(g, ticket);
                    }
                    ++cursor;
                }
            }
            return -1;
        }
        if (next >= end) return -1;
        const int t = next;
        next += stride;
        return t;
    }

    // Static modes only: the next tiles of this worker's order, at most `max` of them.  They
    // form the run first, first + step, first + 2 step, ...; returns how many (0 when done).
    __device__ __forceinline__ int fetch_run(int max, int& first, int& step) {
        first = next;
        step = stride;
        if (next >= end) return 0;
        const int left = (end - next + stride - 1) / stride;
        const int n = left < max ? left : max;
        next += n * stride;
        return n;
    }

    // Work stealing: called once by every worker after its last fetch.  The last worker
    // to finish returns every counter to zero for the next launch.
    // The done counter's add releases this worker's tickets and acquires those of the workers
    // that finished before it, so the last one resets counters no other worker still uses;
    // the next launch (a later kernel) sees the zeros.
    __device__ __forceinline__ void finish() {
        if (p.mode != kWorkStealing || solo) return;  // (T <= P: no counter was touched)
        const int prev = atom_add_acq_rel_gpu(p.done, 1);
        if (prev == p.workers - 1) {
            for (int g = 0; g < p.ws_groups; ++g) st_relaxed_gpu(p.counters + g * kCounterStride, 0);
            st_relaxed_gpu(p.done, 0);
        }
    }
};

}  // namespace pgt
