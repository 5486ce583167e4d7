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

// Range of counter group g: [g*T/G, (g+1)*T/G).
__device__ __forceinline__ int ws_group_start(int g, int T, int G) {
    return static_cast<int>((static_cast<long long>(g) * T) / G);
}

// Tiles owned by counter group g, and the tile its ticket j stands for.  Ranges: the
// contiguous [g*T/G, (g+1)*T/G) (one region per group, as the per-XCD counters of the
// tritonBLAS PR).  Striped: g, g+G, g+2G, ... (every group on the same front of the
// decode order: one shared L2).
__device__ __forceinline__ int ws_group_size(int g, int T, int G, int layout) {
    if (layout == 1) return T / G + (g < T % G ? 1 : 0);
    return ws_group_start(g + 1, T, G) - ws_group_start(g, T, G);
}

__device__ __forceinline__ int ws_group_tile(int g, int ticket, int T, int G, int layout) {
    if (layout == 1) return ticket * G + g;
    return ws_group_start(g, T, G) + ticket;
}

// Per-worker scheduler.  Static modes are pure functions of (worker, iteration); work
// stealing draws tickets from the counters.
struct Scheduler {
    SchedParams p;
    int next;    // static: next tile id
    int end;     // static: one past the last tile id
    int stride;  // static: step between tile ids
    int home;    // work stealing: home group
    int cursor;  // work stealing: groups found exhausted, counted from home

    __device__ __forceinline__ void init(const SchedParams& params, int worker) {
        p = params;
        home = 0;
        cursor = 0;
        if (p.mode == kBlocked || p.mode == kBlockedGroupedM) {
            const int B = (p.tiles + p.workers - 1) / p.workers;
            const long long s = static_cast<long long>(worker) * B;
            next = static_cast<int>(s < p.tiles ? s : p.tiles);
            end = static_cast<int>(s + B < p.tiles ? s + B : p.tiles);
            stride = 1;
        } else if (p.mode == kWorkStealing) {
            home = worker % p.ws_groups;
            next = end = 0;
            stride = 0;
        } else {
            next = worker;
            end = p.tiles;
            stride = p.workers;
        }
    }

    // Next tile id, or -1 when this worker is done.
    __device__ __forceinline__ int fetch() {
        if (p.mode == kWorkStealing) {
            // cooperative release: a raised flag of the home group (never group 0, whose
            // workers finish whatever is left) stops this worker before its next tile
            if (p.release != nullptr && home != 0 &&
                *reinterpret_cast<const volatile int*>(p.release + home) != 0)
                return -1;
            // home group first; once it is exhausted, steal from the following groups.  Counters
            // only grow during a launch, so a group whose counter already reads >= its size is
            // exhausted: the steal scan reads up to kScan counters at once (independent loads)
            // and takes an atomic ticket only where one may be left.
            constexpr int kScan = 8;
            while (cursor < p.ws_groups) {
                if (cursor == 0) {
                    const int size = ws_group_size(home, p.tiles, p.ws_groups, p.ws_layout);
                    const int ticket = atomicAdd(p.counters + home * kCounterStride, 1);
                    if (ticket < size) return ws_group_tile(home, ticket, p.tiles, p.ws_groups, p.ws_layout);
                    cursor = 1;
                    continue;
                }
                int seen[kScan];
#pragma unroll
                for (int j = 0; j < kScan; ++j) {
                    int g = home + cursor + j;
                    while (g >= p.ws_groups) g -= p.ws_groups;
                    seen[j] = cursor + j < p.ws_groups
                                  ? *reinterpret_cast<const volatile int*>(p.counters + g * kCounterStride)
                                  : 0;
                }
                // invariant: seen[j] belongs to the group `cursor` points at in step j
#pragma unroll
                for (int j = 0; j < kScan; ++j) {
                    if (cursor >= p.ws_groups) break;
                    int g = home + cursor;
                    while (g >= p.ws_groups) g -= p.ws_groups;
                    const int size = ws_group_size(g, p.tiles, p.ws_groups, p.ws_layout);
                    if (seen[j] < size) {
                        const int ticket = atomicAdd(p.counters + g * kCounterStride, 1);
                        if (ticket < size) return ws_group_tile(g, ticket, p.tiles, p.ws_groups, p.ws_layout);
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

    // Work stealing: called once by every worker after its last fetch.  The last worker
    // to finish returns every counter to zero for the next launch.
    __device__ __forceinline__ void finish() {
        if (p.mode != kWorkStealing) return;
        __threadfence();
        const int prev = atomicAdd(p.done, 1);
        if (prev == p.workers - 1) {
            for (int g = 0; g < p.ws_groups; ++g) atomicExch(p.counters + g * kCounterStride, 0);
            atomicExch(p.done, 0);
            __threadfence();
        }
    }
};

}  // namespace pgt
