"""Tile-scheduler oracle: which output tiles each persistent worker visits, in order.

Test infrastructure only.  A *worker* is one persistent CTA (1-CTA kernels) or one
CTA pair (2-CTA clusters); ``P`` is the number of workers launched.  Tiles are
numbered ``t in [0, T)``; the decode maps ``t`` to ``(m_idx, n_idx)`` where ``m_idx``
counts cluster rows (``cs * BM`` rows of C each) and ``n_idx`` counts ``BN`` columns.
For a CTA of rank ``cta_id`` inside its pair the tile row is ``bx = m_idx * cs + cta_id``.

Orders (helion "Implement persistent kernels", persistent_blocked / persistent_interleaved
kernels; tilelang "Introduce tile scheduler", the waves loop of the 2-CTA kernel):

* blocked: worker p visits ``[p*B, min((p+1)*B, T))`` with ``B = ceil(T / P)``.
* interleaved: worker p visits ``p, p+P, p+2P, ...``; the iteration index is the
  tilelang "wave" ``w`` with ``tile_id = num_clusters * w + cluster_id``.

Decodes:

* linear (helion): ``m = t mod m_tiles``, ``n = t div m_tiles`` (rows vary fastest).
* swizzled (tilelang, group of ``G`` column blocks): within a group of ``G*mc`` tiles the
  column cycles fastest over the group's width, then the cluster row advances.  This is
  the page's ``bx_cluster = (t // G) % mc``, ``by = t % G + (t // G) // mc * G`` whenever
  ``n_blocks % G == 0``; a ragged last group takes the width ``n_blocks - g*G``
  (reading: the page asserts divisibility instead).  ``mc = ceil(m_blocks / cs)``
  (reading: the page floors it, which drops rows; the review on that kernel notes the
  out-of-range ``bx`` this produces).
* grouped-M (helion "PERSISTENT BLOCKED WITH L2 GROUPING"): bands of ``G`` tile rows,
  rows fastest inside a band.

Work stealing (tritonBLAS "Work Stealing Scheduler Kernel": per-XCD int32 tile counters
indexed by ``pid % NUM_XCDS``, reset before each launch).  The fetch body is not on that
page; the reading adopted here: ``G_ws`` counters; worker ``c`` of ``P`` has the home group
``c mod G_ws``, so ``n_g`` workers are homed on group ``g``; group ``g`` owns the contiguous
tile range ``[floor(T*S_g/P), floor(T*S_{g+1}/P))`` with ``S_g = n_0 + ... + n_{g-1}``, a share
of the tiles in proportion to its home workers (on the page's GPU every XCD holds the same
number of CUs, so this is the even split ``[floor(g*T/G_ws), floor((g+1)*T/G_ws))`` whenever
``G_ws`` divides ``P``); a fetch is ``ticket = atomic_add(counter[g], 1)`` and succeeds when
``ticket < size_g`` (tile ``start_g + ticket``); an exhausted group sends the worker on to
``g+1, g+2, ...`` (mod ``G_ws``) and it stops once it has found all ``G_ws`` groups
exhausted.  Stolen tiles are decoded with the swizzled decode (linear when ``G <= 1``).
The visit order is not deterministic, so only the properties in :func:`check_ws_trace`
are fixed.

Tile ownership ``layout``: ``WS_RANGES`` is the reading above (the page's per-XCD
counters, each over its own contiguous range, so each XCD's L2 sees one region).
``WS_STRIPED`` is a variant for a GPU whose L2 all groups share: tile ``t`` belongs to the
home group of worker ``t mod P``, i.e. group ``(t mod P) mod G_ws``, in increasing order (the
tiles that worker would visit in the interleaved order), so the groups advance together
along the decode order; whenever ``G_ws`` divides ``P`` that is ``t mod G_ws == g``, ticket
``j`` being tile ``j*G_ws + g``.  Counters, homes, stealing, release and reset are
unchanged.

First tickets assigned at launch (``implied_first``): the page's loop takes every ticket
from a counter; the GB300 build assigns worker ``c``'s first ticket without an atomic:
ticket ``c div G_ws`` of its home group, which is exactly the ticket it would draw if every
worker fetched once before any fetched twice.  The counter of group ``g`` then stands for
tickets from ``n_g`` on, ``n_g`` being the number of workers homed on ``g``, and still
starts at zero.  A worker released before launch keeps its assigned tile (release gates
only the tickets drawn from counters).  The invariants of :func:`check_ws_trace` hold
unchanged.
"""
from __future__ import annotations

from dataclasses import dataclass

BLOCKED, INTERLEAVED, SWIZZLED, WORK_STEALING, BLOCKED_GROUPED_M, LAUNCH_CONTROL = 0, 1, 2, 3, 4, 5
WS_RANGES, WS_STRIPED = 0, 1
MODE_NAMES = {
    BLOCKED: "blocked",
    INTERLEAVED: "interleaved",
    SWIZZLED: "swizzled",
    WORK_STEALING: "work_stealing",
    BLOCKED_GROUPED_M: "blocked_grouped_m",
    LAUNCH_CONTROL: "launch_control",
}


def cdiv(a: int, b: int) -> int:
    return -(-a // b)


@dataclass(frozen=True)
class Grid:
    """Tile-grid geometry for C (M x N) cut into (cs*BM) x BN cluster tiles."""

    m_blocks: int  # CTA tile rows: ceil(M / BM)
    n_blocks: int  # tile columns: ceil(N / BN)
    cs: int  # CTAs per cluster along M (1 or 2)

    @property
    def m_clusters(self) -> int:
        return cdiv(self.m_blocks, self.cs)

    @property
    def tiles(self) -> int:
        return self.m_clusters * self.n_blocks


def grid_for(M: int, N: int, BM: int, BN: int, cs: int = 1) -> Grid:
    return Grid(cdiv(M, BM), cdiv(N, BN), cs)


# ----------------------------------------------------------------------------- decodes
def decode_linear(t: int, m_tiles: int) -> tuple[int, int]:
    return t % m_tiles, t // m_tiles


def decode_swizzled(t: int, G: int, mc: int, n_blocks: int) -> tuple[int, int]:
    """Tile id -> (cluster row, column) with column groups of width G."""
    span = G * mc
    g, r = divmod(t, span)
    gw = min(G, n_blocks - g * G)
    return r // gw, g * G + r % gw


def decode_grouped_m(t: int, G: int, m_tiles: int, n_tiles: int) -> tuple[int, int]:
    per_group = G * n_tiles
    group_id = t // per_group
    first_m = group_id * G
    gsm = min(m_tiles - first_m, G)
    local = t % per_group
    return first_m + local % gsm, local // gsm


def decode(mode: int, t: int, grid: Grid, G: int) -> tuple[int, int]:
    mc, nb = grid.m_clusters, grid.n_blocks
    if mode in (BLOCKED, INTERLEAVED):
        return decode_linear(t, mc)
    if mode == BLOCKED_GROUPED_M:
        return decode_grouped_m(t, max(G, 1), mc, nb)
    if mode in (SWIZZLED, WORK_STEALING, LAUNCH_CONTROL):
        if G <= 1:
            return decode_linear(t, mc)
        return decode_swizzled(t, G, mc, nb)
    raise ValueError(f"unknown mode {mode}")


# ------------------------------------------------------------------------------ orders
def order_blocked(T: int, P: int) -> list[list[int]]:
    B = cdiv(T, P) if T else 0
    return [list(range(p * B, min((p + 1) * B, T))) for p in range(P)]


def order_interleaved(T: int, P: int) -> list[list[int]]:
    return [list(range(p, T, P)) for p in range(P)]


def static_schedule(mode: int, grid: Grid, P: int, G: int) -> list[list[tuple[int, int, int, int]]]:
    """Per worker, the ordered visits ``(iter, tile_id, m_idx, n_idx)`` of a static mode."""
    T = grid.tiles
    if mode in (BLOCKED, BLOCKED_GROUPED_M):
        orders = order_blocked(T, P)
    elif mode in (INTERLEAVED, SWIZZLED):
        orders = order_interleaved(T, P)
    else:
        raise ValueError("work stealing has no static schedule; use ws_simulate")
    out = []
    for tiles in orders:
        out.append([(i, t, *decode(mode, t, grid, G)) for i, t in enumerate(tiles)])
    return out


# ------------------------------------------------------------------------ work stealing
def ws_homed(P: int, groups: int) -> list[int]:
    """Workers homed on each counter group (worker c's home is c mod groups)."""
    return [sum(1 for c in range(P) if c % groups == g) for g in range(groups)]


def ws_partition(T: int, groups: int, P: int) -> list[tuple[int, int]]:
    """(start, size) of each counter group's contiguous tile range: group g's share of the T
    tiles is in proportion to the workers homed on it."""
    S = [0]
    for n in ws_homed(P, groups):
        S.append(S[-1] + n)
    bounds = [(T * s) // P for s in S]
    return [(bounds[g], bounds[g + 1] - bounds[g]) for g in range(groups)]


def ws_group_tiles(T: int, groups: int, layout: int, P: int) -> list[list[int]]:
    """Each counter group's tiles in ticket order (ticket j is the list's j-th tile)."""
    if layout == WS_RANGES:
        return [list(range(s, s + n)) for s, n in ws_partition(T, groups, P)]
    if layout == WS_STRIPED:
        return [[t for t in range(T) if (t % P) % groups == g] for g in range(groups)]
    raise ValueError(f"unknown tile layout {layout}")


class WsState:
    """Counters plus each worker's cursor: the sequential model of the ticket protocol.
    With ``implied_first`` each worker's first ticket is assigned at launch (module notes)."""

    def __init__(self, T: int, P: int, groups: int, layout: int = WS_RANGES, implied_first: bool = False):
        self.T, self.P, self.groups = T, P, groups
        self.tiles = ws_group_tiles(T, groups, layout, P)
        self.counter = [0] * groups
        self.cursor = [0] * P  # groups already found exhausted, counted from home
        self.done = [False] * P
        self.implied_first = implied_first
        self.started = [False] * P
        # tickets assigned at launch per group: one per worker homed there
        self.offset = ws_homed(P, groups) if implied_first else [0] * groups

    def fetch(self, c: int, released=frozenset()) -> int:
        """One fetch by worker c; returns a tile id or -1 once every group is exhausted.

        Cooperative release (tritonBLAS "Work Stealing Scheduler Kernel", the commits "one
        live flag per XCD" and "Request CU release"; the mechanism is not on the page).
        Reading: before each fetch a worker reads its home group's flag and, if the group is
        in ``released``, stops taking tiles; group 0 is never released, so its workers
        always finish the remaining tiles by stealing."""
        home = c % self.groups
        if self.implied_first and not self.started[c]:
            self.started[c] = True
            j = c // self.groups  # the ticket assigned at launch
            if j < len(self.tiles[home]):
                return self.tiles[home][j]
            self.cursor[c] = 1  # home holds no ticket for this worker: all of them are assigned
        if home != 0 and home in released:
            self.done[c] = True
            return -1
        while self.cursor[c] < self.groups:
            g = (home + self.cursor[c]) % self.groups
            ticket = self.counter[g] + self.offset[g]
            self.counter[g] += 1  # the atomic add
            if ticket < len(self.tiles[g]):
                return self.tiles[g][ticket]
            self.cursor[c] += 1
        self.done[c] = True
        return -1


def ws_simulate(T: int, P: int, groups: int, pick, release_at=None, layout: int = WS_RANGES,
                implied_first: bool = False) -> list[list[int]]:
    """Run the protocol with workers fetching in the order chosen by ``pick(live) -> c``.
    ``release_at(step) -> set of released groups`` models flags raised while it runs."""
    st = WsState(T, P, groups, layout, implied_first)
    visits: list[list[int]] = [[] for _ in range(P)]
    live = list(range(P))
    step = 0
    while live:
        c = pick(live)
        released = release_at(step) if release_at else frozenset()
        step += 1
        t = st.fetch(c, released)
        if t < 0:
            live.remove(c)
        else:
            visits[c].append(t)
    return visits


def check_ws_trace(visits: list[list[int]], T: int, groups: int, layout: int = WS_RANGES) -> None:
    """Validate a work-stealing visit log (per worker, tile ids in visit order).

    Raises AssertionError unless: every tile in [0, T) is visited exactly once; inside each
    counter group a worker's tickets increase; and a worker's groups follow its cyclic
    order from home (home, home+1, ...), never going back to a group it left.  The worker
    count P, on which the groups' tiles depend, is the number of lists.
    """
    flat = sorted(t for v in visits for t in v)
    assert flat == list(range(T)), "work-stealing visits are not a permutation of the tiles"
    owner, ticket = {}, {}
    for g, tiles in enumerate(ws_group_tiles(T, groups, layout, len(visits))):
        for j, t in enumerate(tiles):
            owner[t], ticket[t] = g, j
    for c, v in enumerate(visits):
        home = c % groups
        last_off, last_j = -1, -1
        for t in v:
            off = (owner[t] - home) % groups
            assert off >= last_off, f"worker {c} went back to an earlier group"
            if off == last_off:
                assert ticket[t] > last_j, f"worker {c} tickets not increasing in group {owner[t]}"
            last_off, last_j = off, ticket[t]


# --------------------------------------------------------------- fused multi-space loops
def multi_space_schedule(mode: int, grids: list[Grid], P: int) -> list[list[tuple[int, int, int, int, int]]]:
    """helion "Implement persistent kernels", the multi-loop listings: several independent
    tile spaces share one id range; a worker's ids follow the blocked or interleaved order
    over the total, and each id belongs to the first space whose range holds it, decoded
    linearly (rows fastest) inside that space.  Per worker: (iter, tile_id, space, m, n)."""
    firsts, total = [], 0
    for g in grids:
        firsts.append(total)
        total += g.tiles
    orders = order_blocked(total, P) if mode == BLOCKED else order_interleaved(total, P)
    out = []
    for tiles in orders:
        visits = []
        for i, t in enumerate(tiles):
            s = max(k for k in range(len(grids)) if firsts[k] <= t)
            m, n = decode_linear(t - firsts[s], grids[s].m_clusters)
            visits.append((i, t, s, m, n))
        out.append(visits)
    return out


# ------------------------------------------------------------- hardware launch control
def check_launch_control_trace(visits: list[list[int]], T: int) -> None:
    """Validate a launch-control visit log: one list per launched worker w = 0..T-1 (one per
    tile), tile ids in visit order.  Dynamic scheduling through the hardware (an idiomatic
    Blackwell counterpart of the atomic counters, not on the pages): a worker that ran
    starts with its own tile w and then takes the tiles of workers it cancelled before they
    started; a cancelled worker visits nothing.  Raises AssertionError unless every tile is
    visited exactly once, every non-empty list starts with its own id, and every tile other
    than a list's first belongs to a worker whose own list is empty."""
    assert len(visits) == T, "one list per tile-worker expected"
    flat = sorted(t for v in visits for t in v)
    assert flat == list(range(T)), "launch-control visits are not a permutation of the tiles"
    for w, v in enumerate(visits):
        if v:
            assert v[0] == w, f"worker {w} did not start with its own tile"
            for t in v[1:]:
                assert not visits[t], f"tile {t} was taken from a worker that also ran"
