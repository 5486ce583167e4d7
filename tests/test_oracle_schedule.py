"""Pins for oracle.schedule: hand-evaluated page fixtures, the pages' literal formulas,
brute-force bijection checks and planted mistakes in the work-stealing validator."""
import itertools
import random
import threading

import pytest

from oracle import schedule as S


# --------------------------------------------------------------- the pages' formulas, literal
def helion_blocked(total, nsm, pid):
    block_size = -(-total // nsm)
    start = pid * block_size
    end = min(start + block_size, total)
    return list(range(start, end))


def helion_interleaved(total, nsm, pid):
    return list(range(pid, total, nsm))


def helion_l2_group(vpid, num_pid_m, num_pid_n, group=8):
    num_pid_in_group = group * num_pid_n
    group_id = vpid // num_pid_in_group
    first_pid_m = group_id * group
    group_size_m = min(num_pid_m - first_pid_m, group)
    pid_0 = first_pid_m + vpid % num_pid_in_group % group_size_m
    pid_1 = vpid % num_pid_in_group // group_size_m
    return pid_0, pid_1


def tilelang_swizzle(tile_id, group_size, m_clusters):
    bx_cluster = (tile_id // group_size) % m_clusters
    by = (tile_id % group_size) + (tile_id // group_size) // m_clusters * group_size
    return bx_cluster, by


# ------------------------------------------------------------------------- golden fixtures
def test_golden_helion_blocked(golden):
    grid = S.grid_for(64, 48, 32, 16)
    sched = S.static_schedule(S.BLOCKED, grid, 4, 1)
    rows = [(p, i, t, m, n) for p, v in enumerate(sched) for (i, t, m, n) in v]
    assert rows == golden("helion_persistent_blocked_64x48.txt")


def test_golden_helion_interleaved(golden):
    grid = S.grid_for(64, 48, 32, 16)
    sched = S.static_schedule(S.INTERLEAVED, grid, 4, 1)
    rows = [(p, i, t, m, n) for p, v in enumerate(sched) for (i, t, m, n) in v]
    assert rows == golden("helion_persistent_interleaved_64x48.txt")


def test_golden_helion_l2_grouping(golden):
    grid = S.grid_for(320, 32, 32, 16)
    sched = S.static_schedule(S.BLOCKED_GROUPED_M, grid, 8, 8)
    rows = [(p, i, t, m, n) for p, v in enumerate(sched) for (i, t, m, n) in v]
    assert rows == golden("helion_blocked_l2_grouping_320x32.txt")


def test_golden_tilelang_swizzle(golden):
    grid = S.grid_for(512, 512, 128, 128, cs=2)
    sched = S.static_schedule(S.SWIZZLED, grid, 2, 2)  # 2 clusters = 4 CTAs
    rows = []
    for block_id in range(4):
        cluster, cta = divmod(block_id, 2)
        for (w, t, mi, n) in sched[cluster]:
            rows.append((block_id, w, t, mi * 2 + cta, n))
    assert sorted(rows) == sorted(golden("tilelang_swizzle_2cta_512x512.txt"))


# ----------------------------------------------------------------- literal formulas, brute
@pytest.mark.parametrize("T,P", [(t, p) for t in range(0, 40) for p in (1, 2, 3, 5, 8, 13)])
def test_blocked_and_interleaved_match_helion(T, P):
    assert S.order_blocked(T, P) == [helion_blocked(T, P, p) for p in range(P)]
    assert S.order_interleaved(T, P) == [helion_interleaved(T, P, p) for p in range(P)]


@pytest.mark.parametrize("mt,nt,G", list(itertools.product(range(1, 12), range(1, 7), (1, 2, 3, 8))))
def test_grouped_m_matches_helion(mt, nt, G):
    for t in range(mt * nt):
        assert S.decode_grouped_m(t, G, mt, nt) == helion_l2_group(t, mt, nt, G)


@pytest.mark.parametrize("mc,G,ngroups", list(itertools.product(range(1, 7), (1, 2, 3, 4, 16), (1, 2, 3))))
def test_swizzle_matches_tilelang_when_divisible(mc, G, ngroups):
    nb = G * ngroups
    for t in range(mc * nb):
        assert S.decode_swizzled(t, G, mc, nb) == tilelang_swizzle(t, G, mc)


# ----------------------------------------------------------------------------- invariants
MODES = [S.BLOCKED, S.INTERLEAVED, S.SWIZZLED, S.BLOCKED_GROUPED_M]


@pytest.mark.parametrize("mb,nb,cs,G,P", [
    (mb, nb, cs, G, P)
    for mb in (1, 2, 3, 5, 6) for nb in (1, 2, 4, 5) for cs in (1, 2) for G in (1, 2, 3, 4) for P in (1, 3, 4, 8)
])
def test_every_tile_visited_exactly_once(mb, nb, cs, G, P):
    grid = S.Grid(mb, nb, cs)
    cells = {(m, n) for m in range(grid.m_clusters) for n in range(nb)}
    for mode in MODES:
        sched = S.static_schedule(mode, grid, P, G)
        seen = [(m, n) for v in sched for (_, _, m, n) in v]
        assert len(seen) == grid.tiles and set(seen) == cells, S.MODE_NAMES[mode]
        ids = sorted(t for v in sched for (_, t, _, _) in v)
        assert ids == list(range(grid.tiles))
        for v in sched:
            assert [i for (i, _, _, _) in v] == list(range(len(v)))


def test_blocked_contiguous_and_interleaved_stride():
    grid = S.Grid(19, 32, 1)  # 608 tiles, the (4864, 4096) ragged case with 256 x 128 tiles
    P = 152
    blk = S.static_schedule(S.BLOCKED, grid, P, 1)
    assert all(v[-1][1] - v[0][1] == len(v) - 1 for v in blk if v)
    assert sum(1 for v in blk if v) == 152 and {len(v) for v in blk} == {4}
    inter = S.static_schedule(S.INTERLEAVED, grid, P, 1)
    assert all(b[1] - a[1] == P for v in inter for a, b in zip(v, v[1:]))


def test_blocked_idle_workers_when_tiles_do_not_divide():
    # T = 608 tiles, P = 160 workers: ceil(608/160) = 4, so only 152 workers get work
    blk = S.order_blocked(608, 160)
    assert sum(1 for v in blk if v) == 152


def test_decode_reductions():
    for mc, nb in itertools.product(range(1, 9), range(1, 9)):
        for t in range(mc * nb):
            assert S.decode_swizzled(t, 1, mc, nb) == S.decode_linear(t, mc)
            assert S.decode_grouped_m(t, mc, mc, nb) == S.decode_linear(t, mc)
            r, c = divmod(t, nb)  # one group spanning all columns: columns fastest
            assert S.decode_swizzled(t, nb, mc, nb) == (r, c)


def test_ragged_last_swizzle_group_is_a_bijection():
    for mc, nb, G in itertools.product(range(1, 8), range(1, 20), (2, 3, 4, 16)):
        cells = [S.decode_swizzled(t, G, mc, nb) for t in range(mc * nb)]
        assert sorted(cells) == [(m, n) for m in range(mc) for n in range(nb)]


# -------------------------------------------------------------------------- work stealing
def test_ws_partition_covers_tiles():
    for T, G, P in itertools.product(range(0, 50), (1, 2, 3, 8), (1, 3, 8, 9, 76)):
        G = min(G, P)
        part = S.ws_partition(T, G, P)
        ids = [t for (s, n) in part for t in range(s, s + n)]
        assert ids == list(range(T))
        # each group's share is within one tile of T times its part of the workers
        for (_, n), h in zip(part, S.ws_homed(P, G)):
            assert abs(n * P - T * h) < P


def test_ws_homed_counts_workers_by_residue():
    assert S.ws_homed(76, 8) == [10, 10, 10, 10, 9, 9, 9, 9]
    assert S.ws_homed(4, 3) == [2, 1, 1]
    assert S.ws_homed(8, 8) == [1] * 8


def test_ws_group_tiles_hand_evaluated():
    # T = 10 tiles on 3 counters and 3 or 6 workers (one or two homed per group): ranges
    # split at floor(g*10/3) = 0, 3, 6, 10; stripes take every third tile from the group's
    # index
    for P in (3, 6):
        assert S.ws_group_tiles(10, 3, S.WS_RANGES, P) == [[0, 1, 2], [3, 4, 5], [6, 7, 8, 9]]
        assert S.ws_group_tiles(10, 3, S.WS_STRIPED, P) == [[0, 3, 6, 9], [1, 4, 7], [2, 5, 8]]
    # 4 workers: homes 0, 1, 2, 0, so group 0 has two of them.  Ranges: the workers before
    # each group number 0, 2, 3, 4 and the bounds are floor(10*S/4) = 0, 5, 7, 10.  Stripes:
    # tile t goes with worker t mod 4, whose home is (t mod 4) mod 3
    assert S.ws_group_tiles(10, 3, S.WS_RANGES, 4) == [[0, 1, 2, 3, 4], [5, 6], [7, 8, 9]]
    assert S.ws_group_tiles(10, 3, S.WS_STRIPED, 4) == [[0, 3, 4, 7, 8], [1, 5, 9], [2, 6]]
    with pytest.raises(ValueError):
        S.ws_group_tiles(10, 3, 2, 3)


@pytest.mark.parametrize("layout", [S.WS_RANGES, S.WS_STRIPED])
def test_ws_group_tiles_partition_exactly_once(layout):
    for T, G, P in itertools.product(range(0, 60), (1, 2, 3, 7, 8, 16), (16, 19, 76)):
        groups = S.ws_group_tiles(T, G, layout, P)
        assert len(groups) == G
        assert sorted(t for g in groups for t in g) == list(range(T))
        for g, h in zip(groups, S.ws_homed(P, G)):
            assert abs(len(g) * P - T * h) < P * (1 if layout == S.WS_RANGES else 2)
        assert all(g == sorted(g) for g in groups)  # tickets follow tile order
        if P % G == 0:  # the even split of the page's GPU, whatever the worker count
            assert groups == S.ws_group_tiles(T, G, layout, G)


def test_ws_balanced_when_tiles_are_a_multiple_of_workers():
    """T = k P: every group holds exactly k tiles per home worker, in both layouts, so with
    the launch tickets and equal progress no worker needs to steal."""
    for P, G, k in itertools.product((76, 152, 19), (1, 4, 8, 16), (1, 4, 13)):
        G = min(G, P)
        for layout in (S.WS_RANGES, S.WS_STRIPED):
            sizes = [len(g) for g in S.ws_group_tiles(k * P, G, layout, P)]
            assert sizes == [k * h for h in S.ws_homed(P, G)]


def test_ws_striped_first_wave_is_the_static_first_wave():
    # the reason for the striped layout: when P workers (P a multiple of G) take their first
    # home ticket together, worker c gets tile (c div G) * G + c mod G = c, the same tiles
    # the interleaved order runs in its first wave; contiguous ranges spread them instead
    for P, G in ((16, 8), (76, 4), (24, 3)):
        T = 10 * P
        st = S.WsState(T, P, G, S.WS_STRIPED)
        assert sorted(st.fetch(c) for c in range(P)) == list(range(P))
        st = S.WsState(T, P, G, S.WS_RANGES)
        assert sorted(st.fetch(c) for c in range(P)) != list(range(P))


@pytest.mark.parametrize("seed", range(10))
def test_ws_striped_random_interleavings_valid(seed):
    rnd = random.Random(100 + seed)
    T, P, G = rnd.randint(0, 300), rnd.randint(1, 20), rnd.choice([1, 2, 3, 8])
    visits = S.ws_simulate(T, P, G, lambda live: rnd.choice(live), layout=S.WS_STRIPED)
    S.check_ws_trace(visits, T, G, S.WS_STRIPED)


def test_ws_striped_trace_fails_the_ranges_check():
    # a striped log read as if groups owned ranges breaks the ticket-order rule, so the
    # layout argument of the checker matters
    rnd = random.Random(7)
    visits = S.ws_simulate(200, 8, 4, lambda live: rnd.choice(live), layout=S.WS_STRIPED)
    with pytest.raises(AssertionError):
        S.check_ws_trace(visits, 200, 4, S.WS_RANGES)


@pytest.mark.parametrize("plant", ["dup", "drop", "swap"])
def test_ws_striped_checker_rejects_planted_mistakes(plant):
    rnd = random.Random(5)
    visits = [list(v) for v in S.ws_simulate(60, 6, 3, lambda live: rnd.choice(live), layout=S.WS_STRIPED)]
    S.check_ws_trace(visits, 60, 3, S.WS_STRIPED)
    c = max(range(len(visits)), key=lambda i: len(visits[i]))
    if plant == "dup":
        visits[c].append(visits[c][0])
    elif plant == "drop":
        visits[c].pop()
    else:
        visits[c][0], visits[c][1] = visits[c][1], visits[c][0]
    with pytest.raises(AssertionError):
        S.check_ws_trace(visits, 60, 3, S.WS_STRIPED)


# --------------------------------------------- first tickets assigned at launch (reading 22)
@pytest.mark.parametrize("layout", [S.WS_RANGES, S.WS_STRIPED])
@pytest.mark.parametrize("seed", range(6))
def test_ws_implied_first_equals_one_round_in_worker_order(layout, seed):
    """Assigning worker c ticket c div G of its home group at launch is what the page's
    protocol gives when every worker fetches once, in worker order, before any fetches
    again: under that schedule the two models produce the same visits.  (With T >= P + G
    every home group holds a ticket for each of its home workers; with fewer tiles a
    first-round worker of the page's protocol may already steal, and the two models may
    give a stolen tile to different workers, both valid.)"""
    rnd = random.Random(300 + seed)
    P, G = rnd.randint(1, 24), rnd.choice([1, 2, 3, 8])
    G = min(G, P)
    T = rnd.randint(P + G, 400)
    first_round = list(range(P))

    def pick_factory():
        queue = list(first_round)
        r = random.Random(seed)

        def pick(live):
            while queue:
                c = queue.pop(0)
                if c in live:
                    return c
            return r.choice(live)
        return pick
    plain = S.ws_simulate(T, P, G, pick_factory(), layout=layout)
    implied = S.ws_simulate(T, P, G, pick_factory(), layout=layout, implied_first=True)
    assert implied == plain


@pytest.mark.parametrize("layout", [S.WS_RANGES, S.WS_STRIPED])
@pytest.mark.parametrize("seed", range(10))
def test_ws_implied_first_random_interleavings_valid(layout, seed):
    rnd = random.Random(400 + seed)
    T, P = rnd.randint(0, 300), rnd.randint(1, 20)
    G = min(rnd.choice([1, 2, 3, 8]), P)
    visits = S.ws_simulate(T, P, G, lambda live: rnd.choice(live), layout=layout, implied_first=True)
    S.check_ws_trace(visits, T, G, layout)
    for c, v in enumerate(visits):  # each worker's first tile is its launch ticket, when it has one
        tiles = S.ws_group_tiles(T, G, layout, P)[c % G]
        if c // G < len(tiles):
            assert v[0] == tiles[c // G]


@pytest.mark.parametrize("T,P,G", [(0, 4, 4), (1, 8, 4), (3, 20, 8), (9, 12, 5), (30, 30, 8)])
def test_ws_implied_first_few_tiles_valid(T, P, G):
    """Fewer tiles than launch tickets: workers whose launch ticket lies past their group's
    size go straight to stealing, and every tile is still visited once."""
    for layout in (S.WS_RANGES, S.WS_STRIPED):
        for seed in range(5):
            rnd = random.Random(seed)
            visits = S.ws_simulate(T, P, G, lambda live: rnd.choice(live), layout=layout, implied_first=True)
            S.check_ws_trace(visits, T, G, layout)


def test_ws_implied_first_release_from_start_keeps_the_launch_tile():
    T, P, G = 120, 16, 4
    rnd = random.Random(9)
    visits = S.ws_simulate(T, P, G, lambda live: rnd.choice(live), release_at=lambda step: frozenset({1, 2}),
                           implied_first=True)
    S.check_ws_trace(visits, T, G)
    for c, v in enumerate(visits):
        if c % G in (1, 2):
            assert v == S.ws_group_tiles(T, G, S.WS_RANGES, P)[c % G][c // G: c // G + 1]


def test_ws_implied_first_without_the_counter_offset_is_rejected():
    """Planted mistake: counters standing for tickets from 0 instead of from the number of
    home workers hand the launch tickets out twice; the validator must reject the trace."""
    T, P, G = 96, 12, 4
    st = S.WsState(T, P, G, S.WS_RANGES, implied_first=True)
    st.offset = [0] * G
    visits = [[] for _ in range(P)]
    live = list(range(P))
    rnd = random.Random(3)
    while live:
        c = rnd.choice(live)
        t = st.fetch(c)
        if t < 0:
            live.remove(c)
        else:
            visits[c].append(t)
    with pytest.raises(AssertionError):
        S.check_ws_trace(visits, T, G)


def test_ws_single_group_round_robin_is_interleaved():
    T, P = 37, 5
    order = itertools.cycle(range(P))
    visits = S.ws_simulate(T, P, 1, lambda live: next(c for c in order if c in live))
    assert visits == S.order_interleaved(T, P)


@pytest.mark.parametrize("seed", range(20))
def test_ws_random_interleavings_valid(seed):
    rnd = random.Random(seed)
    T, P, G = rnd.randint(0, 300), rnd.randint(1, 20), rnd.choice([1, 2, 3, 8])
    visits = S.ws_simulate(T, P, G, lambda live: rnd.choice(live))
    S.check_ws_trace(visits, T, G)


@pytest.mark.parametrize("layout", [S.WS_RANGES, S.WS_STRIPED])
def test_ws_threads_with_atomic_counters_valid(layout):
    T, P, G = 500, 12, 8
    st = S.WsState(T, P, G, layout)
    lock = threading.Lock()
    visits = [[] for _ in range(P)]

    def fetch(c):
        home = c % G
        while st.cursor[c] < G:
            g = (home + st.cursor[c]) % G
            with lock:  # the atomic add
                ticket = st.counter[g]
                st.counter[g] += 1
            if ticket < len(st.tiles[g]):
                return st.tiles[g][ticket]
            st.cursor[c] += 1
        return -1

    def worker(c):
        while True:
            t = fetch(c)
            if t < 0:
                return
            visits[c].append(t)

    th = [threading.Thread(target=worker, args=(c,)) for c in range(P)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    S.check_ws_trace(visits, T, G, layout)
    # every counter ends at or above its group size (exhausted), never below
    assert all(st.counter[g] >= len(st.tiles[g]) for g in range(G))


def _valid_trace():
    rnd = random.Random(3)
    return S.ws_simulate(60, 6, 3, lambda live: rnd.choice(live))


@pytest.mark.parametrize("plant", ["dup", "drop", "swap", "back"])
def test_ws_checker_rejects_planted_mistakes(plant):
    visits = [list(v) for v in _valid_trace()]
    c = max(range(len(visits)), key=lambda i: len(visits[i]))
    if plant == "dup":
        visits[c].append(visits[c][0])
    elif plant == "drop":
        visits[c].pop()
    elif plant == "swap":
        visits[c][0], visits[c][1] = visits[c][1], visits[c][0]
    elif plant == "back":
        # worker 0 (home group 0) visiting a group-2 tile before a group-0 tile
        part = S.ws_partition(60, 3, 6)
        t_g2 = part[2][0]
        for v in visits:
            if t_g2 in v:
                v.remove(t_g2)
        visits[0].insert(0, t_g2)
        if not any(part[0][0] <= t < part[0][0] + part[0][1] for t in visits[0][1:]):
            t_g0 = part[0][0]
            for v in visits:
                if t_g0 in v:
                    v.remove(t_g0)
            visits[0].append(t_g0)
    with pytest.raises(AssertionError):
        S.check_ws_trace(visits, 60, 3)


# ------------------------------------------------------------------ multi-loop spaces
def helion_multi_loop(total_x, nb0_x, nb0_y, pid):
    """The multi-loop listing's per-pid branch, written literally."""
    pid_shared = pid
    if pid_shared < total_x:
        return 0, pid_shared % nb0_x, pid_shared // nb0_x
    pid_shared -= total_x
    return 1, pid_shared % nb0_y, pid_shared // nb0_y


def test_golden_helion_multi_loop(golden):
    grids = [S.grid_for(64, 32, 32, 16), S.grid_for(32, 48, 32, 16)]
    rows = []
    for order, mode in ((0, S.BLOCKED), (1, S.INTERLEAVED)):
        for p, v in enumerate(S.multi_space_schedule(mode, grids, 3)):
            rows += [(order, p, i, t, s, m, n) for (i, t, s, m, n) in v]
    assert rows == golden("helion_multi_loop_64x32_32x48.txt")


@pytest.mark.parametrize("P", [1, 2, 5, 9])
def test_multi_loop_matches_helion_branch(P):
    grids = [S.Grid(3, 4, 1), S.Grid(5, 2, 1)]
    for mode in (S.BLOCKED, S.INTERLEAVED):
        for v in S.multi_space_schedule(mode, grids, P):
            for (_, t, s, m, n) in v:
                assert (s, m, n) == helion_multi_loop(12, 3, 5, t)
        ids = sorted(t for v in S.multi_space_schedule(mode, grids, P) for (_, t, _, _, _) in v)
        assert ids == list(range(22))


# ------------------------------------------------------------------ cooperative release
@pytest.mark.parametrize("seed", range(12))
def test_ws_release_still_covers_every_tile(seed):
    rnd = random.Random(100 + seed)
    T, P, G = rnd.randint(1, 300), rnd.randint(1, 24), rnd.choice([2, 3, 8])
    rel = frozenset(rnd.sample(range(G), rnd.randint(1, G)))
    switch = rnd.randint(0, T)
    visits = S.ws_simulate(T, P, G, lambda live: rnd.choice(live),
                           release_at=lambda step: rel if step >= switch else frozenset())
    S.check_ws_trace(visits, T, G)


def test_ws_release_from_the_start_leaves_all_to_group_zero():
    T, P, G = 100, 16, 4
    rnd = random.Random(5)
    visits = S.ws_simulate(T, P, G, lambda live: rnd.choice(live), release_at=lambda step: frozenset({0, 1, 2, 3}))
    S.check_ws_trace(visits, T, G)
    assert all(not v for c, v in enumerate(visits) if c % G != 0)
    assert sum(len(v) for c, v in enumerate(visits) if c % G == 0) == T


# ------------------------------------------------------------------ launch control
def _clc_trace():
    # workers 0 and 3 ran; 0 took the tiles of workers 1, 2, 5; 3 took 4
    return [[0, 1, 2, 5], [], [], [3, 4], [], []]


def test_launch_control_checker_accepts_valid_and_decodes_like_swizzled():
    S.check_launch_control_trace(_clc_trace(), 6)
    grid = S.Grid(5, 7, 2)
    for t in range(grid.tiles):
        assert S.decode(S.LAUNCH_CONTROL, t, grid, 4) == S.decode(S.SWIZZLED, t, grid, 4)


@pytest.mark.parametrize("plant", ["dup", "drop", "first", "ran_twice"])
def test_launch_control_checker_rejects_planted_mistakes(plant):
    v = [list(x) for x in _clc_trace()]
    if plant == "dup":
        v[3].append(1)
    elif plant == "drop":
        v[0].pop()
    elif plant == "first":
        v[3] = [4, 3]
    elif plant == "ran_twice":  # worker 2 also ran its own tile, yet 0 claims to have taken it
        v[2] = [2]
        v[0].remove(5)
        v[3].append(5)
    with pytest.raises(AssertionError):
        S.check_launch_control_trace(v, 6)


# ------------------------------------------------- failure injection in the ticket model
@pytest.mark.parametrize("layout", [S.WS_RANGES, S.WS_STRIPED])
def test_ws_stale_counter_is_detected(layout):
    # a counter left non-zero by an earlier launch (what the in-kernel reset and the host
    # reset prevent) skips that group's first tickets: the log misses tiles
    T, P, G = 120, 8, 4
    st = S.WsState(T, P, G, layout)
    st.counter[2] = 5
    rnd = random.Random(11)
    visits = [[] for _ in range(P)]
    live = list(range(P))
    while live:
        c = rnd.choice(live)
        t = st.fetch(c)
        if t < 0:
            live.remove(c)
        else:
            visits[c].append(t)
    assert sum(len(v) for v in visits) == T - 5
    with pytest.raises(AssertionError):
        S.check_ws_trace(visits, T, G, layout)


@pytest.mark.parametrize("layout", [S.WS_RANGES, S.WS_STRIPED])
def test_ws_lost_ticket_is_detected(layout):
    # a worker that takes a ticket and then stops without running the tile (an aborted
    # worker) leaves a hole the validator reports
    T, P, G = 90, 6, 3
    rnd = random.Random(12)
    visits = S.ws_simulate(T, P, G, lambda live: rnd.choice(live), layout=layout)
    S.check_ws_trace(visits, T, G, layout)
    c = max(range(P), key=lambda i: len(visits[i]))
    visits[c].pop(len(visits[c]) // 2)
    with pytest.raises(AssertionError):
        S.check_ws_trace(visits, T, G, layout)


def test_ws_counter_overflow_past_group_size_is_harmless():
    # every exhausted group's counter ends above its size (the failing fetch still adds one);
    # tickets beyond the size never become tiles
    T, P, G = 50, 9, 4
    rnd = random.Random(13)
    st = S.WsState(T, P, G, S.WS_STRIPED)
    live, seen = list(range(P)), []
    while live:
        c = rnd.choice(live)
        t = st.fetch(c)
        if t < 0:
            live.remove(c)
        else:
            seen.append(t)
    assert sorted(seen) == list(range(T))
    assert all(st.counter[g] > len(st.tiles[g]) for g in range(G))
