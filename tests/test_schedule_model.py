"""The index algebra of the GPU schedules, restated in Python and checked exhaustively on
random shapes (no GPU): the decode kernel's stream-K shares, partial slots and merge
counters (rk_decode_tc.cu), and the prefill planner's chunking of units into items
(rk_plan.cu).  The kernels rely on these invariants -- every tile has exactly one owner,
no two pieces of work share a partial slot or a counter -- so a wrong formula shows up
here as a collision rather than as a silent race on the GPU."""
import numpy as np
import pytest

MERGE_FAN = 12      # kMergeFan
MAX_GRID = 1024     # kDecMaxGrid


SHORT = 8           # kShortTiles


TAPER_STRONG, TAPER_MILD, MAX_TAPER_GRID = (3, 60), (6, 40), 256   # kTaperStrong*, kTaperMild*, kMaxTaperGrid


def taper_setting(max_nt, T, gs):
    """(div, pct): strong when the longest segment spans more CTAs than one merge group."""
    return TAPER_STRONG if max_nt * gs > MERGE_FAN * T else TAPER_MILD


def share_weight(c, gs, L, pct):
    m = max(0, c - (gs - L))
    return 200 * L * c - pct * m * (m + 1)


def taper_count(early, T, gs, div=TAPER_MILD[0], pct=TAPER_MILD[1]):
    """Tapered shares of a call (0: equal shares)."""
    L = gs // div if early and gs <= MAX_TAPER_GRID else 0
    if L == 0:
        return 0
    return L if T * (2 * L * (100 - pct)) >= share_weight(gs, gs, L, pct) else 0


def share_raw(c, T, gs, L, pct=TAPER_MILD[1]):
    if c <= 0:
        return 0
    if c >= gs:
        return T
    return T * share_weight(c, gs, L, pct) // share_weight(gs, gs, L, pct) if L else c * T // gs


def owner(t, T, gs, L=0, pct=TAPER_MILD[1]):
    """The CTA whose share holds tile t of a long segment: closed form for equal shares,
    else the last c whose raw cut is at or before t."""
    if not L:
        return ((t + 1) * gs + T - 1) // T - 1
    return max(c for c in range(gs) if share_raw(c, T, gs, L, pct) <= t)


LATE_SHARES = 8     # kLateShares


def sequence(nt, grid):
    """The single-launch tile sequence: when the short segments fill at most LATE_SHARES
    shares, segments of more than SHORT tiles first, then the others, each class in segment
    order; else segment order.  Returns (order, tile0) -- the segment at each sequence
    position and the first tile of each segment."""
    nt = np.asarray(nt, dtype=np.int64)
    T, TS = int(nt.sum()), int(nt[nt <= SHORT].sum())
    if TS * min(grid, max(T, 1)) <= LATE_SHARES * T:
        order = [s for s in range(len(nt)) if nt[s] > SHORT] + [s for s in range(len(nt)) if nt[s] <= SHORT]
    else:
        order = list(range(len(nt)))
    tile0 = np.zeros(len(nt), np.int64)
    t = 0
    for s in order:
        tile0[s] = t
        t += nt[s]
    return np.array(order), tile0


def short_limit(T, grid):
    """Segments of at most this many tiles are never split: SHORT, or 0 (every tile its own
    CTA) when there are no more tiles than CTAs."""
    return 0 if T <= grid else SHORT


def share_cut(c, T, gs, tile0, nt, order, L=0, short=SHORT, pct=TAPER_MILD[1]):
    """First tile of CTA c's share: its raw cut (c*T/gs, or tapered), moved to the nearer end
    (ties: its start) of the segment it falls in when that segment has at most `short` tiles."""
    if c <= 0:
        return 0
    if c >= gs:
        return T
    raw = share_raw(c, T, gs, L, pct)
    pos = int(np.searchsorted(tile0[order], raw, side="right")) - 1   # last position starting <= raw
    s = int(order[pos])
    t0, n = int(tile0[s]), int(nt[s])
    if raw <= t0 or raw >= t0 + n or n > short:
        return raw
    return t0 if raw - t0 <= t0 + n - raw else t0 + n


def split_slot(c, cta0, c0_later):
    return 2 * c + 1 if (c == cta0 and c0_later) else 2 * c


def decode_schedule(nt, grid, early=False):
    """Per head segment: (tile0, cta0, n_splits, c0_later) as the producer derives them; per
    (segment, CTA) piece of the shares: the slot the producer gives it (2c for the CTA's
    first portion, 2c+1 for a later one).  early: shares tapered as with early start."""
    nt = np.asarray(nt, dtype=np.int64)
    order, tile0 = sequence(nt, grid)
    T = int(nt.sum())
    gs = min(grid, T)
    short = short_limit(T, grid)
    div, pct = taper_setting(int(nt.max()) if len(nt) else 0, T, gs)
    L = taper_count(early, T, gs, div, pct)
    cuts = [share_cut(c, T, gs, tile0, nt, order, L, short, pct) for c in range(gs + 1)]
    segs, pieces = [], {}
    for s, (t0, n) in enumerate(zip(tile0, nt)):
        if n == 0:
            segs.append(None)
            continue
        if n > short:
            c0, c1 = owner(int(t0), T, gs, L, pct), owner(int(t0 + n - 1), T, gs, L, pct)
        else:
            c0 = c1 = -1
        later = int(c1 > c0 and cuts[c0] < t0)
        segs.append((int(t0), c0, c1 - c0 + 1, later))
    for c in range(gs):
        tb, te = cuts[c], cuts[c + 1]
        first = True
        for s in order:                                       # the share's segments in sequence order
            t0, n = tile0[s], nt[s]
            if n == 0 or t0 + n <= tb or t0 >= te:
                continue
            pieces[(s, c)] = 2 * c + (0 if first else 1)
            first = False
    return T, gs, cuts, segs, pieces, (L, pct)


@pytest.mark.parametrize("early", [False, True])
@pytest.mark.parametrize("seed", range(60))
def test_decode_shares_slots_and_counters(seed, early):
    rng = np.random.default_rng(seed)
    grid = int(rng.choice([1, 3, 8, 40, 148]))
    nseg = int(rng.integers(1, 400))
    kind = seed % 5
    if kind == 0:
        nt = rng.integers(0, 6, nseg)                       # short (local) segments, some empty
    elif kind == 1:
        nt = rng.integers(0, 3, nseg); nt[rng.integers(nseg)] = int(rng.integers(200, 1200))   # one long head
    elif kind == 2:
        nt = rng.integers(1, 80, nseg)
    elif kind == 3:
        nt = np.zeros(nseg, np.int64); nt[rng.integers(nseg)] = int(rng.integers(1, 3000))
    else:                                                   # windows of 5 tiles and a few long heads
        nt = np.full(nseg, 5, np.int64); nt[rng.integers(nseg, size=3)] = rng.integers(9, 1100, 3)
    T, gs, cuts, segs, pieces, (L, pct) = decode_schedule(nt, grid, early)
    # the cuts are monotone and the shares tile [0, T)
    assert cuts[0] == 0 and cuts[-1] == T and all(a <= b for a, b in zip(cuts, cuts[1:]))
    _, tile0 = sequence(nt, grid)
    for s, (t0, n) in enumerate(zip(tile0, nt)):
        held = [c for c in range(gs) if n and cuts[c] < t0 + n and cuts[c + 1] > t0]
        if n == 0:
            continue
        if n <= short_limit(T, grid):                       # short segments: one CTA, no split
            assert len(held) == 1 and segs[s][2] == 1
        else:                                               # long ones: the CTAs c*T/gs gives
            t0_, c0, k, _ = segs[s]
            assert held == list(range(c0, c0 + k))
            for t in range(int(t0), int(t0 + n)):
                c = owner(t, T, gs, L, pct)
                assert cuts[c] <= t < cuts[c + 1]
    # slots: the kernel's split_slot formula gives the producer's slot; all distinct, < 2*grid
    split_slots = {}
    for (s, c), slot in pieces.items():
        t0, c0, n, later = segs[s]
        if n > 1:
            assert c0 <= c < c0 + n
            assert split_slot(c, c0, later) == slot
            split_slots[(s, c)] = slot
    assert len(set(split_slots.values())) == len(split_slots)
    assert all(0 <= v < 2 * grid for v in split_slots.values())
    # merge counters: per split segment its first CTA (single level) or the segment
    # counter plus one group counter per MERGE_FAN CTAs (two levels), all distinct
    seg_ctr, grp_ctr = [], []
    for s, rec in enumerate(segs):
        if rec is None or rec[2] == 1:
            continue
        t0, c0, n, later = rec
        seg_ctr.append(c0)
        if n > MERGE_FAN:
            for q in range((n + MERGE_FAN - 1) // MERGE_FAN):
                grp_ctr.append(split_slot(c0 + q * MERGE_FAN, c0, later))
    assert len(set(seg_ctr)) == len(seg_ctr) and all(c < MAX_GRID for c in seg_ctr)
    assert len(set(grp_ctr)) == len(grp_ctr) and all(g < 2 * MAX_GRID for g in grp_ctr)
    # the pieces of a split segment are exactly its CTAs' slots
    for s, rec in enumerate(segs):
        if rec is not None and rec[2] > 1:
            t0, c0, n, later = rec
            assert sorted(v for (ss, c), v in split_slots.items() if ss == s) == \
                sorted(split_slot(c, c0, later) for c in range(c0, c0 + n))


def test_long_segments_come_first_so_the_last_ctas_hold_only_windows():
    # a 128K-stack layer with a global head: 1024 tiles of it and seven 5-tile windows over
    # 148 CTAs; the CTAs dispatched last take windows, never a piece of the global head
    nt = [5] * 8
    nt[3] = 1024
    T, gs, cuts, segs, pieces, _ = decode_schedule(nt, 148)
    order, tile0 = sequence(nt, 148)
    assert list(order[:1]) == [3] and tile0[3] == 0
    last = [c for (s, c) in pieces if s != 3]
    assert min(last) > max(c for (s, c) in pieces if s == 3) - 1 and max(last) == gs - 1


def test_many_windows_keep_segment_order():
    # the decode microbenchmark: 32 global heads of 64 tiles and 224 windows of 3 -- the
    # windows would fill 36 shares, so the sequence stays in segment order
    nt = np.tile([64] + [3] * 7, 32)
    order, tile0 = sequence(nt, 148)
    assert list(order) == list(range(len(nt)))


def test_windows_spread_one_tile_per_cta_on_a_local_only_layer():
    # eight local heads of five key tiles each over 148 CTAs: 40 tiles, no more than CTAs, so
    # every tile gets its own CTA and each window is merged from five pieces
    T, gs, cuts, segs, pieces, _ = decode_schedule([5] * 8, 148)
    assert gs == 40 and all(cuts[c + 1] - cuts[c] == 1 for c in range(gs))
    assert all(rec[2] == 5 for rec in segs)
    # more tiles than CTAs: windows stay whole
    T, gs, cuts, segs, pieces, _ = decode_schedule([5] * 40, 148)
    assert all(rec[2] == 1 for rec in segs)


def prefill_plan(n_vis, chunk):
    """Items as the planner emits them, in item order: full chunks, a remainder that joins the
    last full chunk when it is at most half a chunk; the units in three classes -- single
    items of at least a chunk, then the units of several items (unit order, each unit's items
    consecutive), then single items shorter than a chunk.  Also returns each unit's first
    item (the kernel's unit_item(u, s) = first_item + s) and the split-unit list."""
    per_unit, cls = [], []
    for u, nv in enumerate(n_vis):
        r, nf = nv % chunk, nv // chunk
        rm = 1 if (nv == 0 or (r != 0 and (nf == 0 or 2 * r > chunk))) else 0
        ns = nf + rm
        per_unit.append([(u, s * chunk, nv if s == ns - 1 else (s + 1) * chunk) for s in range(ns)])
        cls.append(1 if ns > 1 else 0 if nf >= 1 else 2)
    items, first = [], [0] * len(n_vis)
    for c in (0, 1, 2):
        for u in range(len(n_vis)):
            if cls[u] == c:
                first[u] = len(items)
                items += per_unit[u]
    return items, first, [u for u in range(len(n_vis)) if cls[u] == 1]


def prefill_items(n_vis, chunk):
    return prefill_plan(n_vis, chunk)[0]


@pytest.mark.parametrize("seed", range(20))
def test_prefill_items_cover_each_unit_once(seed):
    rng = np.random.default_rng(100 + seed)
    chunk = int(rng.choice([8, 16, 32, 112, 912]))
    n_vis = rng.integers(0, 4 * chunk, int(rng.integers(1, 300)))
    items = prefill_items(n_vis, chunk)
    for u, nv in enumerate(n_vis):
        mine = sorted((b, e) for (uu, b, e) in items if uu == u)
        assert mine, "every unit has at least one item (an empty one writes its zero output)"
        assert mine[0][0] == 0 and mine[-1][1] == nv
        assert all(a[1] == b[0] for a, b in zip(mine, mine[1:]))          # contiguous, no overlap
        assert all(e - b <= chunk + chunk // 2 for b, e in mine)         # merged remainder at most 1.5 chunks
        if len(mine) > 1:
            assert all(e - b >= chunk // 2 for b, e in mine)             # no slivers
    # the kernel finds split s of unit u at first_item + s; split units are listed in the
    # order their items are handed out, and come after the long single items
    items, first, split = prefill_plan(n_vis, chunk)
    for u, nv in enumerate(n_vis):
        mine = [i for i, it in enumerate(items) if it[0] == u]
        assert mine == list(range(first[u], first[u] + len(mine)))
        assert (len(mine) > 1) == (u in split)
    assert [first[u] for u in split] == sorted(first[u] for u in split)
    singles_long = [u for u in range(len(n_vis)) if u not in split and n_vis[u] >= chunk]
    assert all(first[a] < first[b] for a in singles_long for b in split)


def test_tapered_shares_shrink_towards_the_last_cta():
    # the decode microbenchmark's 2720 tiles over 148 CTAs with early start: its long
    # segments span ~3.5 CTAs, so the mild taper -- the first 124 shares equal, the last 24
    # shrinking step by step to 60 % of a full share
    nt = np.tile([64] + [3] * 7, 32)
    T, gs, cuts, segs, pieces, (L, pct) = decode_schedule(nt, 148, early=True)
    assert (L, pct) == (24, 40)
    raw = [share_raw(c, T, gs, L, pct) for c in range(gs + 1)]
    w = np.diff(raw)
    full = T * 200 * L / share_weight(gs, gs, L, pct)
    assert abs(w[:gs - L].mean() - full) < 1 and abs(w[-1] - 0.6 * full) <= 1
    assert all(w[i] >= w[i + 1] - 1 for i in range(gs - L - 1, gs - 1))
    assert sum(w) == T and min(w) >= 1
    # a 128K-stack layer with a global head spans ~143 CTAs: the strong taper, the last 49
    # shares down to 40 %
    nt = [5] * 8
    nt[3] = 1032
    T, gs, cuts, segs, pieces, (L, pct) = decode_schedule(nt, 148, early=True)
    assert (L, pct) == (49, 60)
    # no taper without early start, or when a share would hold less than a tile
    assert taper_count(False, T, gs) == 0 and taper_count(True, 150, 148) == 0


def simulate_prefill_merges(n_vis, chunk, grid, rng):
    """Discrete-event model of the prefill kernel's merge protocol: per CTA a producer takes
    items (its blockIdx first, then tickets from a counter), its softmax warps finish them in
    order and count them on their unit; a background worker (warps 10-11) claims the next
    merge job only while items remain and only when that job's unit is complete (a
    compare-and-swap on the job counter); once a CTA's items are done its softmax warps claim
    jobs outright and wait for the unit.  Returns the merge log [(job, unit, time,
    worker kind)] and the time every unit completed."""
    items, first, split = prefill_plan(n_vis, chunk)
    rb = 32                                        # jobs per split unit (256 rows / 8)
    n_jobs = len(split) * rb
    ns = {u: 0 for u in range(len(n_vis))}
    for (u, _, _) in items:
        ns[u] += 1
    done = {u: 0 for u in range(len(n_vis))}
    complete_at = {}
    counter = 0                                    # item tickets taken
    job_counter = 0
    log = []
    # per CTA: queue of (finish time) items; time advances in events
    t = 0.0
    cta_items = {c: [] for c in range(grid)}
    busy_until = {c: 0.0 for c in range(grid)}
    next_item = {c: (c if c < len(items) else None) for c in range(grid)}
    fast_state = {c: None for c in range(grid)}    # job a CTA's softmax warps wait on
    bg_free_at = {c: 0.0 for c in range(grid)}
    finished = {c: False for c in range(grid)}
    for _ in range(100000):
        progressed = False
        for c in range(grid):
            # producer + softmax: process the next item when free
            if next_item[c] is not None and busy_until[c] <= t:
                it = next_item[c]
                u = items[it][0]
                dur = 1.0 + (items[it][2] - items[it][1]) * rng.uniform(0.8, 1.2) / max(chunk, 1)
                busy_until[c] = t + dur
                cta_items[c].append((t + dur, u))
                tk = counter
                counter += 1
                nxt = grid + tk
                next_item[c] = nxt if nxt < len(items) else None
                progressed = True
            # completions
            for (ft, u) in list(cta_items[c]):
                if ft <= t:
                    cta_items[c].remove((ft, u))
                    done[u] += 1
                    if done[u] == ns[u]:
                        complete_at[u] = ft
                    progressed = True
            items_left = counter + grid < len(items)
            # background worker: claims only completed units while items remain
            if bg_free_at[c] <= t and items_left and job_counter < n_jobs:
                u = split[job_counter // rb]
                if done[u] == ns[u]:
                    log.append((job_counter, u, t, "bg"))
                    job_counter += 1
                    bg_free_at[c] = t + 0.3
                    progressed = True
            # softmax warps after their items: claim outright, wait for the unit
            if next_item[c] is None and not cta_items[c] and busy_until[c] <= t and not finished[c]:
                if fast_state[c] is None:
                    if job_counter >= n_jobs:
                        finished[c] = True
                    else:
                        fast_state[c] = job_counter
                        job_counter += 1
                    progressed = True
                else:
                    j = fast_state[c]
                    u = split[j // rb]
                    if done[u] == ns[u]:
                        log.append((j, u, t, "tail"))
                        fast_state[c] = None
                        busy_until[c] = t + 0.1
                        progressed = True
        if all(finished.values()):
            return log, complete_at, n_jobs
        if not progressed:
            t += 0.05
    raise AssertionError("the merge protocol did not terminate")


@pytest.mark.parametrize("seed", range(12))
def test_prefill_merge_jobs_run_once_each_after_their_unit(seed):
    rng = np.random.default_rng(500 + seed)
    chunk = int(rng.choice([12, 24, 96]))
    grid = int(rng.choice([4, 16, 40]))
    n_vis = np.concatenate([rng.integers(1, chunk, int(rng.integers(5, 60))),          # short singles
                            rng.integers(2 * chunk, 8 * chunk, int(rng.integers(1, 8)))])  # split units
    rng.shuffle(n_vis)
    log, complete_at, n_jobs = simulate_prefill_merges(n_vis, chunk, grid, rng)
    jobs = [j for (j, _, _, _) in log]
    assert sorted(jobs) == list(range(n_jobs))                       # every job, once
    for (j, u, t, kind) in log:
        assert t >= complete_at[u]                                   # only after its unit completed
