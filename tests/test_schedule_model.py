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


def owner(t, T, gs):
    return ((t + 1) * gs + T - 1) // T - 1


def split_slot(c, cta0, tile0, T, gs):
    return 2 * c + 1 if (c == cta0 and c * T // gs < tile0) else 2 * c


def decode_schedule(nt, grid):
    """Per head segment: (tile0, cta0, n_splits); per (segment, CTA) piece: the slot the
    producer gives it (2c for the CTA's first portion, 2c+1 for a later one)."""
    nt = np.asarray(nt, dtype=np.int64)
    tile0 = np.concatenate([[0], np.cumsum(nt)[:-1]])
    T = int(nt.sum())
    gs = min(grid, T)
    segs, pieces = [], {}
    for s, (t0, n) in enumerate(zip(tile0, nt)):
        if n == 0:
            segs.append(None)
            continue
        c0, c1 = owner(int(t0), T, gs), owner(int(t0 + n - 1), T, gs)
        segs.append((int(t0), c0, c1 - c0 + 1))
    for c in range(gs):
        tb, te = c * T // gs, (c + 1) * T // gs
        first = True
        for s, (t0, n) in enumerate(zip(tile0, nt)):
            if n == 0 or t0 + n <= tb or t0 >= te:
                continue
            pieces[(s, c)] = 2 * c + (0 if first else 1)
            first = False
    return T, gs, segs, pieces


@pytest.mark.parametrize("seed", range(40))
def test_decode_shares_slots_and_counters(seed):
    rng = np.random.default_rng(seed)
    grid = int(rng.choice([1, 3, 8, 148]))
    nseg = int(rng.integers(1, 400))
    kind = seed % 4
    if kind == 0:
        nt = rng.integers(0, 6, nseg)                       # short (local) segments, some empty
    elif kind == 1:
        nt = rng.integers(0, 3, nseg); nt[rng.integers(nseg)] = int(rng.integers(200, 1200))   # one long head
    elif kind == 2:
        nt = rng.integers(1, 80, nseg)
    else:
        nt = np.zeros(nseg, np.int64); nt[rng.integers(nseg)] = int(rng.integers(1, 3000))
    T, gs, segs, pieces = decode_schedule(nt, grid)
    # every tile has exactly one owner and the shares tile [0, T)
    owners = [owner(t, T, gs) for t in range(T)]
    for c in range(gs):
        tb, te = c * T // gs, (c + 1) * T // gs
        assert te > tb and all(owners[t] == c for t in range(tb, te))
    # slots: the kernel's split_slot formula gives the producer's slot; all distinct, < 2*grid
    split_slots = {}
    for (s, c), slot in pieces.items():
        t0, c0, n = segs[s]
        assert c0 <= c < c0 + n
        if n > 1:
            assert split_slot(c, c0, t0, T, gs) == slot
            split_slots[(s, c)] = slot
    assert len(set(split_slots.values())) == len(split_slots)
    assert all(0 <= v < 2 * grid for v in split_slots.values())
    # merge counters: per split segment its first CTA (single level) or the segment
    # counter plus one group counter per MERGE_FAN CTAs (two levels), all distinct
    seg_ctr, grp_ctr = [], []
    for s, rec in enumerate(segs):
        if rec is None or rec[2] == 1:
            continue
        t0, c0, n = rec
        seg_ctr.append(c0)
        if n > MERGE_FAN:
            for q in range((n + MERGE_FAN - 1) // MERGE_FAN):
                grp_ctr.append(split_slot(c0 + q * MERGE_FAN, c0, t0, T, gs))
    assert len(set(seg_ctr)) == len(seg_ctr) and all(c < MAX_GRID for c in seg_ctr)
    assert len(set(grp_ctr)) == len(grp_ctr) and all(g < 2 * MAX_GRID for g in grp_ctr)
    # the pieces of a split segment are exactly its CTAs' slots
    for s, rec in enumerate(segs):
        if rec is not None and rec[2] > 1:
            t0, c0, n = rec
            assert sorted(v for (ss, c), v in split_slots.items() if ss == s) == \
                sorted(split_slot(c, c0, t0, T, gs) for c in range(c0, c0 + n))


def prefill_items(n_vis, chunk):
    """Items of each unit as the planner emits them: full chunks, and a remainder that
    joins the last full chunk when it is at most half a chunk."""
    items = []
    for u, nv in enumerate(n_vis):
        r, nf = nv % chunk, nv // chunk
        rm = 1 if (nv == 0 or (r != 0 and (nf == 0 or 2 * r > chunk))) else 0
        ns = nf + rm
        for s in range(ns):
            items.append((u, s * chunk, nv if s == ns - 1 else (s + 1) * chunk))
    return items


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
