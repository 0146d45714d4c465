"""Pins of the fp64 oracle against facts that do not come from the oracle itself:
worked examples printed on the pages (tests/golden), closed forms, special cases
that reduce to library routines, and invariants stated by the pages."""
import dataclasses
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import rk_oracle as O
from workloads import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------ bf16 rounding
def test_bf16_rounding_matches_torch_on_float32_values():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * s for s in (1e-3, 1.0, 1e3)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.f64_to_bf16(x.astype(np.float64)), ref)


def test_bf16_rounding_ties_and_no_double_rounding():
    one = 0x3F80
    assert O.f64_to_bf16(np.array([1 + 2.0 ** -8]))[0] == one                     # tie -> even (1.0)
    assert O.f64_to_bf16(np.array([1 + 3 * 2.0 ** -8]))[0] == one + 2             # tie -> even (1+2^-6)
    # just above a tie: float32 would round it onto the tie first and then to 1.0
    assert O.f64_to_bf16(np.array([1 + 2.0 ** -8 + 2.0 ** -30]))[0] == one + 1
    assert O.f64_to_bf16(np.array([-2.5]))[0] == 0xC020
    assert np.array_equal(O.bf16_to_f64(np.array([0x3F80, 0xC020], np.uint16)), [1.0, -2.5])


def test_bf16_ordinal_is_ulp_distance():
    b = np.array([0x3F80, 0x3F81, 0x0000, 0x8000, 0x8001, 0x0001], np.uint16)
    o = O.bf16_ordinal(b)
    assert o[1] - o[0] == 1 and o[2] == o[3] == 0 and o[5] - o[4] == 2


# ------------------------------------------------------------------ RoPE
@pytest.mark.parametrize("case", _load("rope_unit_vectors.json")["cases"])
def test_rope_unit_vectors(case):
    g = _load("rope_unit_vectors.json")
    style = O.ROPE_HALF_SPLIT if case["style"] == "half_split" else O.ROPE_INTERLEAVED
    y = O.rope_rotate(np.array([case["x"]], float), np.array([case["pos"]]), g["theta"], style)
    assert np.allclose(y[0], case["y"], atol=1e-15)


@pytest.mark.parametrize("style", [O.ROPE_HALF_SPLIT, O.ROPE_INTERLEAVED])
def test_rope_equals_complex_multiplication(style):
    # the same rotation written as multiplication by e^{i*angle} of the complex pair (a + i b)
    rng = np.random.default_rng(1)
    d, theta = 128, 1e6
    x = rng.standard_normal((64, d))
    pos = rng.integers(0, 200000, 64)
    a, b = O.rope_pairs(d, style)
    z = (x[:, a] + 1j * x[:, b]) * np.exp(1j * pos[:, None] * theta ** (-np.arange(0, d, 2) / d))
    y = O.rope_rotate(x, pos, theta, style)
    assert np.allclose(y[:, a], z.real, atol=1e-9) and np.allclose(y[:, b], z.imag, atol=1e-9)


def test_rope_composition_closed_form():
    # R(p2) R(p1)^-1 = R(p2 - p1), identity at equal positions, pair norms preserved
    rng = np.random.default_rng(2)
    d, theta = 128, 1e6
    x = rng.standard_normal((256, d))
    p1 = rng.integers(0, 5000, 256)
    p2 = p1 + rng.integers(0, 30000, 256)
    y = O.rope_reposition(x, p1, p2, theta)
    assert np.allclose(y, O.rope_rotate(x, p2 - p1, theta), atol=1e-10)
    assert np.allclose(O.rope_reposition(x, p1, p1, theta), x, atol=1e-12)
    a, b = O.rope_pairs(d, 0)
    assert np.allclose(y[:, a] ** 2 + y[:, b] ** 2, x[:, a] ** 2 + x[:, b] ** 2, atol=1e-10)


def test_reposition_removes_position_offset_error():
    """K cached at offline positions and repositioned to online positions equals K rotated
    at the online positions directly, so attention scores only see relative positions."""
    rng = np.random.default_rng(3)
    d, theta = 64, 1e4
    k_raw = rng.standard_normal((300, d))
    q_raw = rng.standard_normal((5, d))
    p_off = np.arange(300)
    p_on = 7000 + np.arange(300)
    cached = O.rope_rotate(k_raw, p_off, theta)
    moved = O.rope_reposition(cached, p_off, p_on, theta)
    direct = O.rope_rotate(k_raw, p_on, theta)
    assert np.allclose(moved, direct, atol=1e-10)
    qpos = np.array([7300, 7301, 7302, 7303, 7304])
    q = O.rope_rotate(q_raw, qpos, theta)
    # <R(a) q, R(b) k> = <q, R(b - a) k>
    lhs = q @ moved.T
    rhs = np.stack([q_raw[i] @ O.rope_rotate(k_raw, p_on - qpos[i], theta).T for i in range(5)])
    assert np.allclose(lhs, rhs, atol=1e-9)


def test_paged_rope_reposition_follows_tables():
    w = synth.tiny_prefill()
    r = w.rope
    pages, slots, rows = O.paged_rope_reposition(r.k_src, r.src_tables, r.dst_tables, r.runs, w.theta, r.P)
    assert len(pages) == r.total_tok
    # every destination row is written once
    assert len(set(zip(pages.tolist(), slots.tolist()))) == len(pages)
    # the run with delta 0 (segment 0 stays at 0..255) gives back its source rows: to fp64
    # rounding of the two rotations, and exactly once stored as bf16
    run = r.runs[0]
    assert run[4] == run[5] == 0
    src_bits = r.k_src[r.src_tables[run[0] + np.arange(256) // 16], np.arange(256) % 16]
    assert np.allclose(rows[:256], O.bf16_to_f64(src_bits), rtol=0, atol=1e-12)
    assert np.array_equal(O.f64_to_bf16(rows[:256]), src_bits)


# ------------------------------------------------------------------ page tables / visibility
def test_vllm_worked_example_block_table():
    g = _load("vllm_block_table.json")
    for tok in g["tokens"]:
        assert O.token_to_physical(g["block_table"], g["block_size"], tok["t"]) == (tok["physical"], tok["slot"])
    used = set(g["block_table"])
    assert sorted(set(range(g["n_physical_blocks"])) - used) == g["free_blocks"]


@pytest.mark.parametrize("case", _load("visibility_cases.json")["cases"], ids=lambda c: c["name"])
def test_visibility_hand_cases(case):
    listed = O.listed_positions(np.array(case["listed_pages"]), len(case["listed_pages"]), case["P"])
    got = O.visible_set(case["cls"], case["W"], case["S"], case["seq_len"], case["p"], listed)
    assert got.tolist() == case["visible"]


def _small_batch(cls_row, window_row, seed=7, P=16, ctx=300, suffix=37, Hq=4, Hkv=2, d=32):
    rng = np.random.default_rng(seed)
    return synth._build("t", rng, B=1, Hq=Hq, Hkv=Hkv, d=d, P=P, theta=1e4, ctx_len=[ctx],
                        n_suffix=[suffix], classes=[cls_row], windows=[window_row],
                        sinks=[[0] * Hkv], seg_tokens=[128]).attn


def _outs(batch):
    return O.segpaged_attention(batch)


def test_local_with_huge_window_equals_global():
    a = _small_batch([O.GLOBAL, O.LOCAL], [0, 10 ** 6])
    res = _outs(a)
    b = dataclasses.replace(a, head_class=np.array([O.GLOBAL, O.GLOBAL], np.int32))
    res2 = _outs(b)
    for key in res:
        assert np.array_equal(res[key][0], res2[key][0])


def test_retrieval_with_full_list_equals_global():
    a = _small_batch([O.RETRIEVAL, O.GLOBAL], [0, 0])
    res = _outs(a)
    b = dataclasses.replace(a, head_class=np.array([O.GLOBAL, O.GLOBAL], np.int32))
    for key, v in _outs(b).items():
        assert np.array_equal(res[key][0], v[0])


def test_physical_page_permutation_invariance():
    a = _small_batch([O.GLOBAL, O.LOCAL], [0, 40])
    res = _outs(a)
    rng = np.random.default_rng(11)
    n = a.k_pool.shape[0]
    perm = rng.permutation(n)                       # new position of each old page
    inv = np.empty(n, np.int64)
    inv[perm] = np.arange(n)
    k2 = a.k_pool[inv]
    v2 = a.v_pool[inv]
    tab2 = np.where(a.page_table >= 0, perm[np.maximum(a.page_table, 0)], -1).astype(np.int32)
    b = dataclasses.replace(a, k_pool=k2, v_pool=v2, page_table=tab2)
    for key, v in _outs(b).items():
        assert np.array_equal(res[key][0], v[0]) and np.array_equal(res[key][1], v[1])


# ------------------------------------------------------------------ attention
def test_single_visible_key_returns_its_value():
    rng = np.random.default_rng(4)
    q, k, v = rng.standard_normal((3, 16)), rng.standard_normal((1, 16)), rng.standard_normal((1, 16))
    o, lse = O.softmax_attention(q, k, v, 0.25)
    assert np.allclose(o, np.repeat(v, 3, 0), atol=1e-15)
    assert np.allclose(lse, (q @ k.T)[:, 0] * 0.25, atol=1e-15)


def test_identical_keys_give_mean_of_values():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((4, 8))
    k = np.repeat(rng.standard_normal((1, 8)), 10, 0)
    v = rng.standard_normal((10, 8))
    o, lse = O.softmax_attention(q, k, v, 1.0)
    assert np.allclose(o, np.repeat(v.mean(0, keepdims=True), 4, 0), atol=1e-14)
    assert np.allclose(lse, (q @ k[:1].T)[:, 0] + math.log(10), atol=1e-13)


def test_zero_query_gives_mean_of_values():
    rng = np.random.default_rng(6)
    k, v = rng.standard_normal((50, 8)), rng.standard_normal((50, 8))
    o, _ = O.softmax_attention(np.zeros((2, 8)), k, v, 0.3)
    assert np.allclose(o, np.repeat(v.mean(0, keepdims=True), 2, 0), atol=1e-14)


def test_two_scalar_keys_logistic_closed_form():
    # d = 1, two keys: weight of key 0 is the logistic function of the score difference
    q, k, v = np.array([[1.5]]), np.array([[2.0], [-1.0]]), np.array([[3.0], [5.0]])
    o, lse = O.softmax_attention(q, k, v, 1.0)
    w0 = 1.0 / (1.0 + math.exp(-(3.0 - (-1.5))))
    assert abs(o[0, 0] - (w0 * 3.0 + (1 - w0) * 5.0)) < 1e-15
    assert abs(lse[0] - math.log(math.exp(3.0) + math.exp(-1.5))) < 1e-15


def test_segpaged_attention_matches_torch_sdpa_with_mask():
    """Library cross-check: torch's scaled_dot_product_attention in float64 with an explicit
    boolean mask (the masked path the pages say SegPagedAttention avoids) on the same keys."""
    a = _small_batch([O.GLOBAL, O.LOCAL], [0, 50], suffix=41)
    res = _outs(a)
    G = a.Hq // a.Hkv
    L = int(a.seq_len[0])
    nq = a.total_q
    for h in range(a.Hkv):
        seg = h
        pos = np.arange(L)
        k = O.gather_rows(a.k_pool, a.page_table[seg], a.page_logical[seg], int(a.n_pages[seg]), a.P, pos)
        v = O.gather_rows(a.v_pool, a.page_table[seg], a.page_logical[seg], int(a.n_pages[seg]), a.P, pos)
        qpos = L - nq + np.arange(nq)
        mask = pos[None, :] <= qpos[:, None]
        if a.head_class[seg] == O.LOCAL:
            mask &= pos[None, :] > qpos[:, None] - a.window[seg]
        q = O.bf16_to_f64(a.q[:, h * G:(h + 1) * G])                       # [nq, G, d]
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q).permute(1, 0, 2), torch.from_numpy(k)[None].expand(G, -1, -1),
            torch.from_numpy(v)[None].expand(G, -1, -1), attn_mask=torch.from_numpy(mask)[None],
            scale=1.0 / math.sqrt(a.d)).permute(1, 0, 2).numpy()
        for t in range(nq):
            assert np.allclose(res[(t, h)][0], ref[t], atol=1e-12)


def test_split_combine_equals_unsplit():
    rng = np.random.default_rng(8)
    q, k, v = rng.standard_normal((4, 32)), rng.standard_normal((1000, 32)), rng.standard_normal((1000, 32))
    o, lse = O.softmax_attention(q, k, v, 0.2)
    for bounds in ([0, 1000], [0, 1, 999, 1000], [0, 300, 300, 650, 1000]):
        oc, lc = O.combine_partials(O.split_partials(q, k, v, 0.2, bounds))
        assert np.allclose(oc, o, atol=1e-13) and np.allclose(lc, lse, atol=1e-12)


def test_attention_flops_tiny_hand_count():
    # queries at 512..543; global head sees p+1 keys, local head (W=64) sees 64; 2 q heads per KV head
    pairs = sum(p + 1 for p in range(512, 544)) + 32 * 64
    assert O.attention_flops(synth.tiny_prefill().attn) == 4 * 64 * 2 * pairs == 9707520


def test_rope_tolerance_floor_only_covers_fp64_roundoff():
    # an exact zero kept at zero passes although the fp64 two-step value is ~1e-17
    x = np.zeros((1, 4))
    x[0, 0] = 1.0
    exact = np.array([[1.0, 0.0, 1.4e-17, 0.0]])
    got = np.array([[0x3F80, 0, 0, 0]], np.uint16)
    assert O.rope_within_one_ulp(got, exact, x, O.ROPE_HALF_SPLIT).all()
    # a real error of 2 ulps is still caught
    got2 = np.array([[0x3F82, 0, 0, 0]], np.uint16)
    assert not O.rope_within_one_ulp(got2, exact, x, O.ROPE_HALF_SPLIT)[0, 0]
    # and so is a small absolute error well above the fp64 round-off
    got3 = np.array([[0x3F80, 0, 0x2F00, 0]], np.uint16)      # 1.2e-10 where 1.4e-17 is exact
    assert not O.rope_within_one_ulp(got3, exact, x, O.ROPE_HALF_SPLIT)[0, 2]


# ------------------------------------------------------------------ sparse page lists
def test_gather_rows_on_a_sparse_list_follows_the_block_table():
    """The worked block table of "PagedAttention & RadixAttention" (block size 4; logical
    blocks 0, 1, 2 in physical blocks 7, 1, 3) with logical block 1 dropped from the list,
    as a retrieval head or a window-only local head lists its pages: entry e of the list
    holds logical page [0, 2][e] in physical page [7, 3][e].  gather_rows must return, for
    every position of a listed page, the row token_to_physical gives on the full table --
    not the row of entry position // P (which would be logical block 1's page or past the
    list)."""
    g = _load("vllm_block_table.json")
    P, full = g["block_size"], g["block_table"]
    rng = np.random.default_rng(12)
    pool = rng.integers(0, 2 ** 15, size=(g["n_physical_blocks"], P, 3)).astype(np.uint16)
    listed_logical = np.array([0, 2], np.int32)
    table_row = np.array([full[0], full[2]], np.int32)          # [7, 3]
    positions = np.array([0, 1, 2, 3, 8], np.int64)               # the tokens of logical blocks 0 and 2
    got = O.gather_rows(pool, table_row, listed_logical, 2, P, positions)
    for i, t in enumerate(positions):
        phys, slot = O.token_to_physical(full, P, int(t))
        assert np.array_equal(got[i], O.bf16_to_f64(pool[phys, slot]))
    assert O.listed_positions(listed_logical, 2, P).tolist() == [0, 1, 2, 3, 8, 9, 10, 11]
    with pytest.raises(KeyError):                                # position 5 is on an unlisted page
        O.gather_rows(pool, table_row, listed_logical, 2, P, np.array([5]))


def test_retrieval_head_on_a_sparse_list_equals_hand_indexed_attention():
    """A retrieval head listing logical pages 0, 2 and 5 (of 6) in hand-picked physical
    pages: its output equals softmax attention over the keys read straight from the pool
    at (physical page of the listed logical page, slot), enumerated here by hand from the
    page size and the causal bound -- no table lookup shared with the oracle."""
    P, d, Hq, Hkv = 4, 8, 2, 1
    rng = np.random.default_rng(13)
    n_pool = 9
    k_pool = synth.f32_to_bf16_bits(rng.standard_normal((n_pool, P, d)).astype(np.float32))
    v_pool = synth.f32_to_bf16_bits(rng.standard_normal((n_pool, P, d)).astype(np.float32))
    q = synth.f32_to_bf16_bits(rng.standard_normal((2, Hq, d)).astype(np.float32))
    # logical page 0 -> physical 6, logical 2 -> physical 1, logical 5 -> physical 4
    table = np.array([[6, 1, 4, -1]], np.int32)
    logical = np.array([[0, 2, 5, -1]], np.int32)
    batch = synth.AttnBatch(B=1, Hq=Hq, Hkv=Hkv, d=d, P=P, q=q, cu_seqlens_q=np.array([0, 2], np.int32),
                            seq_len=np.array([23], np.int32), k_pool=k_pool, v_pool=v_pool, page_table=table,
                            page_logical=logical, n_pages=np.array([3], np.int32),
                            head_class=np.array([O.RETRIEVAL], np.int32), window=np.array([0], np.int32),
                            sink=np.array([0], np.int32))
    res = O.segpaged_attention(batch)
    # query 0 at position 21, query 1 at 22: listed positions 0-3, 8-11 and 20-23, causal
    by_hand = {21: [(6, 0), (6, 1), (6, 2), (6, 3), (1, 0), (1, 1), (1, 2), (1, 3), (4, 0), (4, 1)],
               22: [(6, 0), (6, 1), (6, 2), (6, 3), (1, 0), (1, 1), (1, 2), (1, 3), (4, 0), (4, 1), (4, 2)]}
    for t, p in ((0, 21), (1, 22)):
        rows = by_hand[p]
        kk = np.stack([O.bf16_to_f64(k_pool[pg, s]) for pg, s in rows])
        vv = np.stack([O.bf16_to_f64(v_pool[pg, s]) for pg, s in rows])
        qq = O.bf16_to_f64(q[t])
        s = qq @ kk.T / math.sqrt(d)
        w = np.exp(s - s.max(axis=1, keepdims=True))
        o = (w @ vv) / w.sum(axis=1, keepdims=True)
        got_o, got_l = res[(t, 0)]
        assert np.allclose(got_o, o, atol=1e-13)
        assert np.allclose(got_l, np.log(np.exp(s).sum(axis=1)), atol=1e-12)


# ------------------------------------------------------------------ decode storage
def test_append_rows_follows_the_worked_block_table():
    """The generated tokens of the worked example ("fathers" at t = 7, "brought" at t = 8)
    land in the physical block and slot the example prints."""
    g = _load("vllm_block_table.json")
    P = g["block_size"]
    tab = np.array([g["block_table"]], np.int32)
    lg = np.arange(3, dtype=np.int32)[None]
    k = np.zeros((g["n_physical_blocks"], P, 2), np.uint16)
    for tok in g["tokens"][7:]:
        new = np.array([[[1000 + tok["t"], 7]]], np.uint16)
        k2, v2 = O.append_rows(k, k, tab, lg, np.array([3]), np.array([tok["t"]]), new, new, 1, P)
        assert np.array_equal(k2[tok["physical"], tok["slot"]], new[0, 0])
        assert np.count_nonzero(k2 != k) == 2                    # that row, nothing else


def test_ring_advance_worked_example():
    g = _load("page_ring.json")
    P, W, S, R = g["P"], g["W"], g["S"], g["R"]
    tab = np.array([g["initial"]["physical"]], np.int32)
    lg = np.array([g["initial"]["logical"]], np.int32)
    n = np.array([len(g["initial"]["logical"])], np.int32)
    k = np.zeros((8, P, 1), np.uint16)
    for step in g["after"]:
        tab, lg = O.ring_advance(tab, lg, n, np.array([R]), np.array([W]), np.array([S]), np.array([step["pos"]]), 1, P)
        assert lg[0].tolist() == step["logical"] and tab[0].tolist() == step["physical"]
        new = np.array([[[step["pos"]]]], np.uint16)
        k, _ = O.append_rows(k, k, tab, lg, n, np.array([step["pos"]]), new, new, 1, P)
        assert k[step["slot"][0], step["slot"][1], 0] == step["pos"]


def test_ring_keeps_every_window_visible_over_a_long_decode():
    """Invariants over 3000 appended tokens for several (P, W, S): the list stays ascending,
    holds the same physical pages (the ring reuses only its own), and lists every position
    of the newest token's window and of the sink; each appended token stays readable until
    it leaves the window."""
    for P, W, S in ((16, 512, 0), (16, 256, 4), (32, 100, 0), (4, 6, 2), (16, 16, 0), (16, 1, 0)):
        R = -(-W // P) + 1
        start = 4 * P + 8 * W                                   # the first decode position
        sink_pages = list(range(-(-S // P)))
        hi = start // P + (start % P != 0)                      # one past the page holding start - 1
        win_pages = list(range(hi - R, hi))
        lg = np.array([sink_pages + win_pages], np.int32)
        tab = np.arange(lg.shape[1], dtype=np.int32)[None] + 40
        n = np.array([lg.shape[1]], np.int32)
        phys0 = set(tab[0].tolist())
        written = {}
        k = np.zeros((40 + lg.shape[1], P, 1), np.uint16)
        for pos in range(start, start + 3000):
            tab, lg = O.ring_advance(tab, lg, n, np.array([R]), np.array([W]), np.array([S]), np.array([pos]), 1, P)
            assert np.all(np.diff(lg[0]) > 0) and set(tab[0].tolist()) == phys0
            new = np.array([[[pos % 60000]]], np.uint16)
            k, _ = O.append_rows(k, k, tab, lg, n, np.array([pos]), new, new, 1, P)
            written[pos] = pos % 60000
            listed = set(O.listed_positions(lg[0], int(n[0]), P).tolist())
            vis = O.visible_set(O.LOCAL, W, S, pos + 1, pos, np.array(sorted(listed)))
            want = [j for j in range(pos + 1) if j > pos - W or j < S]
            assert vis.tolist() == want
            for j in range(max(0, pos - W + 1), pos + 1):       # appended tokens still in the window
                if j in written:
                    e = int(np.searchsorted(lg[0], j // P))
                    assert k[tab[0, e], j % P, 0] == written[j]


# ------------------------------------------------------------------ sparse FFN
@pytest.mark.parametrize("case", _load("token_selection.json")["cases"])
def test_token_selection_hand_cases(case):
    imp = np.array([float(v) for v in case["importance"]], dtype=np.float32)
    assert O.select_tokens(imp, case["keep"]).tolist() == case["kept"]


def test_token_selection_brute_force():
    # against every subset of the right size: the chosen one has the largest sorted scores,
    # and among equal ones the lexicographically smallest index set
    import itertools
    rng = np.random.default_rng(21)
    for _ in range(200):
        T = int(rng.integers(1, 8))
        imp = rng.integers(0, 4, T).astype(np.float32)          # many ties
        keep = int(rng.integers(0, T + 1))
        best = max(itertools.combinations(range(T), keep),
                   key=lambda c: (sorted(imp[list(c)].tolist(), reverse=True), [-i for i in c]))
        assert O.select_tokens(imp, keep).tolist() == list(best)


def test_silu_closed_forms():
    x = np.array([-30.0, -2.0, -0.5, 0.0, 0.5, 2.0, 30.0])
    y = O.silu(x)
    assert y[3] == 0.0 and abs(y[-1] - 30.0) < 1e-10 and abs(y[0]) < 1e-10
    assert np.allclose(O.silu(-x), y - x, atol=1e-11)   # silu(-x) = silu(x) - x (cancels near x = 30)
    assert abs(O.silu(np.array([1.0]))[0] - 1.0 / (1.0 + math.exp(-1.0))) < 1e-16


def test_gated_ffn_hand_example():
    # d_model 2, d_ff 1: g = x . (1, 0) = 1, u = x . (0, 1) = 2, a = silu(1) * 2, y = (a, 2a)
    x = np.array([[1.0, 2.0]])
    y = O.gated_ffn(x, np.array([[1.0, 0.0]]), np.array([[0.0, 1.0]]), np.array([[1.0], [2.0]]))
    a = 2.0 / (1.0 + math.exp(-1.0))
    assert np.allclose(y, [[a, 2 * a]], atol=1e-15)


def test_gated_ffn_matches_torch():
    rng = np.random.default_rng(22)
    x, wg, wu, wd = (rng.standard_normal(s) for s in ((5, 16), (24, 16), (24, 16), (16, 24)))
    t = torch.from_numpy
    ref = (torch.nn.functional.silu(t(x) @ t(wg).T) * (t(x) @ t(wu).T)) @ t(wd).T
    assert np.allclose(O.gated_ffn(x, wg, wu, wd), ref.numpy(), atol=1e-12)


def test_sparse_ffn_is_the_dense_ffn_on_kept_rows_and_zero_elsewhere():
    w = synth.sparse_ffn_workload(T=40, d_model=16, d_ff=32, keep_frac=0.3)
    kept, rows = O.sparse_ffn(w.x, w.importance, w.keep, w.w_gate, w.w_up, w.w_down)
    dense = O.gated_ffn(O.bf16_to_f64(w.x), O.bf16_to_f64(w.w_gate), O.bf16_to_f64(w.w_up), O.bf16_to_f64(w.w_down))
    assert len(kept) == w.keep and set(rows) == set(kept.tolist())
    for t, y in rows.items():
        assert np.array_equal(y, dense[t]) or np.allclose(y, dense[t], atol=1e-12)
    top = np.argsort(-w.importance.astype(np.float64), kind="stable")[:w.keep]
    assert sorted(top.tolist()) == kept.tolist()
