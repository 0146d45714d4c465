"""fp64 CPU oracle for RoPE repositioning and SegPagedAttention.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's CPU
baseline leg may import this module; the library path never does.  It shares no
code with the CUDA library: it reads the same numpy inputs (bf16 as uint16 bit
patterns) and recomputes everything in float64, slowly and plainly.

What it computes, and where the pages state it:

* RoPE repositioning ("RedKnot" article on is96.com, paragraphs on RoPE and on
  the correction RedKnot applies): cached K was rotated at its offline
  position; it is first rotated *back* at that offline position and then
  rotated *forward* at the online position.  Both rotations are applied here,
  one after the other, exactly as described.  The rotation itself (which
  channels pair up, the frequency of each pair) is not printed on the pages;
  the reading taken is the one of the Qwen/Llama families the pages evaluate:
  channel i pairs with i + d/2 (or, as an option, 2i with 2i+1) and turns by
  position * theta^(-2i/d).
* Per-head page tables ("RedKnot" article, SegPagedAttention paragraph; "小红书
  RedKnot" section 3, fourth component): each (sequence, KV head) segment lists
  the pages it reads; token j of a segment lives in logical page j // P, slot
  j % P, and the table maps the logical page to a physical page of the shared
  pool ("PagedAttention & RadixAttention", "The Solution: Fixed-size blocks").
* Head classes ("小红书 RedKnot", section 3, first component): global heads see
  the whole (causal) context, local heads a window of recent tokens, retrieval
  heads the pages their table lists, dense heads the whole context of freshly
  computed K.  The visible set of the query at position p is materialised
  explicitly:
      V(p) = { j : page j // P is listed, j < seq_len, j <= p,
               and, for a local head, j > p - W or j < S }.
* Attention ("PagedAttention & RadixAttention": the attention math itself is
  the standard dot-product softmax, only storage and gathering change):
      o = sum_{j in V(p)} softmax_j(q . k_j * scale) v_j,   lse = log sum_j e^{q.k_j*scale}
  with scale = 1/sqrt(d) and query head h reading KV head h // (Hq/Hkv).
* Split combine (standard FlashAttention split-KV merge of partial (m, l, o)).
* Decode-time storage ("小红书 RedKnot" section 3, first and fourth components: local
  heads keep only a window of KV; pages as in "PagedAttention & RadixAttention"): the
  new token's K/V go to slot pos % P of the page listed for logical page pos // P; a
  window-only local head reuses the page of its oldest window entry once the window has
  left it (append_rows, ring_advance).
* Token-level sparse FFN ("小红书 RedKnot" section 3, third component): the tokens of
  highest attention importance go through the gated FFN, the others skip it
  (select_tokens, gated_ffn, sparse_ffn).

Readings of silent points are listed in the repository's design notes; the
pins that tie each function to something other than itself live in
tests/test_oracle_pins.py.
"""
from __future__ import annotations

import math
from typing import Dict, Iterable, List, Optional, Sequence, Tuple

import numpy as np

GLOBAL, LOCAL, RETRIEVAL, DENSE = 0, 1, 2, 3
ROPE_HALF_SPLIT, ROPE_INTERLEAVED = 0, 1


# ----------------------------------------------------------------------------- bf16
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def f64_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 to the nearest bf16 (ties to even), returned as uint16 bits.

    Rounds directly from float64 (no intermediate float32 rounding): write
    |x| = m * 2^e with m in [0.5, 1); bf16 keeps 8 significant bits, so the
    quantum is 2^(e-8), or 2^-133 below the normal range.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    e = np.maximum(e, -125)
    quantum = np.ldexp(1.0, e - 8)
    r = np.rint(x / quantum) * quantum          # np.rint rounds half to even; exact in fp64
    # r has at most 8 significant bits, so the float32 conversion below is exact
    return (np.asarray(r, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def bf16_ordinal(bits: np.ndarray) -> np.ndarray:
    """Monotone integer map of bf16 values, so that ordinal distance = ulp distance."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


# ----------------------------------------------------------------------------- RoPE
def rope_inv_freq(theta: float, d: int) -> np.ndarray:
    """Frequency of channel pair i: theta^(-2i/d), i < d/2, in float64."""
    i = np.arange(d // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * i / d)


def rope_pairs(d: int, style: int) -> Tuple[np.ndarray, np.ndarray]:
    """Channel indices (a_i, b_i) of pair i."""
    i = np.arange(d // 2)
    if style == ROPE_HALF_SPLIT:
        return i, i + d // 2
    if style == ROPE_INTERLEAVED:
        return 2 * i, 2 * i + 1
    raise ValueError("unknown RoPE style")


def rope_rotate(x: np.ndarray, pos: np.ndarray, theta: float, style: int = ROPE_HALF_SPLIT,
                inverse: bool = False) -> np.ndarray:
    """Rotate each row x[t, :] by its position pos[t]: pair (a_i, b_i) turns by
    angle pos * theta^(-2i/d) (clockwise when inverse)."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    a, b = rope_pairs(d, style)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * rope_inv_freq(theta, d)[None, :]
    c, s = np.cos(ang), np.sin(ang)
    if inverse:
        s = -s
    y = np.empty_like(x)
    y[:, a] = x[:, a] * c - x[:, b] * s
    y[:, b] = x[:, a] * s + x[:, b] * c
    return y


def rope_reposition(k: np.ndarray, pos_off: np.ndarray, pos_on: np.ndarray, theta: float,
                    style: int = ROPE_HALF_SPLIT) -> np.ndarray:
    """Inverse rotation at the offline position, then forward rotation at the online one."""
    back = rope_rotate(k, pos_off, theta, style, inverse=True)
    return rope_rotate(back, pos_on, theta, style, inverse=False)


def token_to_physical(table: Sequence[int], P: int, t: int) -> Tuple[int, int]:
    """Logical token t -> (physical page, slot) through a dense block table."""
    return int(table[t // P]), t % P


def paged_rope_reposition(k_src: np.ndarray, src_tables: np.ndarray, dst_tables: np.ndarray,
                          runs: np.ndarray, theta: float, P: int, style: int = ROPE_HALF_SPLIT,
                          return_inputs: bool = False):
    """Apply every run; returns (dst_page, dst_slot, rows): the fp64 rows written and where
    (plus the fp64 input rows when return_inputs).

    Run fields: src_tab_off, src_tab_len, dst_tab_off, dst_tab_len, pos_off0, pos_on0, n_tok.
    Token t of a run reads slot (pos_off0+t) of its src table and writes slot
    (pos_on0+t) of its dst table.
    """
    pages, slots, rows, inputs = [], [], [], []
    for r in np.asarray(runs):
        s_off, s_len, d_off, d_len, p_off0, p_on0, n = (int(v) for v in r[:7])
        if n == 0:
            continue
        t = np.arange(n, dtype=np.int64)
        p_off = p_off0 + t
        p_on = p_on0 + t
        s_tab = np.asarray(src_tables[s_off:s_off + s_len], dtype=np.int64)
        d_tab = np.asarray(dst_tables[d_off:d_off + d_len], dtype=np.int64)
        x = bf16_to_f64(k_src[s_tab[p_off // P], p_off % P])
        inputs.append(x)
        rows.append(rope_reposition(x, p_off, p_on, theta, style))
        pages.append(d_tab[p_on // P])
        slots.append(p_on % P)
    if not rows:
        d = k_src.shape[-1]
        out = (np.zeros(0, np.int64), np.zeros(0, np.int64), np.zeros((0, d)))
        return out + (np.zeros((0, d)),) if return_inputs else out
    out = (np.concatenate(pages), np.concatenate(slots), np.concatenate(rows))
    return out + (np.concatenate(inputs),) if return_inputs else out


def rope_within_one_ulp(got_bits: np.ndarray, exact: np.ndarray, inputs: np.ndarray, style: int,
                        floor_rel: float = 1e-12) -> np.ndarray:
    """Per element: is the bf16 value within 1 bf16 ulp of the fp64 result?

    The fp64 result itself carries round-off of about 1e-16 of its pair's magnitude
    (two rotations), which near zero is any number of bf16 ulps; so an element also
    passes when it is within floor_rel * |pair| of the fp64 value (e.g. an exact zero
    kept at zero by a zero turn)."""
    d = exact.shape[-1]
    a, b = rope_pairs(d, style)
    pair = np.sqrt(inputs[:, a] ** 2 + inputs[:, b] ** 2)
    mag = np.empty_like(exact)
    mag[:, a] = pair
    mag[:, b] = pair
    ulp_ok = np.abs(bf16_ordinal(got_bits) - bf16_ordinal(f64_to_bf16(exact))) <= 1
    abs_ok = np.abs(bf16_to_f64(got_bits) - exact) <= floor_rel * mag
    return ulp_ok | abs_ok


def apply_rope_to_pool(k_pool: np.ndarray, written) -> np.ndarray:
    """Store the oracle's repositioned rows into a copy of a bf16 pool (RNE to bf16:
    the pool's storage type)."""
    pages, slots, rows = written
    out = np.array(k_pool, copy=True)
    out[pages, slots] = f64_to_bf16(rows)
    return out


# ----------------------------------------------------------------------------- visibility
def listed_positions(page_logical_row: np.ndarray, n_listed: int, P: int) -> np.ndarray:
    """Logical token positions covered by the listed pages of one head segment."""
    lp = np.asarray(page_logical_row[:n_listed], dtype=np.int64)
    return (lp[:, None] * P + np.arange(P)[None, :]).reshape(-1)


def visible_set(cls: int, window: int, sink: int, seq_len: int, p: int,
                listed: np.ndarray) -> np.ndarray:
    """Sorted logical key positions visible to the query at position p."""
    j = np.asarray(listed, dtype=np.int64)
    keep = (j < seq_len) & (j <= p)
    if cls == LOCAL:
        keep &= (j > p - window) | (j < sink)
    elif cls not in (GLOBAL, RETRIEVAL, DENSE):
        raise ValueError("unknown head class")
    return np.sort(j[keep])


def gather_rows(pool: np.ndarray, table_row: np.ndarray, logical_row: np.ndarray, n_listed: int,
                P: int, positions: np.ndarray) -> np.ndarray:
    """fp64 rows of the given logical positions, read through the head's page list."""
    lp2phys = {int(logical_row[e]): int(table_row[e]) for e in range(n_listed)}
    pg = np.array([lp2phys[int(p) // P] for p in positions], dtype=np.int64)
    return bf16_to_f64(pool[pg, np.asarray(positions, dtype=np.int64) % P])


# ----------------------------------------------------------------------------- attention
def softmax_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float):
    """Dense softmax attention of query rows q [G, d] over keys k/v [n, d] (fp64).
    Returns (o [G, d], lse [G]); an empty key set gives o = 0, lse = -inf."""
    if k.shape[0] == 0:
        return np.zeros((q.shape[0], v.shape[1])), np.full(q.shape[0], -np.inf)
    s = (q @ k.T) * scale
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=1, keepdims=True)
    o = (e @ v) / l
    return o, (m + np.log(l))[:, 0]


def segpaged_attention(batch, rows: Optional[Iterable[Tuple[int, int]]] = None,
                       scale: Optional[float] = None):
    """Reference outputs of one SegPaged attention launch.

    rows: iterable of (query token index into q, KV head) to compute; None = all.
    Returns dict {(t, h_kv): (o [G, d], lse [G])} for the G query heads of group h_kv.
    """
    B, Hq, Hkv, d, P = batch.B, batch.Hq, batch.Hkv, batch.d, batch.P
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    cu = np.asarray(batch.cu_seqlens_q)
    tok_seq = np.repeat(np.arange(B), np.diff(cu))
    if rows is None:
        rows = [(t, h) for t in range(int(cu[-1])) for h in range(Hkv)]
    # group requested rows by head segment so each segment's keys are gathered once
    by_seg: Dict[Tuple[int, int], List[int]] = {}
    for t, h in rows:
        by_seg.setdefault((int(tok_seq[t]), int(h)), []).append(int(t))
    out = {}
    for (b, h), toks in by_seg.items():
        seg = b * Hkv + h
        nl = int(batch.n_pages[seg])
        listed = listed_positions(batch.page_logical[seg], nl, P)
        L = int(batch.seq_len[b])
        nq = int(cu[b + 1] - cu[b])
        cls, W, S = int(batch.head_class[seg]), int(batch.window[seg]), int(batch.sink[seg])
        cand = np.sort(listed[listed < L])
        kk = gather_rows(batch.k_pool, batch.page_table[seg], batch.page_logical[seg], nl, P, cand)
        vv = gather_rows(batch.v_pool, batch.page_table[seg], batch.page_logical[seg], nl, P, cand)
        for t in toks:
            p = L - nq + (t - int(cu[b]))
            vis = visible_set(cls, W, S, L, p, cand)
            idx = np.searchsorted(cand, vis)      # vis is a subset of the sorted cand
            qg = bf16_to_f64(batch.q[t, h * G:(h + 1) * G])
            out[(t, h)] = softmax_attention(qg, kk[idx], vv[idx], scale)
    return out


def split_partials(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float, bounds: Sequence[int]):
    """Unnormalised partial results (m, l, o) of attention over key ranges [bounds[i], bounds[i+1])."""
    parts = []
    for a, b in zip(bounds[:-1], bounds[1:]):
        if b <= a:
            parts.append((np.full(q.shape[0], -np.inf), np.zeros(q.shape[0]), np.zeros((q.shape[0], v.shape[1]))))
            continue
        s = (q @ k[a:b].T) * scale
        m = s.max(axis=1)
        e = np.exp(s - m[:, None])
        parts.append((m, e.sum(axis=1), e @ v[a:b]))
    return parts


def combine_partials(parts):
    """Merge split partials: m = max m_i, l = sum e^{m_i-m} l_i, o = sum e^{m_i-m} o_i / l."""
    ms = np.stack([p[0] for p in parts])
    m = ms.max(axis=0)
    w = np.where(np.isfinite(ms), np.exp(ms - m[None, :]), 0.0)
    l = sum(w[i] * parts[i][1] for i in range(len(parts)))
    o = sum(w[i][:, None] * parts[i][2] for i in range(len(parts)))
    return o / l[:, None], m + np.log(l)


def attention_flops(batch) -> int:
    """Algorithmic FLOPs: 4 * d * visible (query head, key) pairs, by explicit count."""
    B, Hq, Hkv, d, P = batch.B, batch.Hq, batch.Hkv, batch.d, batch.P
    G = Hq // Hkv
    cu = np.asarray(batch.cu_seqlens_q)
    pairs = 0
    for b in range(B):
        L = int(batch.seq_len[b])
        nq = int(cu[b + 1] - cu[b])
        for h in range(Hkv):
            seg = b * Hkv + h
            listed = listed_positions(batch.page_logical[seg], int(batch.n_pages[seg]), P)
            cls, W, S = int(batch.head_class[seg]), int(batch.window[seg]), int(batch.sink[seg])
            for i in range(nq):
                pairs += len(visible_set(cls, W, S, L, L - nq + i, listed))
    return 4 * d * G * pairs


# ----------------------------------------------------------------------------- decode storage
def append_rows(k_pool: np.ndarray, v_pool: np.ndarray, page_table: np.ndarray, page_logical: np.ndarray,
                n_pages: np.ndarray, pos: np.ndarray, k_new: np.ndarray, v_new: np.ndarray, Hkv: int, P: int):
    """Copies of the pools with the new token of every head segment stored: segment
    s = b*Hkv + h writes k_new[b, h] / v_new[b, h] (bf16 bits, unchanged) to slot pos[b] % P
    of the physical page its list gives for logical page pos[b] // P."""
    k_out, v_out = np.array(k_pool, copy=True), np.array(v_pool, copy=True)
    B = len(pos)
    for b in range(B):
        for h in range(Hkv):
            s = b * Hkv + h
            lp = int(pos[b]) // P
            listed = [int(x) for x in page_logical[s, :int(n_pages[s])]]
            e = listed.index(lp)                     # the page must be listed
            phys = int(page_table[s, e])
            k_out[phys, int(pos[b]) % P] = k_new[b, h]
            v_out[phys, int(pos[b]) % P] = v_new[b, h]
    return k_out, v_out


def ring_advance(page_table: np.ndarray, page_logical: np.ndarray, n_pages: np.ndarray, ring: np.ndarray,
                 window: np.ndarray, sink: np.ndarray, pos: np.ndarray, Hkv: int, P: int):
    """Copies of the tables after the page ring of each window-only local head (ring[s] > 0)
    has made room for the token at pos[b]: if logical page pos // P is not listed yet, the
    oldest window page (the first entry after the sink pages) leaves the window -- it must
    end at or before pos - W -- and its physical page holds the new logical page, which
    becomes the last entry."""
    tab, lg = np.array(page_table, copy=True), np.array(page_logical, copy=True)
    for s in range(len(ring)):
        R = int(ring[s])
        if R <= 0:
            continue
        p = int(pos[s // Hkv])
        n = int(n_pages[s])
        entries = list(zip(lg[s, :n].tolist(), tab[s, :n].tolist()))   # (logical, physical)
        if entries[-1][0] >= p // P:
            continue
        sink_pages = -(-int(sink[s]) // P)
        sinks = [x for x in entries if x[0] < sink_pages]
        win = [x for x in entries if x[0] >= sink_pages]
        assert len(win) == R, "the ring holds R window pages"
        oldest_lp, oldest_phys = win[0]
        assert (oldest_lp + 1) * P - 1 <= p - int(window[s]), "the oldest page is outside the window"
        new = sinks + win[1:] + [(p // P, oldest_phys)]
        lg[s, :n] = [x[0] for x in new]
        tab[s, :n] = [x[1] for x in new]
    return tab, lg


# ----------------------------------------------------------------------------- sparse FFN
# "小红书 RedKnot", section 3, third component: tokens ranked by attention importance; only
# the most important go through the FFN, the others skip it.  The FFN is the gated form of
# the Qwen / Llama models the pages evaluate.
def silu(g: np.ndarray) -> np.ndarray:
    """g * sigmoid(g) = g / (1 + e^-g), in float64."""
    g = np.asarray(g, dtype=np.float64)
    return g / (1.0 + np.exp(-g))


def select_tokens(importance: np.ndarray, keep: int) -> np.ndarray:
    """The `keep` tokens with the largest importance (equal scores: lower index first; NaN
    below every number), in ascending token order."""
    imp = np.asarray(importance, dtype=np.float64)
    key = np.where(np.isnan(imp), -np.inf, imp)
    idx = np.arange(len(imp))
    nan_last = np.isnan(imp).astype(np.int64)
    order = np.lexsort((idx, nan_last, -key))        # by score descending, NaN after, then index
    return np.sort(order[:keep])


def gated_ffn(x: np.ndarray, w_gate: np.ndarray, w_up: np.ndarray, w_down: np.ndarray) -> np.ndarray:
    """W_down (silu(W_gate x) * (W_up x)) for each row x, all in float64."""
    g = x @ w_gate.T
    u = x @ w_up.T
    return (silu(g) * u) @ w_down.T


def sparse_ffn(x_bits, importance, keep, w_gate_bits, w_up_bits, w_down_bits, rows=None):
    """(kept tokens, {token: FFN output row in float64}) for the kept tokens in `rows` (all
    kept tokens when rows is None); every other token's output is zero."""
    kept = select_tokens(importance, keep)
    want = kept if rows is None else np.array([t for t in rows if t in set(kept.tolist())], dtype=np.int64)
    if len(want) == 0:
        return kept, {}
    y = gated_ffn(bf16_to_f64(x_bits[want]), bf16_to_f64(w_gate_bits), bf16_to_f64(w_up_bits),
                  bf16_to_f64(w_down_bits))
    return kept, {int(t): y[i] for i, t in enumerate(want)}
