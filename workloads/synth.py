"""Seeded synthetic inputs for the paged-RoPE / SegPagedAttention path.

This module only *draws* inputs: random bf16 tensors, seeded page permutations,
per-head class picks and the page tables that follow from them.  It holds none
of the method's arithmetic (no rotation, no softmax, no visibility predicate):
both the fp64 oracle and the CUDA library consume what it produces.

Shapes follow the workloads the RedKnot pages describe:
  * "小红书 RedKnot" product page, section 3: four head classes (global, local,
    retrieval, dense), offline KV reuse with RoPE repositioning, per-head page
    tables;
  * "RedKnot HotpotQA Demo" tutorial, step 2: 6 reusable segments x 5000 tokens,
    about 15 % global KV heads and the rest local with window 256; the
    SegPagedAttention microbenchmark at 8K / 32K / 128K;
  * "PagedAttention & RadixAttention", section "The Solution: Fixed-size
    blocks": fixed-size pages of 16 or 32 tokens drawn from one global pool,
    logical block -> physical block through a per-sequence block table.

Conventions shared by both sides (data layout only):
  * bf16 tensors are numpy uint16 bit patterns.
  * K/V pools are [n_pages][P][d]; page id p refers to k_pool[p] and v_pool[p].
  * A head segment is one (sequence b, KV head h) pair, index b*Hkv + h.
  * page_table[b*Hkv+h][e] is the physical page of the e-th listed page and
    page_logical[...][e] its logical page index (ascending); token position j
    lives in logical page j // P, slot j % P.
  * Query i of sequence b sits at position seq_len[b] - nq_b + i.
  * head_class: 0 global, 1 local, 2 retrieval, 3 dense.
  * A RoPE run moves n_tok consecutive tokens of one head segment from the
    offline store (token t at offline position pos_off0 + t, looked up in the
    run's src table) to the online pool (online position pos_on0 + t, looked
    up in the run's dst table).  Cached K is drawn directly as the content of
    the offline store: it stands for K that was rotated at its offline
    positions when the segment was prefilled offline.
"""
from __future__ import annotations

import concurrent.futures
import dataclasses
import os
from typing import List, Optional

import numpy as np

GLOBAL, LOCAL, RETRIEVAL, DENSE = 0, 1, 2, 3
RUN_FIELDS = 8  # src_tab_off, src_tab_len, dst_tab_off, dst_tab_len, pos_off0, pos_on0, n_tok, reserved


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round-to-nearest-even), as uint16 bits."""
    u = np.array(x, dtype=np.float32, copy=True).view(np.uint32)
    t = u >> 16
    t &= 1
    t += np.uint32(0x7FFF)
    u += t
    u >>= 16
    return u.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


_CHUNK = 1 << 22          # values per independently seeded chunk (fixed: results do not depend on threads)
_POOL = concurrent.futures.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1))


def _normal_bf16(rng: np.random.Generator, shape, scale=None) -> np.ndarray:
    """bf16 N(0,1) draws.  The draw is split into fixed-size chunks, each from its own
    PCG64 stream spawned from one seed taken from `rng`, and filled on worker threads."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    if n == 0:
        return out.reshape(shape)
    seeds = np.random.SeedSequence(int(rng.integers(0, 2 ** 63))).spawn((n + _CHUNK - 1) // _CHUNK)

    def fill(i):
        lo, hi = i * _CHUNK, min(n, (i + 1) * _CHUNK)
        x = np.random.Generator(np.random.PCG64(seeds[i])).standard_normal(hi - lo, dtype=np.float32)
        out[lo:hi] = f32_to_bf16_bits(x)

    list(_POOL.map(fill, range(len(seeds))))
    out = out.reshape(shape)
    if scale is not None:
        out = f32_to_bf16_bits(bf16_bits_to_f32(out) * scale)
    return out


@dataclasses.dataclass
class AttnBatch:
    """Inputs of one SegPaged attention launch (prefill or decode)."""
    B: int
    Hq: int
    Hkv: int
    d: int
    P: int
    q: np.ndarray              # uint16 [T][Hq][d]
    cu_seqlens_q: np.ndarray   # int32 [B+1]
    seq_len: np.ndarray        # int32 [B]
    k_pool: np.ndarray         # uint16 [n_pages][P][d]
    v_pool: np.ndarray         # uint16 [n_pages][P][d]
    page_table: np.ndarray     # int32 [B*Hkv][max_pages]
    page_logical: np.ndarray   # int32 [B*Hkv][max_pages]
    n_pages: np.ndarray        # int32 [B*Hkv]
    head_class: np.ndarray     # int32 [B*Hkv]
    window: np.ndarray         # int32 [B*Hkv]
    sink: np.ndarray           # int32 [B*Hkv]
    name: str = ""

    @property
    def max_pages(self) -> int:
        return int(self.page_table.shape[1])

    @property
    def total_q(self) -> int:
        return int(self.cu_seqlens_q[-1])

    @property
    def nq(self) -> np.ndarray:
        return np.diff(self.cu_seqlens_q).astype(np.int32)

    @property
    def max_q(self) -> int:
        return int(self.nq.max()) if self.B else 0


@dataclasses.dataclass
class RopeJob:
    """Inputs of one RoPE repositioning launch.

    The destination pool is the K pool of the AttnBatch it feeds.
    """
    k_src: np.ndarray          # uint16 [n_src_pages][P][d]  offline store
    src_tables: np.ndarray     # int32 [n_src_entries]
    dst_tables: np.ndarray     # int32 [n_dst_entries]  dense logical->physical tables
    runs: np.ndarray           # int32 [n_runs][RUN_FIELDS]
    theta: float
    P: int
    d: int
    style: int = 0             # 0 half-split pairs (i, i+d/2), 1 interleaved (2i, 2i+1)
    run_seg: Optional[np.ndarray] = None   # int32 [n_runs] head segment (b*Hkv + h) of each run

    @property
    def n_runs(self) -> int:
        return int(self.runs.shape[0])

    @property
    def max_tok(self) -> int:
        return int(self.runs[:, 6].max()) if self.n_runs else 0

    @property
    def total_tok(self) -> int:
        return int(self.runs[:, 6].sum()) if self.n_runs else 0


@dataclasses.dataclass
class Workload:
    name: str
    attn: AttnBatch
    rope: Optional[RopeJob]
    theta: float
    decode_q: Optional[np.ndarray] = None   # uint16 [steps][B][Hq][d] for decode steps after the prefill
    # decode with appended tokens (ring_decode): the K/V each step appends, and the tables the
    # decode starts from -- window-only local heads keep a ring of their last `ring` window pages
    decode_k: Optional[np.ndarray] = None   # uint16 [steps][B][Hkv][d]
    decode_v: Optional[np.ndarray] = None   # uint16 [steps][B][Hkv][d]
    dec_page_table: Optional[np.ndarray] = None     # int32 [B*Hkv][max_pages]
    dec_page_logical: Optional[np.ndarray] = None   # int32 [B*Hkv][max_pages]
    dec_n_pages: Optional[np.ndarray] = None        # int32 [B*Hkv]
    ring: Optional[np.ndarray] = None               # int32 [B*Hkv]: ring pages of a window-only local head, else 0


class _PageAllocator:
    """Hands out physical page ids from a seeded permutation of the pool."""

    def __init__(self, rng: np.random.Generator, n_pool: int):
        self.order = rng.permutation(n_pool).astype(np.int32)
        self.next = 0
        self.n_pool = n_pool

    def take(self, n: int) -> np.ndarray:
        if self.next + n > self.n_pool:
            raise ValueError("page pool exhausted")
        out = self.order[self.next:self.next + n]
        self.next += n
        return out


def _cdiv(a: int, b: int) -> int:
    return -(-a // b)


def _build(name, rng, *, B, Hq, Hkv, d, P, theta, ctx_len, n_suffix, classes, windows, sinks,
           seg_tokens, k_scale=None, retrieval_frac=0.25, retrieval_window=256,
           local_window_only=False, pool_slack=1.0, n_decode=0, style=0, with_rope=True, ring_decode=False):
    """Common builder.

    ctx_len[b]: context tokens (made of reusable segments of seg_tokens[b] each, the
    last one possibly shorter); n_suffix[b]: suffix queries; classes/windows/sinks:
    [B][Hkv].  Storage of every head segment is dense over [0, seq_len + n_decode);
    what a head *lists* for attention depends on its class.  With local_window_only,
    local heads store (and list) only their sink pages and the pages covering the
    windows of their queries.  With ring_decode as well, local heads store nothing for
    the decode steps: each step appends its token (decode_k / decode_v), and a local
    head starts the decode from its last ceil(W/P) + 1 window pages, which it reuses as
    a ring (dec_* tables, ring); other heads have their decode pages allocated already.
    """
    ctx_len = np.asarray(ctx_len, dtype=np.int64)
    n_suffix = np.asarray(n_suffix, dtype=np.int64)
    seq_len = ctx_len + n_suffix                     # prefill length
    store_len = seq_len + n_decode                   # tokens stored per head segment
    pages_per_head = [_cdiv(int(s), P) for s in store_len]
    if ring_decode:
        local_window_only = True

    # page lists (logical indices) per head segment
    lists = []
    for b in range(B):
        npg = pages_per_head[b]
        for h in range(Hkv):
            c = int(classes[b][h])
            if c == LOCAL and local_window_only:
                # sink pages + pages covering the windows of the queries (prefill or decode)
                first_q = int(seq_len[b] - n_suffix[b])
                lo_pos = max(0, first_q - int(windows[b][h]) + 1)
                lp = set(range(0, _cdiv(int(sinks[b][h]), P)))
                lp.update(range(lo_pos // P, _cdiv(int(seq_len[b]), P) if ring_decode else npg))
                lists.append(np.array(sorted(lp), dtype=np.int32))
            elif c == RETRIEVAL:
                n_ctx_pages = _cdiv(int(ctx_len[b]), P)
                pick = rng.permutation(n_ctx_pages)[: max(1, int(round(retrieval_frac * n_ctx_pages)))]
                lp = set(int(x) for x in pick)
                lo_pos = max(0, int(ctx_len[b]) - retrieval_window)
                lp.update(range(lo_pos // P, n_ctx_pages))        # last window of the context
                lp.update(range(int(ctx_len[b]) // P, npg))        # the suffix's own pages
                lists.append(np.array(sorted(lp), dtype=np.int32))
            else:
                lists.append(np.arange(npg, dtype=np.int32))

    # which logical pages each head segment stores: everything, except local heads that
    # keep only their listed (sink + window) pages
    stored = []
    for b in range(B):
        for h in range(Hkv):
            i = b * Hkv + h
            if int(classes[b][h]) == LOCAL and local_window_only:
                stored.append(lists[i])
            else:
                stored.append(np.arange(pages_per_head[b], dtype=np.int32))
    n_store_pages = sum(len(x) for x in stored)
    n_pool = max(n_store_pages, int(np.ceil(n_store_pages * pool_slack)))
    alloc = _PageAllocator(rng, n_pool)

    # dense storage tables (logical page -> physical page, -1 where nothing is stored)
    storage = []
    for b in range(B):
        for h in range(Hkv):
            i = b * Hkv + h
            tab = np.full(pages_per_head[b], -1, dtype=np.int32)
            tab[stored[i]] = alloc.take(len(stored[i]))
            storage.append(tab)

    max_pages = max(1, max(len(x) for x in lists))
    page_table = np.full((B * Hkv, max_pages), -1, dtype=np.int32)
    page_logical = np.full((B * Hkv, max_pages), -1, dtype=np.int32)
    n_pages = np.zeros(B * Hkv, dtype=np.int32)
    for i, lp in enumerate(lists):
        page_table[i, :len(lp)] = storage[i][lp]
        page_logical[i, :len(lp)] = lp
        n_pages[i] = len(lp)

    # pool contents: V everywhere; K everywhere (segment K of non-dense heads is
    # overwritten by the RoPE step on the path; the drawn values there stand for stale data)
    k_pool = _normal_bf16(rng, (n_pool, P, d))
    v_pool = _normal_bf16(rng, (n_pool, P, d))
    if k_scale is not None:
        # per (KV head, channel) scale on every K the head stores
        kf = bf16_bits_to_f32(k_pool)
        for b in range(B):
            for h in range(Hkv):
                pg = storage[b * Hkv + h]
                pg = pg[pg >= 0]
                kf[pg] *= k_scale[h][None, None, :]
        k_pool = f32_to_bf16_bits(kf)

    cu = np.zeros(B + 1, dtype=np.int32)
    cu[1:] = np.cumsum(n_suffix)
    q = _normal_bf16(rng, (int(cu[-1]), Hq, d))

    head_class = np.asarray(classes, dtype=np.int32).reshape(-1)
    window = np.asarray(windows, dtype=np.int32).reshape(-1)
    sink = np.asarray(sinks, dtype=np.int32).reshape(-1)
    attn = AttnBatch(B=B, Hq=Hq, Hkv=Hkv, d=d, P=P, q=q, cu_seqlens_q=cu,
                     seq_len=seq_len.astype(np.int32), k_pool=k_pool, v_pool=v_pool,
                     page_table=page_table, page_logical=page_logical, n_pages=n_pages,
                     head_class=head_class, window=window, sink=sink, name=name)

    rope = None
    if with_rope:
        # offline store: each (sequence, segment, non-dense KV head) keeps its cached K at
        # offline positions 0..n-1 in its own pages
        src_tabs, dst_tabs, runs = [], [], []
        src_off = 0
        dst_off = 0
        dst_index = {}
        for b in range(B):
            for h in range(Hkv):
                dst_index[(b, h)] = dst_off
                dst_tabs.append(storage[b * Hkv + h])
                dst_off += len(storage[b * Hkv + h])
        seg_plan = []
        for b in range(B):
            st = int(seg_tokens[b])
            pos = 0
            while pos < int(ctx_len[b]):
                n = min(st, int(ctx_len[b]) - pos)
                seg_plan.append((b, pos, n))
                pos += n
        n_src_pages = 0
        src_list = []
        for (b, pos_on0, n) in seg_plan:
            for h in range(Hkv):
                if int(classes[b][h]) == DENSE:
                    continue
                npg = _cdiv(n, P)
                src_list.append((b, h, pos_on0, n, npg))
                n_src_pages += npg
        src_alloc = _PageAllocator(rng, n_src_pages)
        run_seg = []
        for (b, h, pos_on0, n, npg) in src_list:
            pages = src_alloc.take(npg)
            src_tabs.append(pages)
            runs.append([src_off, npg, dst_index[(b, h)], len(storage[b * Hkv + h]), 0, pos_on0, n, 0])
            run_seg.append(b * Hkv + h)
            src_off += npg
        k_src = _normal_bf16(rng, (max(n_src_pages, 1), P, d))
        if k_scale is not None:
            kf = bf16_bits_to_f32(k_src)
            for r, (b, h, pos_on0, n, npg) in enumerate(src_list):
                pages = src_tabs[r]
                kf[pages] *= k_scale[h][None, None, :]
            k_src = f32_to_bf16_bits(kf)
        if local_window_only:
            # a window-only local head repositions only the tokens it stores: the run is cut
            # to the stored logical pages (sink pages, then the window pages)
            cut, cut_seg = [], []
            for r, (b, h, pos_on0, n, npg) in zip(runs, src_list):
                if int(classes[b][h]) != LOCAL:
                    cut.append(r)
                    cut_seg.append(b * Hkv + h)
                    continue
                st = stored[b * Hkv + h]
                lo_s, hi_s = pos_on0, pos_on0 + n
                for a0, a1 in _page_ranges(st):
                    x0, x1 = max(lo_s, a0 * P), min(hi_s, a1 * P)
                    if x0 < x1:
                        cut.append([r[0], r[1], r[2], r[3], x0 - pos_on0, x0, x1 - x0, 0])
                        cut_seg.append(b * Hkv + h)
            runs, run_seg = cut, cut_seg
        rope = RopeJob(k_src=k_src,
                       src_tables=np.concatenate(src_tabs).astype(np.int32) if src_tabs else np.zeros(1, np.int32),
                       dst_tables=np.concatenate(dst_tabs).astype(np.int32),
                       runs=np.asarray(runs, dtype=np.int32).reshape(-1, RUN_FIELDS),
                       theta=theta, P=P, d=d, style=style, run_seg=np.asarray(run_seg, dtype=np.int32))

    decode_q = None
    if n_decode:
        decode_q = _normal_bf16(rng, (n_decode, B, Hq, d))
    wl = Workload(name=name, attn=attn, rope=rope, theta=theta, decode_q=decode_q)
    if ring_decode and n_decode:
        wl.decode_k = _normal_bf16(rng, (n_decode, B, Hkv, d))
        wl.decode_v = _normal_bf16(rng, (n_decode, B, Hkv, d))
        tab, lg, nn = page_table.copy(), page_logical.copy(), n_pages.copy()
        ring = np.zeros(B * Hkv, dtype=np.int32)
        for b in range(B):
            for h in range(Hkv):
                i = b * Hkv + h
                if int(classes[b][h]) != LOCAL:
                    continue
                R = _cdiv(int(windows[b][h]), P) + 1
                n = int(n_pages[i])
                n_sink = int(np.count_nonzero(page_logical[i, :n] < _cdiv(int(sinks[b][h]), P)))
                if n - n_sink < R:
                    raise ValueError("the prefill lists fewer window pages than the ring needs")
                keep = list(range(n_sink)) + list(range(n - R, n))
                tab[i, :] = -1
                lg[i, :] = -1
                tab[i, :len(keep)] = page_table[i, keep]
                lg[i, :len(keep)] = page_logical[i, keep]
                nn[i] = len(keep)
                ring[i] = R
        wl.dec_page_table, wl.dec_page_logical, wl.dec_n_pages, wl.ring = tab, lg, nn, ring
    return wl


@dataclasses.dataclass
class OnLoadView:
    """Inputs of attention that repositions K as it reads it (zero-copy reuse): the K pool
    with every repositioned page holding its offline rows instead, the per-entry coefficient
    rows (k_rot, -1 for pages read as they are) of the prefill and decode tables, and the
    delta of each coefficient row."""
    k_pool: np.ndarray          # uint16 [n_pages][P][d]
    deltas: np.ndarray          # int32 [n_rot]: online minus offline position
    k_rot: np.ndarray           # int32 [B*Hkv][max_pages] for attn.page_logical
    dec_k_rot: Optional[np.ndarray] = None   # int32 for dec_page_logical


def reposition_on_load_view(wl: Workload) -> OnLoadView:
    """Rearrange a workload for repositioning on load: each page a RoPE run writes gets the
    offline page the run reads (bits copied, no arithmetic), and the entries listing it get
    the run's coefficient row.  Runs must start on a page boundary of both positions and
    fill whole pages (a page holds one run's tokens)."""
    r, a, P = wl.rope, wl.attn, wl.rope.P
    k_pool = np.array(a.k_pool, copy=True)
    deltas, row_of = [], {}
    page_rot = {}                                   # (segment, logical page) -> coefficient row
    for run, seg in zip(r.runs, r.run_seg):
        s_off, s_len, d_off, d_len, p_off0, p_on0, n = (int(x) for x in run[:7])
        if p_off0 % P or p_on0 % P:
            raise ValueError("a run starts inside a page")
        delta = p_on0 - p_off0
        if delta not in row_of:
            row_of[delta] = len(deltas)
            deltas.append(delta)
        for j in range(_cdiv(n, P)):
            rows = min(P, n - j * P)
            if rows < P:   # the rest of the page holds other tokens, which must not be turned
                raise ValueError("a run ends inside a page")
            dst = int(r.dst_tables[d_off + p_on0 // P + j])
            src = int(r.src_tables[s_off + p_off0 // P + j])
            k_pool[dst, :rows] = r.k_src[src, :rows]
            page_rot[(int(seg), p_on0 // P + j)] = row_of[delta]

    def rot_table(logical, n_pages):
        out = np.full(logical.shape, -1, dtype=np.int32)
        for s in range(logical.shape[0]):
            for e in range(int(n_pages[s])):
                out[s, e] = page_rot.get((s, int(logical[s, e])), -1)
        return out

    view = OnLoadView(k_pool=k_pool, deltas=np.asarray(deltas, dtype=np.int32),
                      k_rot=rot_table(a.page_logical, a.n_pages))
    if wl.dec_page_logical is not None:
        view.dec_k_rot = rot_table(wl.dec_page_logical, wl.dec_n_pages)
    return view


def _page_ranges(pages) -> List:
    """Maximal runs [a, b) of consecutive logical pages in a sorted page list."""
    out = []
    for x in (int(v) for v in pages):
        if out and out[-1][1] == x:
            out[-1][1] = x + 1
        else:
            out.append([x, x + 1])
    return out


# --------------------------------------------------------------------------------------
# The five workloads (seed = 1000 + workload id), each with optional size overrides so the
# same recipe also gives small cases the oracle finishes in seconds.
# --------------------------------------------------------------------------------------

def tiny_prefill(seed: int = 1001, style: int = 0) -> Workload:
    """1 layer, Hq 4 / Hkv 2, d 64, theta 1e6; 2 segments x 256 tokens cached at 0..255 and
    repositioned to 0 and 256; 32-token suffix at 512..543; page 16; KV head 0 global,
    KV head 1 local window 64."""
    rng = np.random.default_rng(seed)
    return _build("tiny_prefill", rng, B=1, Hq=4, Hkv=2, d=64, P=16, theta=1e6,
                  ctx_len=[512], n_suffix=[32], classes=[[GLOBAL, LOCAL]], windows=[[0, 64]],
                  sinks=[[0, 0]], seg_tokens=[256], style=style)


def decode_microbench(seed: int = 1002, B: int = 32, ctx: int = 8192, Hq: int = 32, Hkv: int = 8,
                      d: int = 128, P: int = 16, window: int = 256, sink: int = 4,
                      pool_slack: float = 2.0) -> Workload:
    """B independent sequences x ctx tokens, 1 query each at the last position; per sequence
    one seeded KV head global, the rest local (window + sink) listing only their sink and
    window pages; physical pages scattered over a pool of pool_slack x the needed pages."""
    rng = np.random.default_rng(seed)
    classes, windows, sinks = [], [], []
    for b in range(B):
        g = int(rng.integers(Hkv))
        classes.append([GLOBAL if h == g else LOCAL for h in range(Hkv)])
        windows.append([0 if h == g else window for h in range(Hkv)])
        sinks.append([0 if h == g else sink for h in range(Hkv)])
    return _build("decode_microbench", rng, B=B, Hq=Hq, Hkv=Hkv, d=d, P=P, theta=1e6,
                  ctx_len=[ctx - 1] * B, n_suffix=[1] * B, classes=classes, windows=windows,
                  sinks=sinks, seg_tokens=[ctx] * B, local_window_only=True,
                  pool_slack=pool_slack, with_rope=False)


def rag_prefill(seed: int = 1003, n_segments: int = 6, seg_tokens: int = 5000, n_suffix: int = 512,
                Hq: int = 64, Hkv: int = 8, d: int = 128, P: int = 16, window: int = 256,
                global_frac: float = 0.15, theta: float = 1e6) -> Workload:
    """Qwen3-32B-shaped RAG prefill, one layer: n_segments reusable segments, K of each
    repositioned from offline offset 0 to online offset s*seg_tokens; then the suffix;
    round(global_frac*Hkv) global KV heads (seeded pick), the rest local; K carries
    per-(KV head, channel) scales drawn LogUniform(0.5, 4)."""
    rng = np.random.default_rng(seed)
    n_glob = max(1, int(round(global_frac * Hkv)))
    glob = set(int(x) for x in rng.permutation(Hkv)[:n_glob])
    classes = [[GLOBAL if h in glob else LOCAL for h in range(Hkv)]]
    windows = [[0 if h in glob else window for h in range(Hkv)]]
    k_scale = np.exp(rng.uniform(np.log(0.5), np.log(4.0), size=(Hkv, d))).astype(np.float32)
    return _build("rag_prefill", rng, B=1, Hq=Hq, Hkv=Hkv, d=d, P=P, theta=theta,
                  ctx_len=[n_segments * seg_tokens], n_suffix=[n_suffix], classes=classes,
                  windows=windows, sinks=[[0] * Hkv], seg_tokens=[seg_tokens], k_scale=k_scale)


def stack_classes(seed: int = 1004, n_layers: int = 8, Hkv: int = 8, global_frac: float = 0.04):
    """(layer, KV head) classes of the long-context stack: exactly round(global_frac * L * Hkv)
    global pairs picked by a seeded permutation, the rest local."""
    rng = np.random.default_rng(seed)
    n = n_layers * Hkv
    n_glob = int(round(global_frac * n))
    pick = set(int(x) for x in rng.permutation(n)[:n_glob])
    return [[GLOBAL if (l * Hkv + h) in pick else LOCAL for h in range(Hkv)] for l in range(n_layers)]


def stack_layer(layer: int, seed: int = 1004, n_layers: int = 8, n_segments: int = 32,
                seg_tokens: int = 4096, n_suffix: int = 1024, n_decode: int = 64, Hq: int = 64,
                Hkv: int = 8, d: int = 128, P: int = 16, window: int = 512,
                global_frac: float = 0.04, theta: float = 1e6, ring_decode: bool = True) -> Workload:
    """One layer of the 128K long-context stack: n_segments x seg_tokens context, suffix
    prefill of n_suffix tokens, then n_decode decode steps (step s appends the token at
    position ctx + n_suffix + s and sees seq_len = ctx + n_suffix + s + 1).  With ring_decode
    (the default) local heads store only their window -- the pages covering the windows of
    the suffix queries, so only the tail of the last segment is repositioned for them --
    and recycle a ring of ceil(W/P) + 1 pages during the decode; without it every head
    stores every token and the decode tokens are stored in advance."""
    classes = stack_classes(seed, n_layers, Hkv, global_frac)[layer]
    rng = np.random.default_rng([seed, layer])
    windows = [[0 if c == GLOBAL else window for c in classes]]
    return _build(f"stack_layer{layer}", rng, B=1, Hq=Hq, Hkv=Hkv, d=d, P=P, theta=theta,
                  ctx_len=[n_segments * seg_tokens], n_suffix=[n_suffix], classes=[classes],
                  windows=windows, sinks=[[0] * Hkv], seg_tokens=[seg_tokens], n_decode=n_decode,
                  ring_decode=ring_decode)


def mixed_classes(seed: int = 1005, B: int = 8, lengths=(2048, 4096, 8192, 16384),
                  suffix_range=(128, 1024), seg_tokens: int = 2048, Hq: int = 32, Hkv: int = 8,
                  d: int = 128, P: int = 32, window: int = 256, theta: float = 1e6) -> Workload:
    """Batch of B sequences with context lengths drawn from `lengths`; per sequence a seeded
    permutation gives Hkv/4 KV heads to each class (global, local, retrieval, dense); the
    retrieval list is a seeded 25 % of context pages plus the last window plus the suffix
    pages; dense heads keep fresh K (no repositioning); suffixes ~ U{suffix_range}."""
    rng = np.random.default_rng(seed)
    ctx = [int(x) for x in rng.choice(np.asarray(lengths), size=B)]
    suf = [int(x) for x in rng.integers(suffix_range[0], suffix_range[1] + 1, size=B)]
    classes, windows = [], []
    per = max(1, Hkv // 4)
    for b in range(B):
        perm = rng.permutation(Hkv)
        cls = [0] * Hkv
        for i, h in enumerate(perm):
            cls[int(h)] = min(3, i // per)
        classes.append(cls)
        windows.append([window if c in (LOCAL,) else 0 for c in cls])
    return _build("mixed_classes", rng, B=B, Hq=Hq, Hkv=Hkv, d=d, P=P, theta=theta,
                  ctx_len=ctx, n_suffix=suf, classes=classes, windows=windows,
                  sinks=[[0] * Hkv for _ in range(B)], seg_tokens=[seg_tokens] * B,
                  retrieval_window=window)


def decode_batch_from(wl: Workload, step: int) -> AttnBatch:
    """The decode launch at `step` after a prefill workload built with n_decode > 0 whose
    decode tokens are stored in advance: one query per sequence at position seq_len + step."""
    if wl.ring is not None:
        raise ValueError("this workload appends its decode tokens: its tables change every step")
    a = wl.attn
    B = a.B
    return dataclasses.replace(
        a, q=np.ascontiguousarray(wl.decode_q[step]), cu_seqlens_q=np.arange(B + 1, dtype=np.int32),
        seq_len=(a.seq_len + step + 1).astype(np.int32), name=f"{a.name}_decode{step}")


def dense_listing(batch: AttnBatch, n_tokens) -> AttnBatch:
    """The same launch with every head listing every logical page below n_tokens[b] / P,
    for counting work: a window-only head that lists its whole window (as the page ring
    guarantees) has the same visible keys as with a full list."""
    B, Hkv, P = batch.B, batch.Hkv, batch.P
    n = np.repeat([_cdiv(int(x), P) for x in n_tokens], Hkv).astype(np.int32)
    mp = max(int(n.max()), 1)
    lg = np.tile(np.arange(mp, dtype=np.int32), (B * Hkv, 1))
    return dataclasses.replace(batch, page_logical=lg, page_table=np.zeros_like(lg), n_pages=n)


WORKLOADS = {
    "tiny_prefill": tiny_prefill,
    "decode_microbench": decode_microbench,
    "rag_prefill": rag_prefill,
    "stack_layer": stack_layer,
    "mixed_classes": mixed_classes,
}


@dataclasses.dataclass
class FfnWorkload:
    """Inputs of one sparse FFN call: token rows, importance scores and synthetic weights."""
    x: np.ndarray              # uint16 [T][d_model]
    importance: np.ndarray     # float32 [T]
    w_gate: np.ndarray         # uint16 [d_ff][d_model]
    w_up: np.ndarray           # uint16 [d_ff][d_model]
    w_down: np.ndarray         # uint16 [d_model][d_ff]
    keep: int


def sparse_ffn_workload(seed: int = 1006, T: int = 4096, d_model: int = 5120, d_ff: int = 25600,
                        keep_frac: float = 0.5, ties: bool = False) -> FfnWorkload:
    """Token rows x ~ N(0, 1), weights ~ N(0, 1/fan_in) (so that activations stay of order
    one), importance ~ LogNormal(0, 1) per token -- a stand-in for attention mass, which is
    positive and heavy-tailed; with `ties`, scores are rounded to 1/8 so that many are equal.
    Shapes default to the Qwen3-32B feed-forward block (d_model 5120, d_ff 25600) over a
    4096-token segment, half of it kept."""
    rng = np.random.default_rng(seed)
    x = _normal_bf16(rng, (T, d_model))
    w_gate = _normal_bf16(rng, (d_ff, d_model), scale=np.float32(1.0 / np.sqrt(d_model)))
    w_up = _normal_bf16(rng, (d_ff, d_model), scale=np.float32(1.0 / np.sqrt(d_model)))
    w_down = _normal_bf16(rng, (d_model, d_ff), scale=np.float32(1.0 / np.sqrt(d_ff)))
    imp = np.exp(rng.standard_normal(T)).astype(np.float32)
    if ties:
        imp = (np.round(imp * 8) / 8).astype(np.float32)
    return FfnWorkload(x=x, importance=imp, w_gate=w_gate, w_up=w_up, w_down=w_down, keep=int(round(keep_frac * T)))
