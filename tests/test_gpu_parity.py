"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the same
seeded inputs.

Tolerances (stated for this path):
  * RoPE-repositioned K: at most 1 bf16 ulp from the correctly rounded fp64 result.
  * attention output (bf16): max-abs error <= 3e-2 and relative L2 error <= 5e-3 over the
    compared rows; lse (fp32): abs error <= 1e-3 (fp32 accumulation of up to ~1.3e5
    exponentials whose relative error is below 1e-6).
  * everything that is index work (which rows are written, unchanged rows, page
    permutations) is compared bit for bit.
"""
import dataclasses
import math

import numpy as np
import pytest
import torch

from oracle import rk_oracle as O
from workloads import synth
from workloads.device import attn_to_device, bf16_bits, rope_to_device, to_device

# a decode workspace large enough for every call of these tests (G <= 16, d 128, one CTA per SM):
# counters, plan records and the partial and group slots of the work list
DEC_WS_BYTES = 1 << 25

pytestmark = pytest.mark.gpu

ATOL, RTOL_L2, LSE_TOL = 3e-2, 5e-3, 1e-3


@pytest.fixture(scope="module")
def rk():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from head_aware_paged_rope_b300 import build as b
    b.build()
    import head_aware_paged_rope_b300 as m
    return m


def _status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def _gpu_rope(rk, w, k_pool_bits=None):
    dr = rope_to_device(w.rope, "cuda")
    kp = to_device(w.attn.k_pool if k_pool_bits is None else k_pool_bits, "cuda")
    st = _status()
    dr.run(rk, kp, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return kp


def _check_rope(w, got_pool_bits):
    r = w.rope
    pages, slots, rows, inputs = O.paged_rope_reposition(r.k_src, r.src_tables, r.dst_tables, r.runs, w.theta, r.P,
                                                         r.style, return_inputs=True)
    got = got_pool_bits[pages, slots]
    ok = O.rope_within_one_ulp(got, rows, inputs, r.style)
    assert ok.all(), f"{(~ok).sum()} elements beyond 1 bf16 ulp"
    assert (got == O.f64_to_bf16(rows)).mean() > 0.999
    untouched = np.ones(got_pool_bits.shape[:2], dtype=bool)
    untouched[pages, slots] = False
    assert np.array_equal(got_pool_bits[untouched], w.attn.k_pool[untouched])
    return O.apply_rope_to_pool(w.attn.k_pool, (pages, slots, rows))


def _gpu_attn(rk, batch, decode=False, k_pool=None, use_logical=True, flags=0):
    da = attn_to_device(batch, "cuda", k_pool=k_pool)
    st = _status()
    args = da.args(rk, decode=decode, status=st, use_logical=use_logical, flags=flags)
    (rk.segpaged_decode if decode else rk.segpaged_prefill)(args)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return da.out.float().cpu().numpy(), da.lse.cpu().numpy()


def _compare(batch, out, lse, rows=None):
    ref = O.segpaged_attention(batch, rows)
    G = batch.Hq // batch.Hkv
    got_o, ref_o, got_l, ref_l = [], [], [], []
    for (t, h), (o, l) in ref.items():
        got_o.append(out[t, h * G:(h + 1) * G])
        ref_o.append(o)
        got_l.append(lse[t, h * G:(h + 1) * G])
        ref_l.append(l)
    go, ro = np.concatenate(got_o), np.concatenate(ref_o)
    gl, rl = np.concatenate(got_l), np.concatenate(ref_l)
    err = np.abs(go - ro)
    rel = np.linalg.norm(go - ro) / max(np.linalg.norm(ro), 1e-30)
    assert err.max() <= ATOL, f"max abs {err.max()}"
    assert rel <= RTOL_L2, f"rel L2 {rel}"
    fin = np.isfinite(rl)
    assert np.array_equal(fin, np.isfinite(gl))
    assert np.abs(gl[fin] - rl[fin]).max(initial=0.0) <= LSE_TOL
    return err.max(), rel


def _sample_rows(batch, seed, per_head=64):
    """All rows of one global and one local KV head, plus per_head random rows of every other head."""
    rng = np.random.default_rng(seed)
    T = batch.total_q
    cls = batch.head_class.reshape(batch.B, batch.Hkv)[0]
    full = set()
    for c in (O.GLOBAL, O.LOCAL):
        hs = np.nonzero(cls == c)[0]
        if len(hs):
            full.add(int(hs[0]))
    rows = [(t, h) for h in full for t in range(T)]
    for h in range(batch.Hkv):
        if h not in full:
            rows += [(int(t), h) for t in rng.choice(T, size=min(per_head, T), replace=False)]
    return rows


# ------------------------------------------------------------------------- RoPE
@pytest.mark.parametrize("style", [0, 1])
def test_rope_tiny(rk, style):
    w = synth.tiny_prefill(style=style)
    _check_rope(w, bf16_bits(_gpu_rope(rk, w)))


def test_rope_delta_zero_is_bit_exact(rk):
    w = synth.tiny_prefill()
    got = bf16_bits(_gpu_rope(rk, w))
    r = w.rope.runs[0]
    assert r[4] == r[5] == 0
    t = np.arange(int(r[6]))
    src = w.rope.k_src[w.rope.src_tables[r[0] + t // 16], t % 16]
    dst = got[w.rope.dst_tables[r[2] + t // 16], t % 16]
    assert np.array_equal(src, dst)


def test_rope_rag_full_size_unaligned(rk):
    w = synth.rag_prefill()          # 6 x 5000 tokens: runs start mid-page online
    _check_rope(w, bf16_bits(_gpu_rope(rk, w)))


def test_rope_mixed_d64_interleaved(rk):
    rng = np.random.default_rng(5)
    w = synth._build("m", rng, B=2, Hq=4, Hkv=4, d=64, P=32, theta=5e5, ctx_len=[700, 1300], n_suffix=[5, 9],
                     classes=[[0, 1, 2, 3]] * 2, windows=[[0, 64, 0, 0]] * 2, sinks=[[0] * 4] * 2,
                     seg_tokens=[333, 400], style=1)
    _check_rope(w, bf16_bits(_gpu_rope(rk, w)))


def test_rope_device_bounds_skip_only_bad_rows(rk):
    # run 0 gets a source page id outside the pool for its 4th table entry, run 1 an n_tok
    # above max_tok: both are reported; run 0's other rows and every other run are written
    w = synth.tiny_prefill()
    r = w.rope
    src_tables = r.src_tables.copy()
    runs = r.runs.copy()
    bad_entry = int(runs[0, 0]) + 3
    src_tables[bad_entry] = r.k_src.shape[0] + 5
    runs[1, 6] = r.max_tok + 1
    job = dataclasses.replace(r, src_tables=src_tables, runs=runs)
    dr = rope_to_device(job, "cuda")
    dr.max_tok = r.max_tok                           # the launch's bound stays 256
    kp = to_device(w.attn.k_pool, "cuda")
    st = _status()
    dr.run(rk, kp, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 4                       # RK_ERR_DEVICE_BOUNDS
    got = bf16_bits(kp)
    good = np.ones(len(runs), dtype=bool)
    good[1] = False
    pages, slots, rows, inputs = O.paged_rope_reposition(r.k_src, r.src_tables, r.dst_tables, r.runs[good], w.theta,
                                                         r.P, r.style, return_inputs=True)
    # rows of run 0 that read the bad source entry keep their old content
    n0 = int(r.runs[0, 6])
    t = np.arange(n0)
    bad = np.zeros(len(pages), dtype=bool)
    bad[:n0] = (int(r.runs[0, 4]) + t) // r.P == 3
    assert bad.sum() == r.P
    ok = O.rope_within_one_ulp(got[pages[~bad], slots[~bad]], rows[~bad], inputs[~bad], r.style)
    assert ok.all()
    assert np.array_equal(got[pages[bad], slots[bad]], w.attn.k_pool[pages[bad], slots[bad]])
    # run 1 (skipped whole) leaves its destination rows unchanged
    p1, s1, _ = O.paged_rope_reposition(r.k_src, r.src_tables, r.dst_tables, r.runs[1:2], w.theta, r.P, r.style)
    assert np.array_equal(got[p1, s1], w.attn.k_pool[p1, s1])


# ------------------------------------------------------------------------- prefill
def test_whole_path_tiny(rk):
    """GPU RoPE then GPU attention vs oracle RoPE (stored as bf16) then oracle attention."""
    w = synth.tiny_prefill()
    kp = _gpu_rope(rk, w)
    oracle_pool = _check_rope(w, bf16_bits(kp))
    out, lse = _gpu_attn(rk, w.attn, k_pool=kp)
    _compare(dataclasses.replace(w.attn, k_pool=oracle_pool), out, lse)


def test_prefill_rag_small_ragged(rk):
    w = synth.rag_prefill(n_segments=3, seg_tokens=1000, n_suffix=77)
    kp = _gpu_rope(rk, w)
    oracle_pool = _check_rope(w, bf16_bits(kp))
    out, lse = _gpu_attn(rk, w.attn, k_pool=kp)
    _compare(dataclasses.replace(w.attn, k_pool=oracle_pool), out, lse)


def test_prefill_mixed_small(rk):
    w = synth.mixed_classes(B=4, lengths=(1024, 2048), suffix_range=(50, 200), seg_tokens=512)
    out, lse = _gpu_attn(rk, w.attn)
    _compare(w.attn, out, lse)


def test_prefill_local_sink_and_window_one(rk):
    rng = np.random.default_rng(9)
    w = synth._build("s", rng, B=2, Hq=8, Hkv=4, d=128, P=16, theta=1e6, ctx_len=[300, 517], n_suffix=[33, 64],
                     classes=[[1, 1, 0, 2], [1, 3, 1, 1]], windows=[[1, 40, 0, 0], [17, 0, 256, 1000]],
                     sinks=[[3, 0, 0, 0], [20, 0, 5, 0]], seg_tokens=[128, 128])
    out, lse = _gpu_attn(rk, w.attn)
    _compare(w.attn, out, lse)


def test_prefill_without_logical_table(rk):
    """page_logical = NULL means entry e is logical page e (full lists)."""
    w = synth.rag_prefill(n_segments=2, seg_tokens=800, n_suffix=40, Hq=16, Hkv=4)
    out, lse = _gpu_attn(rk, w.attn, use_logical=False)
    _compare(w.attn, out, lse)


def test_prefill_empty_sequence_and_empty_list(rk):
    rng = np.random.default_rng(4)
    w = synth._build("e", rng, B=3, Hq=4, Hkv=2, d=64, P=16, theta=1e4, ctx_len=[100, 50, 80], n_suffix=[10, 0, 7],
                     classes=[[0, 1]] * 3, windows=[[0, 30]] * 3, sinks=[[0, 0]] * 3, seg_tokens=[64] * 3)
    a = w.attn
    n = a.n_pages.copy()
    n[1] = 0                                            # sequence 0, KV head 1 lists nothing
    a = dataclasses.replace(a, n_pages=n)
    out, lse = _gpu_attn(rk, a)
    _compare(a, out, lse)
    assert np.all(out[:10, 2:4] == 0) and np.all(np.isneginf(lse[:10, 2:4]))


def test_prefill_page_permutation_bit_identical(rk):
    w = synth.mixed_classes(B=2, lengths=(1024,), suffix_range=(60, 100), seg_tokens=512)
    a = w.attn
    out1, lse1 = _gpu_attn(rk, a)
    rng = np.random.default_rng(3)
    n = a.k_pool.shape[0]
    perm = rng.permutation(n)
    inv = np.empty(n, np.int64)
    inv[perm] = np.arange(n)
    b = dataclasses.replace(a, k_pool=a.k_pool[inv], v_pool=a.v_pool[inv],
                            page_table=np.where(a.page_table >= 0, perm[np.maximum(a.page_table, 0)], -1).astype(np.int32))
    out2, lse2 = _gpu_attn(rk, b)
    assert np.array_equal(out1, out2) and np.array_equal(lse1, lse2)


def test_prefill_device_bounds_check(rk):
    """A page id outside the pool is skipped and reported through the status word."""
    w = synth.tiny_prefill()
    a = w.attn
    tab = a.page_table.copy()
    tab[0, 3] = a.k_pool.shape[0] + 5
    da = attn_to_device(dataclasses.replace(a, page_table=tab), "cuda")
    st = _status()
    rk.segpaged_prefill(da.args(rk, status=st))
    torch.cuda.synchronize()
    assert int(st.item()) == 4


# ------------------------------------------------------------------------- decode
@pytest.mark.parametrize("flags", [0, 1, 3])
def test_decode_microbench_full_size(rk, flags):
    # flags 1: RK_ATTN_METADATA_STABLE (work planned before the preceding kernel completes);
    # 3: also RK_ATTN_POOLS_STABLE (the pools read before it completes)
    w = synth.decode_microbench()
    out, lse = _gpu_attn(rk, w.attn, decode=True, flags=flags)
    _compare(w.attn, out, lse)


def test_decode_small_ragged_sink(rk):
    w = synth.decode_microbench(B=5, ctx=2001, Hq=16, Hkv=4, window=100, sink=7)
    out, lse = _gpu_attn(rk, w.attn, decode=True)
    _compare(w.attn, out, lse)


def test_decode_d64_gqa2(rk):
    w = synth.tiny_prefill()
    a = synth.decode_batch_from(dataclasses.replace(w, decode_q=np.stack([w.attn.q[:1]] * 2)), 0)
    a = dataclasses.replace(a, seq_len=w.attn.seq_len.copy())
    out, lse = _gpu_attn(rk, a, decode=True)
    _compare(a, out, lse)


def test_decode_one_segment_over_every_cta(rk):
    # one global head over 70000 keys: its 547 key tiles are cut over the whole grid, so a
    # single segment has one partial per CTA and the merge runs over all of them
    w = synth.decode_microbench(B=1, ctx=70000, Hq=8, Hkv=1, window=256, sink=0)
    out, lse = _gpu_attn(rk, w.attn, decode=True, flags=rk.RK_ATTN_METADATA_STABLE)
    _compare(w.attn, out, lse)


@pytest.mark.parametrize("flags", [0, 1])
def test_decode_empty_lists_and_empty_context(rk, flags):
    # head segments with nothing visible: an empty page list, and a sequence of length 0
    w = synth.decode_microbench(B=4, ctx=900, Hq=16, Hkv=4, window=100, sink=4, seed=21)
    a = w.attn
    n = a.n_pages.copy()
    n[1] = 0                       # sequence 0, KV head 1
    n[9] = 0                       # sequence 2, KV head 1
    seq = a.seq_len.copy()
    seq[3] = 0                     # sequence 3: no context at all
    a = dataclasses.replace(a, n_pages=n, seq_len=seq)
    da = attn_to_device(a, "cuda")
    da.out.fill_(float("nan"))
    st = _status()
    rk.segpaged_decode(da.args(rk, decode=True, status=st, flags=flags))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    out, lse = da.out.float().cpu().numpy(), da.lse.cpu().numpy()
    G = a.Hq // a.Hkv
    for t, h in ((0, 1), (2, 1), (3, 0), (3, 3)):
        assert np.all(out[t, h * G:(h + 1) * G] == 0) and np.all(np.isneginf(lse[t, h * G:(h + 1) * G]))
    rows = [(t, h) for t in range(3) for h in range(a.Hkv)]
    _compare(a, out, lse, rows=rows)


def _last_query_decode(attn):
    """Decode batch from a prefill batch: each sequence's last suffix query, at seq_len - 1."""
    last = np.asarray(attn.cu_seqlens_q[1:]) - 1
    return dataclasses.replace(attn, q=np.ascontiguousarray(attn.q[last]),
                               cu_seqlens_q=np.arange(attn.B + 1, dtype=np.int32), name=attn.name + "_decode")


@pytest.mark.parametrize("flags", [0, 1])
def test_decode_mixed_classes_retrieval_and_dense(rk, flags):
    # every head class, retrieval heads listing a random subset of pages (the planner's
    # search falls back from its guesses), page 32
    w = synth.mixed_classes(B=4, lengths=(1024, 2048, 3000), suffix_range=(40, 90), seg_tokens=512)
    a = _last_query_decode(w.attn)
    out, lse = _gpu_attn(rk, a, decode=True, flags=flags)
    _compare(a, out, lse)


def test_decode_page32_d64(rk):
    w = synth.decode_microbench(B=5, ctx=2500, Hq=16, Hkv=4, d=64, P=32, window=200, sink=4, seed=31)
    out, lse = _gpu_attn(rk, w.attn, decode=True, flags=rk.RK_ATTN_METADATA_STABLE)
    _compare(w.attn, out, lse)


def test_prefill_page32_d64_mixed(rk):
    w = synth.mixed_classes(B=3, lengths=(1024, 2048), suffix_range=(50, 140), seg_tokens=512, Hq=16, Hkv=8, d=64,
                            P=32)
    out, lse = _gpu_attn(rk, w.attn)
    _compare(w.attn, out, lse)


def test_decode_many_segments_separate_planner(rk):
    # 576 head segments: more than every CTA plans for itself, so the separate planning and
    # merging kernels run
    w = synth.decode_microbench(B=72, ctx=700, Hq=32, Hkv=8, window=100, sink=4)
    out, lse = _gpu_attn(rk, w.attn, decode=True)
    _compare(w.attn, out, lse)


def test_decode_workspace_reused_across_shapes(rk):
    # one workspace, zeroed once, serves decode calls of different shapes and both schedules;
    # each call leaves its split counters at zero
    shapes = [dict(B=3, ctx=5000, Hq=32, Hkv=8, window=256, sink=4, seed=11),
              dict(B=72, ctx=700, Hq=32, Hkv=8, window=100, sink=4, seed=12),
              dict(B=1, ctx=30000, Hq=16, Hkv=1, window=64, sink=0, seed=13),
              dict(B=3, ctx=5000, Hq=32, Hkv=8, window=256, sink=4, seed=11)]
    batches = [synth.decode_microbench(**kw).attn for kw in shapes]
    devs = [attn_to_device(b, "cuda") for b in batches]
    st = _status()
    sizes = [rk.segpaged_decode_workspace_size(d.args(rk, decode=True, status=st)) for d in devs]
    ws = torch.zeros(max(sizes), dtype=torch.uint8, device="cuda")
    for flags in (0, rk.RK_ATTN_METADATA_STABLE):
        for b, d in zip(batches, devs):
            d.out.fill_(float("nan"))
            rk.segpaged_decode(d.args(rk, decode=True, status=st, flags=flags), workspace=ws)
            torch.cuda.synchronize()
            assert int(st.item()) == 0
            _compare(b, d.out.float().cpu().numpy(), d.lse.cpu().numpy())
            assert int(ws[256:28928].count_nonzero().item()) == 0


def _ring_decode_steps(rk, w, kp, k_host, check_steps, double_buffered=False):
    """Decode with appended tokens over window-only local heads, as the 128K stack runs it:
    per step rk_ring_advance and rk_segpaged_decode (which stores the new token itself) on
    the GPU, and the oracle's ring and append on the host; the outputs of `check_steps`
    are compared.  Double-buffered: step s decodes on buffer s % 2, and before it the
    tables of step s + 1 are advanced out of place into the other buffer."""
    a = w.attn
    st = _status()
    dev = {k: to_device(v, "cuda") for k, v in dict(tab=w.dec_page_table, lg=w.dec_page_logical, n=w.dec_n_pages,
                                                     ring=w.ring, window=a.window, sink=a.sink, cls=a.head_class,
                                                     vp=a.v_pool).items()}
    v_host = a.v_pool
    tab, lg = w.dec_page_table, w.dec_page_logical
    out = torch.empty((a.B, a.Hq, a.d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((a.B, a.Hq), dtype=torch.float32, device="cuda")
    ws = torch.zeros(DEC_WS_BYTES, dtype=torch.uint8, device="cuda")
    bufs = [(dev["tab"], dev["lg"]), (dev["tab"].clone(), dev["lg"].clone())]
    last = max(check_steps)
    for s in range(last + 1):
        pos = (a.seq_len + s).astype(np.int32)
        pos_d, seq_d = to_device(pos, "cuda"), to_device(pos + 1, "cuda")
        cur = bufs[s % 2] if double_buffered else bufs[0]
        if not double_buffered or s == 0:
            rk.ring_advance(rk.ring_args(pos_d, cur[0], cur[1], dev["n"], dev["ring"], dev["window"], dev["sink"],
                                         Hkv=a.Hkv, P=a.P, status=st))
        if double_buffered and s < last:
            nxt = bufs[(s + 1) % 2]
            rk.ring_advance(rk.ring_args(to_device(pos + 1, "cuda"), nxt[0], nxt[1], dev["n"], dev["ring"],
                                         dev["window"], dev["sink"], Hkv=a.Hkv, P=a.P, status=st,
                                         src_page_table=cur[0], src_page_logical=cur[1]))
        q = to_device(w.decode_q[s], "cuda")
        kn, vn = to_device(w.decode_k[s], "cuda"), to_device(w.decode_v[s], "cuda")
        rk.segpaged_decode(rk.attn_args(q, seq_d, kp, dev["vp"], cur[0], cur[1], dev["n"], dev["cls"],
                                        dev["window"], dev["sink"], out, lse=lse, status=st, total_q=a.B, max_q=1,
                                        flags=rk.RK_ATTN_METADATA_STABLE | rk.RK_ATTN_POOLS_STABLE, k_new=kn,
                                        v_new=vn), workspace=ws)
        tab, lg = O.ring_advance(tab, lg, w.dec_n_pages, w.ring, a.window, a.sink, pos, a.Hkv, a.P)
        k_host, v_host = O.append_rows(k_host, v_host, tab, lg, w.dec_n_pages, pos, w.decode_k[s], w.decode_v[s],
                                       a.Hkv, a.P)
        if s in check_steps:
            torch.cuda.synchronize()
            assert int(st.item()) == 0
            assert np.array_equal(cur[0].cpu().numpy(), tab) and np.array_equal(cur[1].cpu().numpy(), lg)
            gk, gv = bf16_bits(kp), bf16_bits(dev["vp"])
            for h in range(a.Hkv):                   # this step's rows, at the slots the host's tables give
                e = int(np.searchsorted(lg[h, :int(w.dec_n_pages[h])], int(pos[0]) // a.P))
                assert np.array_equal(gk[int(tab[h, e]), int(pos[0]) % a.P], w.decode_k[s][0, h])
                assert np.array_equal(gv[int(tab[h, e]), int(pos[0]) % a.P], w.decode_v[s][0, h])
            d = dataclasses.replace(a, q=w.decode_q[s], cu_seqlens_q=np.arange(a.B + 1, dtype=np.int32),
                                    seq_len=pos + 1, k_pool=k_host, v_pool=v_host, page_table=tab, page_logical=lg,
                                    n_pages=w.dec_n_pages)
            _compare(d, out.float().cpu().numpy(), lse.cpu().numpy())


@pytest.mark.parametrize("double_buffered", [False, True], ids=["in_place", "double_buffered"])
def test_stack_small_prefill_then_decode(rk, double_buffered):
    w = synth.stack_layer(0, n_segments=4, seg_tokens=1024, n_suffix=100, n_decode=40)
    kp = _gpu_rope(rk, w)
    oracle_pool = _check_rope(w, bf16_bits(kp))
    a = dataclasses.replace(w.attn, k_pool=oracle_pool)
    out, lse = _gpu_attn(rk, w.attn, k_pool=kp)
    _compare(a, out, lse)
    _ring_decode_steps(rk, w, kp, oracle_pool, (0, 17, 39), double_buffered)


def test_stack_small_prestored_decode(rk):
    # the same layer with every token stored in advance (no ring, no appends)
    w = synth.stack_layer(0, n_segments=4, seg_tokens=1024, n_suffix=100, n_decode=4, ring_decode=False)
    kp = _gpu_rope(rk, w)
    oracle_pool = _check_rope(w, bf16_bits(kp))
    a = dataclasses.replace(w.attn, k_pool=oracle_pool)
    for step in (0, 3):
        d = synth.decode_batch_from(dataclasses.replace(w, attn=a), step)
        out, lse = _gpu_attn(rk, d, decode=True, flags=rk.RK_ATTN_METADATA_STABLE, k_pool=kp)
        _compare(d, out, lse)


# ------------------------------------------------------------------------- full sizes, sampled rows
@pytest.mark.slow
def test_rag_prefill_full_size_sampled(rk):
    w = synth.rag_prefill()
    kp = _gpu_rope(rk, w)
    oracle_pool = _check_rope(w, bf16_bits(kp))
    out, lse = _gpu_attn(rk, w.attn, k_pool=kp)
    a = dataclasses.replace(w.attn, k_pool=oracle_pool)
    _compare(a, out, lse, rows=_sample_rows(a, 31))


@pytest.mark.slow
def test_mixed_full_size_sampled(rk):
    w = synth.mixed_classes()
    kp = _gpu_rope(rk, w)
    oracle_pool = _check_rope(w, bf16_bits(kp))
    out, lse = _gpu_attn(rk, w.attn, k_pool=kp)
    a = dataclasses.replace(w.attn, k_pool=oracle_pool)
    rng = np.random.default_rng(41)
    rows = [(int(t), h) for t in rng.choice(a.total_q, 300, replace=False) for h in range(a.Hkv)]
    _compare(a, out, lse, rows=rows)


@pytest.mark.slow
def test_stack_layer_full_size_sampled(rk):
    classes = synth.stack_classes()
    layer = next(l for l, c in enumerate(classes) if 0 in c)     # a layer holding a global head
    w = synth.stack_layer(layer)
    kp = _gpu_rope(rk, w)
    oracle_pool = _check_rope(w, bf16_bits(kp))
    a = dataclasses.replace(w.attn, k_pool=oracle_pool)
    out, lse = _gpu_attn(rk, w.attn, k_pool=kp)
    _compare(a, out, lse, rows=_sample_rows(a, 7, per_head=16))
    _ring_decode_steps(rk, w, kp, oracle_pool, (0, 31, 63), double_buffered=True)   # as the bench runs it


# ------------------------------------------------------------------------- group sizes and pairings
@pytest.mark.parametrize("Hq,Hkv", [(64, 4), (8, 8)], ids=["G16", "G1"])
def test_prefill_group_sizes(rk, Hq, Hkv):
    # G = 16 fills the decode MMA's N with no padding and gives 16-token prefill units;
    # G = 1 (one query head per KV head) gives 256-token units
    rng = np.random.default_rng(60 + Hkv)
    cls = [[0, 1, 2, 1, 3, 1, 1, 0][h] for h in range(Hkv)]
    w = synth._build("g", rng, B=2, Hq=Hq, Hkv=Hkv, d=128, P=16, theta=1e6, ctx_len=[700, 1900], n_suffix=[45, 300],
                     classes=[cls] * 2, windows=[[100 if c == 1 else 0 for c in cls]] * 2, sinks=[[0] * Hkv] * 2,
                     seg_tokens=[256, 512])
    kp = _gpu_rope(rk, w)
    oracle_pool = _check_rope(w, bf16_bits(kp))
    out, lse = _gpu_attn(rk, w.attn, k_pool=kp)
    _compare(dataclasses.replace(w.attn, k_pool=oracle_pool), out, lse)


@pytest.mark.parametrize("Hq,Hkv", [(64, 4), (8, 8)], ids=["G16", "G1"])
@pytest.mark.parametrize("flags", [0, 1])
def test_decode_group_sizes(rk, Hq, Hkv, flags):
    w = synth.decode_microbench(B=6, ctx=3333, Hq=Hq, Hkv=Hkv, window=256, sink=4, seed=70 + Hkv)
    out, lse = _gpu_attn(rk, w.attn, decode=True, flags=flags)
    _compare(w.attn, out, lse)


def test_rope_d128_interleaved(rk):
    rng = np.random.default_rng(17)
    w = synth._build("i", rng, B=2, Hq=8, Hkv=4, d=128, P=16, theta=1e6, ctx_len=[5000, 2100], n_suffix=[3, 7],
                     classes=[[0, 1, 2, 3]] * 2, windows=[[0, 64, 0, 0]] * 2, sinks=[[0] * 4] * 2,
                     seg_tokens=[1250, 700], style=1)
    _check_rope(w, bf16_bits(_gpu_rope(rk, w)))


# ------------------------------------------------------------------------- error paths on the device
def test_decode_bounded_wait_runs_out_and_the_workspace_recovers(rk):
    """RK_ATTN_DIAG_EXPIRE_WAIT makes the decode kernel's first CTA wait on a word nothing
    sets: the bounded wait (1 s) runs out, the call reports RK_ERR_TIMEOUT and every role
    of the kernel leaves -- no fault, no hang.  After the workspace is zeroed again, the
    next call on the same workspace is correct and leaves its counters at zero."""
    import time
    w = synth.decode_microbench(B=4, ctx=20000, Hq=32, Hkv=8, window=256, sink=4, seed=81)
    da = attn_to_device(w.attn, "cuda")
    st = _status()
    base = da.args(rk, decode=True, status=st)
    ws = torch.zeros(rk.segpaged_decode_workspace_size(base), dtype=torch.uint8, device="cuda")
    t0 = time.time()
    rk.segpaged_decode(da.args(rk, decode=True, status=st, flags=rk.RK_ATTN_DIAG_EXPIRE_WAIT), workspace=ws)
    torch.cuda.synchronize()
    assert int(st.item()) == 5                       # RK_ERR_TIMEOUT
    assert time.time() - t0 < 20
    ws.zero_()
    st.zero_()
    for flags in (0, rk.RK_ATTN_METADATA_STABLE):
        da.out.fill_(float("nan"))
        rk.segpaged_decode(da.args(rk, decode=True, status=st, flags=flags), workspace=ws)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        _compare(w.attn, da.out.float().cpu().numpy(), da.lse.cpu().numpy())
        assert int(ws[256:28928].count_nonzero().item()) == 0


def test_prefill_merge_wait_runs_out_and_the_next_call_is_correct(rk):
    """With RK_ATTN_DIAG_EXPIRE_WAIT the prefill kernel's merge of split query tiles waits for
    one stored piece more than a tile has: its bounded wait runs out (1 s after the last
    piece was taken), the call reports RK_ERR_TIMEOUT and the kernel ends -- no fault, no
    hang.  The next call on the same workspace, without the flag, is correct."""
    import time
    w = synth.rag_prefill(n_segments=3, seg_tokens=1000, n_suffix=77)
    da = attn_to_device(w.attn, "cuda")
    st = _status()
    base = da.args(rk, decode=False, status=st)
    ws = torch.zeros(rk.segpaged_prefill_workspace_size(base), dtype=torch.uint8, device="cuda")
    t0 = time.time()
    rk.segpaged_prefill(da.args(rk, decode=False, status=st, flags=rk.RK_ATTN_DIAG_EXPIRE_WAIT), workspace=ws)
    torch.cuda.synchronize()
    assert int(st.item()) == 5                       # RK_ERR_TIMEOUT
    assert time.time() - t0 < 20
    st.zero_()
    da.out.fill_(float("nan"))
    rk.segpaged_prefill(da.args(rk, decode=False, status=st), workspace=ws)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    _compare(w.attn, da.out.float().cpu().numpy(), da.lse.cpu().numpy())


def test_non_ascending_logical_list_is_reported(rk):
    """A page list whose logical pages do not ascend (here: last entry below the span its
    length needs) is reported as RK_ERR_DEVICE_ORDER by prefill and decode."""
    w = synth.mixed_classes(B=2, lengths=(1024,), suffix_range=(60, 100), seg_tokens=512)
    a = w.attn
    lg = a.page_logical.copy()
    n = int(a.n_pages[3])
    lg[3, n - 1] = lg[3, 0]                          # duplicate of the first logical page
    bad = dataclasses.replace(a, page_logical=lg)
    for decode in (False, True):
        b = _last_query_decode(bad) if decode else bad
        da = attn_to_device(b, "cuda")
        st = _status()
        (rk.segpaged_decode if decode else rk.segpaged_prefill)(da.args(rk, decode=decode, status=st))
        torch.cuda.synchronize()
        assert int(st.item()) == 7                   # RK_ERR_DEVICE_ORDER
