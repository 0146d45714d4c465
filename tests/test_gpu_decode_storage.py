"""GPU checks of the decode-time storage calls through the C ABI: rk_append_kv against a
host scatter (bit for bit), rk_ring_advance against the oracle's ring (bit for bit, every
step), and decode over recycled pages against the fp64 oracle, with the new token stored
by rk_append_kv or by the decode call itself (k_new / v_new).

Pages follow "PagedAttention & RadixAttention" (slot pos % P of the page listed for
logical page pos / P); window-only local heads follow "小红书 RedKnot", section 3, first
and fourth components (a local head keeps only a window of KV)."""
import dataclasses

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


@pytest.mark.parametrize("d,P", [(128, 16), (64, 32)])
def test_append_kv_matches_host_scatter(rk, d, P):
    rng = np.random.default_rng(d + P)
    B, Hkv, n_pool, max_pages = 5, 4, 200, 9
    k_pool = rng.integers(0, 2 ** 16, size=(n_pool, P, d), dtype=np.uint16)
    v_pool = rng.integers(0, 2 ** 16, size=(n_pool, P, d), dtype=np.uint16)
    perm = rng.permutation(n_pool).astype(np.int32)
    tab = perm[: B * Hkv * max_pages].reshape(B * Hkv, max_pages).copy()
    # ascending logical pages per head segment; every head of sequence b lists page 3*b + 1
    lg = np.zeros((B * Hkv, max_pages), np.int32)
    n = rng.integers(3, max_pages + 1, size=B * Hkv).astype(np.int32)
    pos = np.zeros(B, np.int32)
    for b in range(B):
        common = 3 * b + 1
        for h in range(Hkv):
            s = b * Hkv + h
            others = rng.choice([x for x in range(40) if x != common], size=n[s] - 1, replace=False)
            lg[s, :n[s]] = np.sort(np.concatenate([others, [common]]))
            lg[s, n[s]:] = -1
        pos[b] = common * P + int(rng.integers(P))
    k_new = rng.integers(0, 2 ** 16, size=(B, Hkv, d), dtype=np.uint16)
    v_new = rng.integers(0, 2 ** 16, size=(B, Hkv, d), dtype=np.uint16)
    want_k, want_v = O.append_rows(k_pool, v_pool, tab, lg, n, pos, k_new, v_new, Hkv, P)
    dk, dv = to_device(k_pool, "cuda"), to_device(v_pool, "cuda")
    st = _status()
    a = rk.append_args(to_device(k_new, "cuda"), to_device(v_new, "cuda"), to_device(pos, "cuda"), dk, dv,
                       to_device(tab, "cuda"), to_device(lg, "cuda"), to_device(n, "cuda"), status=st)
    rk.append_kv(a)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.array_equal(bf16_bits(dk), want_k) and np.array_equal(bf16_bits(dv), want_v)


def test_append_kv_reports_an_unlisted_page_and_writes_nothing(rk):
    P, d = 16, 128
    tab = np.array([[3, 4], [5, 6]], np.int32)
    lg = np.array([[0, 1], [0, 2]], np.int32)
    n = np.array([2, 2], np.int32)
    pool = np.zeros((8, P, d), np.uint16)
    dk, dv = to_device(pool, "cuda"), to_device(pool, "cuda")
    new = to_device(np.full((1, 2, d), 7, np.uint16), "cuda")
    st = _status()
    # position 20 is on logical page 1: head 0 lists it (physical 4), head 1 does not
    rk.append_kv(rk.append_args(new, new, to_device(np.array([20], np.int32), "cuda"), dk, dv, to_device(tab, "cuda"),
                                to_device(lg, "cuda"), to_device(n, "cuda"), status=st))
    torch.cuda.synchronize()
    assert int(st.item()) == 4
    got = bf16_bits(dk)
    assert np.all(got[4, 4] == 7) and np.count_nonzero(got) == d


def _ring_workload(seed=5, n_decode=150):
    rng = np.random.default_rng(seed)
    return synth._build("ring", rng, B=2, Hq=16, Hkv=4, d=128, P=16, theta=1e6, ctx_len=[1000, 1536],
                        n_suffix=[100, 64], classes=[[0, 1, 1, 2], [1, 1, 0, 1]],
                        windows=[[0, 64, 200, 0], [33, 100, 0, 16]], sinks=[[0, 0, 4, 0], [0, 20, 0, 0]],
                        seg_tokens=[500, 512], n_decode=n_decode, ring_decode=True)


def _ring_args_dev(rk, wl, st):
    a = wl.attn
    dev = dict(tab=to_device(wl.dec_page_table, "cuda"), lg=to_device(wl.dec_page_logical, "cuda"),
               n=to_device(wl.dec_n_pages, "cuda"), ring=to_device(wl.ring, "cuda"),
               window=to_device(a.window, "cuda"), sink=to_device(a.sink, "cuda"))
    return dev


def test_ring_advance_matches_the_oracle_every_step(rk):
    wl = _ring_workload()
    a = wl.attn
    st = _status()
    dv = _ring_args_dev(rk, wl, st)
    tab, lg = wl.dec_page_table, wl.dec_page_logical
    for s in range(wl.decode_k.shape[0]):
        pos = (a.seq_len + s).astype(np.int32)
        tab, lg = O.ring_advance(tab, lg, wl.dec_n_pages, wl.ring, a.window, a.sink, pos, a.Hkv, a.P)
        rk.ring_advance(rk.ring_args(to_device(pos, "cuda"), dv["tab"], dv["lg"], dv["n"], dv["ring"], dv["window"],
                                     dv["sink"], Hkv=a.Hkv, P=a.P, status=st))
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert np.array_equal(dv["tab"].cpu().numpy(), tab) and np.array_equal(dv["lg"].cpu().numpy(), lg), s


def test_ring_advance_rejects_a_ring_still_in_the_window(rk):
    # a ring one page short of ceil(W/P) + 1: its oldest page is still in the new token's window
    wl = _ring_workload(n_decode=4)
    a = wl.attn
    st = _status()
    dv = _ring_args_dev(rk, wl, st)
    short = wl.ring.copy()
    s = int(np.nonzero(wl.ring)[0][0])
    n = wl.dec_n_pages.copy()
    n[s] -= 1                                     # drop the newest window page
    short[s] -= 1
    before = wl.dec_page_table.copy()
    pos = (a.seq_len + 0).astype(np.int32)
    pos[s // a.Hkv] = (int(wl.dec_page_logical[s, n[s] - 1]) + 1) * a.P   # the next page after the shorter list
    rk.ring_advance(rk.ring_args(to_device(pos, "cuda"), dv["tab"], dv["lg"], to_device(n, "cuda"),
                                 to_device(short, "cuda"), dv["window"], dv["sink"], Hkv=a.Hkv, P=a.P, status=st))
    torch.cuda.synchronize()
    assert int(st.item()) == 4
    assert np.array_equal(dv["tab"].cpu().numpy()[s], before[s])


def _check_appended(kp, vp, tab, lg, n_pages, pos, k_new, v_new, a):
    """The rows appended at this step sit, bit for bit, at the slots the host's tables give."""
    gk, gv = bf16_bits(kp), bf16_bits(vp)
    for b in range(a.B):
        for h in range(a.Hkv):
            s = b * a.Hkv + h
            e = int(np.searchsorted(lg[s, :int(n_pages[s])], int(pos[b]) // a.P))
            phys = int(tab[s, e])
            assert np.array_equal(gk[phys, int(pos[b]) % a.P], k_new[b, h])
            assert np.array_equal(gv[phys, int(pos[b]) % a.P], v_new[b, h])


def _compare(batch, out, lse, rows=None):
    ref = O.segpaged_attention(batch, rows)
    G = batch.Hq // batch.Hkv
    go = np.concatenate([out[t, h * G:(h + 1) * G] for (t, h) in ref])
    ro = np.concatenate([v[0] for v in ref.values()])
    gl = np.concatenate([lse[t, h * G:(h + 1) * G] for (t, h) in ref])
    rl = np.concatenate([v[1] for v in ref.values()])
    assert np.abs(go - ro).max() <= ATOL
    assert np.linalg.norm(go - ro) <= RTOL_L2 * np.linalg.norm(ro)
    assert np.abs(gl - rl).max() <= LSE_TOL


@pytest.mark.parametrize("fused", [False, True], ids=["append_kv", "k_new"])
@pytest.mark.parametrize("flags", [0, 1, 3])
def test_decode_with_appends_over_recycled_pages(rk, flags, fused):
    """RoPE (runs cut to what window-only heads store), prefill, then per step: ring
    advance, append, decode -- compared with the oracle at the first, a middle and the last
    step, on pools and tables the host evolves with the oracle's append and ring."""
    wl = _ring_workload()
    a = wl.attn
    st = _status()
    kp = to_device(a.k_pool, "cuda")
    rope_to_device(wl.rope, "cuda").run(rk, kp, status=st)
    r = wl.rope
    written = O.paged_rope_reposition(r.k_src, r.src_tables, r.dst_tables, r.runs, wl.theta, r.P, r.style)
    k_host = O.apply_rope_to_pool(a.k_pool, written)
    da = attn_to_device(a, "cuda", k_pool=kp)
    rk.segpaged_prefill(da.args(rk, status=st))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    _compare(dataclasses.replace(a, k_pool=k_host), da.out.float().cpu().numpy(), da.lse.cpu().numpy())
    dv = _ring_args_dev(rk, wl, st)
    v_host = a.v_pool
    tab, lg = wl.dec_page_table, wl.dec_page_logical
    n_dec = wl.decode_k.shape[0]
    seq = torch.empty(a.B, dtype=torch.int32, device="cuda")
    pos_d = torch.empty(a.B, dtype=torch.int32, device="cuda")
    out = torch.empty((a.B, a.Hq, a.d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((a.B, a.Hq), dtype=torch.float32, device="cuda")
    ws = torch.zeros(DEC_WS_BYTES, dtype=torch.uint8, device="cuda")
    for s in range(n_dec):
        pos = (a.seq_len + s).astype(np.int32)
        pos_d.copy_(torch.from_numpy(pos))
        seq.copy_(torch.from_numpy(pos + 1))
        rk.ring_advance(rk.ring_args(pos_d, dv["tab"], dv["lg"], dv["n"], dv["ring"], dv["window"], dv["sink"],
                                     Hkv=a.Hkv, P=a.P, status=st))
        kn, vn = to_device(wl.decode_k[s], "cuda"), to_device(wl.decode_v[s], "cuda")
        if not fused:
            rk.append_kv(rk.append_args(kn, vn, pos_d, kp, da.v_pool, dv["tab"], dv["lg"], dv["n"], status=st))
        q = to_device(wl.decode_q[s], "cuda")
        args = rk.attn_args(q, seq, kp, da.v_pool, dv["tab"], dv["lg"], dv["n"], da.head_class, da.window, da.sink,
                            out, lse=lse, status=st, total_q=a.B, max_q=1, flags=flags,
                            k_new=kn if fused else None, v_new=vn if fused else None)
        rk.segpaged_decode(args, workspace=ws)
        tab, lg = O.ring_advance(tab, lg, wl.dec_n_pages, wl.ring, a.window, a.sink, pos, a.Hkv, a.P)
        k_host, v_host = O.append_rows(k_host, v_host, tab, lg, wl.dec_n_pages, pos, wl.decode_k[s], wl.decode_v[s],
                                       a.Hkv, a.P)
        if s in (0, n_dec // 2, n_dec - 1):
            torch.cuda.synchronize()
            assert int(st.item()) == 0
            _check_appended(kp, da.v_pool, tab, lg, wl.dec_n_pages, pos, wl.decode_k[s], wl.decode_v[s], a)
            batch = dataclasses.replace(a, q=wl.decode_q[s], cu_seqlens_q=np.arange(a.B + 1, dtype=np.int32),
                                        seq_len=pos + 1, k_pool=k_host, v_pool=v_host, page_table=tab,
                                        page_logical=lg, n_pages=wl.dec_n_pages)
            _compare(batch, out.float().cpu().numpy(), lse.cpu().numpy())


# ------------------------------------------------------------------------- repositioning on load
@pytest.mark.parametrize("style", [0, 1])
def test_decode_repositions_on_load_bit_identically(rk, style):
    """Decode over the offline pages with their turn applied as they are read (k_rot with
    rk_rope_coefficients) gives, bit for bit, the output of rk_rope_reposition followed by
    decode over the repositioned pages; and it matches the oracle ("RedKnot" article, RoPE
    and SegPagedAttention paragraphs: cached K turned back and forward, pages read per head)."""
    layer = next(l for l, c in enumerate(synth.stack_classes()) if 0 in c)     # holds a global head
    wl = synth.stack_layer(layer, n_segments=5, seg_tokens=1024, n_suffix=100, n_decode=6)
    if style:
        wl.rope.style = 1
    a = wl.attn
    view = synth.reposition_on_load_view(wl)
    st = _status()
    # path A: reposition, then decode
    kp_a = to_device(a.k_pool, "cuda")
    rope_to_device(wl.rope, "cuda").run(rk, kp_a, status=st)
    # path B: the offline pages, turned on load
    kp_b = to_device(view.k_pool, "cuda")
    coef = rk.rope_coefficients(to_device(view.deltas, "cuda"), a.d, wl.theta)
    k_rot = to_device(view.dec_k_rot, "cuda")
    r = wl.rope
    written = O.paged_rope_reposition(r.k_src, r.src_tables, r.dst_tables, r.runs, wl.theta, r.P, r.style)
    k_host, v_host = O.apply_rope_to_pool(a.k_pool, written), a.v_pool
    paths = {}
    for name, kp in (("A", kp_a), ("B", kp_b)):
        dv = _ring_args_dev(rk, wl, st)
        vp = to_device(a.v_pool, "cuda")
        cls, win, sink = (to_device(x, "cuda") for x in (a.head_class, a.window, a.sink))
        ws = torch.zeros(DEC_WS_BYTES, dtype=torch.uint8, device="cuda")
        outs = []
        for s in range(wl.decode_k.shape[0]):
            pos = (a.seq_len + s).astype(np.int32)
            pos_d, seq = to_device(pos, "cuda"), to_device(pos + 1, "cuda")
            rk.ring_advance(rk.ring_args(pos_d, dv["tab"], dv["lg"], dv["n"], dv["ring"], dv["window"], dv["sink"],
                                         Hkv=a.Hkv, P=a.P, status=st))
            out = torch.empty((a.B, a.Hq, a.d), dtype=torch.bfloat16, device="cuda")
            lse = torch.empty((a.B, a.Hq), dtype=torch.float32, device="cuda")
            extra = dict(k_rot=k_rot, rot_coef=coef, rot_style=style) if name == "B" else {}
            rk.segpaged_decode(rk.attn_args(to_device(wl.decode_q[s], "cuda"), seq, kp, vp, dv["tab"], dv["lg"],
                                            dv["n"], cls, win, sink, out, lse=lse, status=st, total_q=a.B, max_q=1,
                                            flags=1, k_new=to_device(wl.decode_k[s], "cuda"),
                                            v_new=to_device(wl.decode_v[s], "cuda"), **extra), workspace=ws)
            outs.append((out, lse))
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        paths[name] = [(o.view(torch.int16).cpu().numpy(), l.cpu().numpy()) for o, l in outs]
    for (oa, la), (ob, lb) in zip(paths["A"], paths["B"]):
        assert np.array_equal(oa, ob) and np.array_equal(la, lb)
    # and against the oracle at the last step
    tab, lg = wl.dec_page_table, wl.dec_page_logical
    for s in range(wl.decode_k.shape[0]):
        pos = (a.seq_len + s).astype(np.int32)
        tab, lg = O.ring_advance(tab, lg, wl.dec_n_pages, wl.ring, a.window, a.sink, pos, a.Hkv, a.P)
        k_host, v_host = O.append_rows(k_host, v_host, tab, lg, wl.dec_n_pages, pos, wl.decode_k[s], wl.decode_v[s],
                                       a.Hkv, a.P)
    batch = dataclasses.replace(a, q=wl.decode_q[s], cu_seqlens_q=np.arange(a.B + 1, dtype=np.int32), seq_len=pos + 1,
                                k_pool=k_host, v_pool=v_host, page_table=tab, page_logical=lg, n_pages=wl.dec_n_pages)
    ob, lb = paths["B"][-1]
    _compare(batch, ob.view(np.uint16).astype(np.uint32).__lshift__(16).view(np.float32), lb)


def test_prefill_rejects_repositioning_on_load(rk):
    w = synth.tiny_prefill()
    from workloads.device import attn_to_device
    da = attn_to_device(w.attn, "cuda")
    coef = torch.zeros((1, 32, 4), dtype=torch.float32, device="cuda")
    k_rot = torch.full(tuple(w.attn.page_table.shape), -1, dtype=torch.int32, device="cuda")
    args = da.args(rk)
    args.k_rot, args.rot_coef, args.n_rot = k_rot.data_ptr(), coef.data_ptr(), 1
    with pytest.raises(rk.RkError) as e:
        rk.segpaged_prefill(args)
    assert e.value.code == 2
