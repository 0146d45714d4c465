"""CPU-side checks of the C ABI: the library loads, exports every symbol the header
declares, and rejects bad arguments on the host before touching the GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rk_api.h")
LIB = os.path.join(ROOT, "head_aware_paged_rope_b300", "librk.so")


@pytest.fixture(scope="module")
def rk():
    from head_aware_paged_rope_b300 import build as b
    b.build()
    import head_aware_paged_rope_b300 as m
    return m


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"RK_API\s+[\w\s\*]+?\b(rk_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ("rk_rope_reposition", "rk_segpaged_prefill", "rk_segpaged_decode", "rk_rope_workspace_size",
              "rk_segpaged_prefill_workspace_size", "rk_segpaged_decode_workspace_size", "rk_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(rk):
    lib = ctypes.CDLL(LIB)
    for n in _declared():
        assert hasattr(lib, n), n


def test_status_strings(rk):
    assert rk.status_string(0) == "ok"
    assert "bounds" in rk.status_string(4)
    assert rk.status_string(99) == "unknown status"
    assert "ascending" in rk.status_string(7)


def _rope_args(rk, **kw):
    base = dict(k_src=1, n_src_pages=1, k_dst=1, n_dst_pages=1, src_tables=1, n_src_entries=1, dst_tables=1,
                n_dst_entries=1, runs=1, n_runs=1, max_tok=16, P=16, d=128, theta=1e6, style=0, status=None)
    base.update(kw)
    return rk.RopeArgs(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(d=96), 2), (dict(P=8), 2), (dict(style=3), 2), (dict(theta=1.0), 1), (dict(theta=float("nan")), 1),
    (dict(n_runs=-1), 1), (dict(max_tok=-5), 1), (dict(k_src=None), 1), (dict(runs=None), 1),
])
def test_rope_host_validation(rk, kw, code):
    a = _rope_args(rk, **kw)
    assert rk.LIB.rk_rope_reposition(ctypes.byref(a), None, 0, None) == code


def test_rope_nothing_to_do_and_workspace(rk):
    a = _rope_args(rk, n_runs=0)
    assert rk.LIB.rk_rope_reposition(ctypes.byref(a), None, 0, None) == 0
    a = _rope_args(rk)
    assert rk.LIB.rk_rope_reposition(ctypes.byref(a), None, 0, None) == 6          # workspace missing
    assert rk.rope_workspace_size(48, 128) == 48 * 64 * 16
    assert rk.rope_workspace_size(-1, 128) == 0


def _attn_args(rk, **kw):
    base = dict(q=1, cu_seqlens_q=1, seq_len=1, k_pool=1, v_pool=1, n_pool_pages=10, page_table=1, page_logical=None,
                n_pages=1, head_class=1, window=1, sink=None, B=2, Hq=8, Hkv=2, d=128, P=16, max_pages=4,
                total_q=10, max_q=5, scale=0.0, out=1, lse=None, status=None)
    base.update(kw)
    return rk.AttnArgs(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(Hq=6, Hkv=4), 1), (dict(d=80), 2), (dict(P=64), 2), (dict(Hq=64, Hkv=2), 2), (dict(Hq=24, Hkv=8), 2),
    (dict(B=-1), 1), (dict(max_q=11), 1), (dict(cu_seqlens_q=None), 1), (dict(q=None), 1), (dict(out=None), 1),
    (dict(scale=float("inf")), 1),
])
def test_prefill_host_validation(rk, kw, code):
    a = _attn_args(rk, **kw)
    assert rk.LIB.rk_segpaged_prefill(ctypes.byref(a), None, 0, None) == code


def test_decode_host_validation(rk):
    a = _attn_args(rk, cu_seqlens_q=None, total_q=2, max_q=1)
    assert rk.segpaged_decode_workspace_size(a) > 0
    assert rk.LIB.rk_segpaged_decode(ctypes.byref(a), None, 0, None) == 6           # workspace missing
    a = _attn_args(rk, cu_seqlens_q=None, total_q=3, max_q=1)                       # decode needs total_q == B
    assert rk.LIB.rk_segpaged_decode(ctypes.byref(a), None, 0, None) == 1


def test_attention_empty_batch_is_ok(rk):
    a = _attn_args(rk, B=0, total_q=0, max_q=0)
    assert rk.LIB.rk_segpaged_prefill(ctypes.byref(a), None, 0, None) == 0
    assert rk.segpaged_prefill_workspace_size(a) == 0


def test_workspace_size_grows_with_queries(rk):
    small = rk.segpaged_prefill_workspace_size(_attn_args(rk, total_q=10))
    big = rk.segpaged_prefill_workspace_size(_attn_args(rk, total_q=10000, max_q=5000))
    assert 0 < small < big


def test_unknown_flag_bits_are_rejected(rk):
    a = _attn_args(rk, flags=4)
    assert rk.LIB.rk_segpaged_prefill(ctypes.byref(a), None, 0, None) == 1
    d = _attn_args(rk, cu_seqlens_q=None, total_q=2, max_q=1, flags=rk.RK_ATTN_METADATA_STABLE | 4)
    assert rk.LIB.rk_segpaged_decode(ctypes.byref(d), None, 0, None) == 1
    d = _attn_args(rk, cu_seqlens_q=None, total_q=2, max_q=1, flags=rk.RK_ATTN_METADATA_STABLE)
    assert rk.LIB.rk_segpaged_decode(ctypes.byref(d), None, 0, None) == 6           # valid flag: workspace next
    d = _attn_args(rk, cu_seqlens_q=None, total_q=2, max_q=1, flags=rk.RK_ATTN_METADATA_STABLE | rk.RK_ATTN_POOLS_STABLE)
    assert rk.LIB.rk_segpaged_decode(ctypes.byref(d), None, 0, None) == 6
    d = _attn_args(rk, cu_seqlens_q=None, total_q=2, max_q=1, flags=rk.RK_ATTN_DIAG_EXPIRE_WAIT)
    assert rk.LIB.rk_segpaged_decode(ctypes.byref(d), None, 0, None) == 6           # the diagnostic bit is known


def test_decode_workspace_holds_the_zeroed_counter_prefix(rk):
    # the split tickets and ready flags (7 x 1024 int32 after a 256-byte header) come first
    for B, Hkv in ((1, 1), (32, 8), (1000, 8)):
        a = _attn_args(rk, cu_seqlens_q=None, B=B, Hq=8 * Hkv, Hkv=Hkv, total_q=B, max_q=1)
        assert rk.segpaged_decode_workspace_size(a) >= 256 + 4 * 7 * 1024


def test_decode_rejects_more_segments_than_supported(rk):
    a = _attn_args(rk, cu_seqlens_q=None, B=4096, Hq=64, Hkv=8, total_q=4096, max_q=1)   # 32768 segments
    assert rk.LIB.rk_segpaged_decode(ctypes.byref(a), ctypes.c_void_p(1 << 20), 1 << 30, None) == 2


def test_misaligned_pools_are_rejected_before_any_launch(rk):
    ws = ctypes.c_void_p(1 << 20)                                          # never dereferenced on the host
    a = _rope_args(rk, k_src=8)                                            # 8-byte aligned only
    assert rk.LIB.rk_rope_reposition(ctypes.byref(a), ws, 1 << 30, None) == 1
    p = _attn_args(rk, q=16, k_pool=24)
    assert rk.LIB.rk_segpaged_prefill(ctypes.byref(p), ws, 1 << 40, None) == 1


def test_missing_library_fails_loudly(tmp_path):
    # the binding has no CPU path: without librk.so it raises instead of computing anything
    import head_aware_paged_rope_b300._binding as B
    with pytest.raises(ImportError):
        B.load_library(str(tmp_path / "librk.so"))


def test_oracle_is_not_imported_by_the_product_path():
    import subprocess
    import sys
    code = ("import sys; sys.path.insert(0, %r); import head_aware_paged_rope_b300 as rk; rk.LIB; "
            "import head_aware_paged_rope_b300.roofline; "
            "assert not any(m == 'oracle' or m.startswith('oracle.') for m in sys.modules), 'oracle imported'" % ROOT)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_argument_structs_keep_their_tensors_alive(rk):
    # the structs hold raw pointers; every builder passes the tensors it points into to
    # _keep, which ties their lifetime to the struct's
    import inspect
    import weakref
    import head_aware_paged_rope_b300._binding as B

    class T:
        pass
    t = T()
    w = weakref.ref(t)
    s = B._keep(B.RingArgs(), t, None)
    del t
    assert w() is not None and s._tensors == (w(),)
    for f in (B.attn_args, B.append_args, B.ring_args, B.sparse_ffn_args):
        assert "return _keep(" in inspect.getsource(f)


def test_ring_advance_source_tables_both_or_neither_and_distinct(rk):
    # host validation only: the pointers are never dereferenced on the host
    a = rk.RingArgs(pos=1 << 20, page_table=2 << 20, page_logical=3 << 20, n_pages=4 << 20, ring=5 << 20,
                    window=6 << 20, B=1, Hkv=1, P=16, max_pages=4, src_page_table=7 << 20)
    assert rk.LIB.rk_ring_advance(ctypes.byref(a), None) == 1          # logical table missing
    a.src_page_logical = 2 << 20                                       # the destination page table
    assert rk.LIB.rk_ring_advance(ctypes.byref(a), None) == 1
    a.src_page_table, a.src_page_logical = 2 << 20, 8 << 20              # source = destination
    assert rk.LIB.rk_ring_advance(ctypes.byref(a), None) == 1
