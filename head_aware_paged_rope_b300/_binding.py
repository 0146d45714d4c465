"""ctypes binding of librk (include/rk_api.h): argument marshalling only.

Every computation runs in the library's CUDA kernels; this module only turns torch
tensors into device pointers and sizes, allocates the caller-side workspace with torch
and raises on a non-OK status.  The library must have been built
(`python -m head_aware_paged_rope_b300.build`); importing this module without it fails.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "librk.so")

(RK_OK, RK_ERR_INVALID_ARG, RK_ERR_UNSUPPORTED, RK_ERR_CUDA, RK_ERR_DEVICE_BOUNDS, RK_ERR_TIMEOUT, RK_ERR_WORKSPACE,
 RK_ERR_DEVICE_ORDER) = range(8)
RK_CLASS_GLOBAL, RK_CLASS_LOCAL, RK_CLASS_RETRIEVAL, RK_CLASS_DENSE = range(4)
RK_ROPE_HALF_SPLIT, RK_ROPE_INTERLEAVED = 0, 1
RK_ATTN_METADATA_STABLE = 1
RK_ATTN_POOLS_STABLE = 2
RK_ATTN_DIAG_EXPIRE_WAIT = 1 << 30


class RkError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {status_string(code)} (status {code})")
        self.code = code


class RopeRun(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("src_tab_off", "src_tab_len", "dst_tab_off", "dst_tab_len", "pos_off0", "pos_on0", "n_tok", "reserved")]


class RopeArgs(ctypes.Structure):
    _fields_ = [
        ("k_src", ctypes.c_void_p), ("n_src_pages", ctypes.c_int64),
        ("k_dst", ctypes.c_void_p), ("n_dst_pages", ctypes.c_int64),
        ("src_tables", ctypes.c_void_p), ("n_src_entries", ctypes.c_int64),
        ("dst_tables", ctypes.c_void_p), ("n_dst_entries", ctypes.c_int64),
        ("runs", ctypes.c_void_p), ("n_runs", ctypes.c_int32), ("max_tok", ctypes.c_int32),
        ("P", ctypes.c_int32), ("d", ctypes.c_int32), ("theta", ctypes.c_double),
        ("style", ctypes.c_int32), ("status", ctypes.c_void_p),
    ]


class AttnArgs(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("cu_seqlens_q", ctypes.c_void_p), ("seq_len", ctypes.c_void_p),
        ("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p), ("n_pool_pages", ctypes.c_int64),
        ("page_table", ctypes.c_void_p), ("page_logical", ctypes.c_void_p), ("n_pages", ctypes.c_void_p),
        ("head_class", ctypes.c_void_p), ("window", ctypes.c_void_p), ("sink", ctypes.c_void_p),
        ("B", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32), ("d", ctypes.c_int32),
        ("P", ctypes.c_int32), ("max_pages", ctypes.c_int32), ("total_q", ctypes.c_int32), ("max_q", ctypes.c_int32),
        ("scale", ctypes.c_float), ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p), ("status", ctypes.c_void_p),
        ("flags", ctypes.c_int32), ("k_new", ctypes.c_void_p), ("v_new", ctypes.c_void_p),
        ("k_rot", ctypes.c_void_p), ("rot_coef", ctypes.c_void_p), ("n_rot", ctypes.c_int32),
        ("rot_style", ctypes.c_int32),
    ]


class AppendArgs(ctypes.Structure):
    _fields_ = [
        ("k_new", ctypes.c_void_p), ("v_new", ctypes.c_void_p), ("pos", ctypes.c_void_p),
        ("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p), ("n_pool_pages", ctypes.c_int64),
        ("page_table", ctypes.c_void_p), ("page_logical", ctypes.c_void_p), ("n_pages", ctypes.c_void_p),
        ("B", ctypes.c_int32), ("Hkv", ctypes.c_int32), ("d", ctypes.c_int32), ("P", ctypes.c_int32),
        ("max_pages", ctypes.c_int32), ("status", ctypes.c_void_p),
    ]


class RingArgs(ctypes.Structure):
    _fields_ = [
        ("pos", ctypes.c_void_p), ("page_table", ctypes.c_void_p), ("page_logical", ctypes.c_void_p),
        ("n_pages", ctypes.c_void_p), ("ring", ctypes.c_void_p), ("window", ctypes.c_void_p),
        ("sink", ctypes.c_void_p), ("B", ctypes.c_int32), ("Hkv", ctypes.c_int32), ("P", ctypes.c_int32),
        ("max_pages", ctypes.c_int32), ("status", ctypes.c_void_p),
        ("src_page_table", ctypes.c_void_p), ("src_page_logical", ctypes.c_void_p),
    ]


class SparseFfnArgs(ctypes.Structure):
    _fields_ = [
        ("x", ctypes.c_void_p), ("importance", ctypes.c_void_p), ("T", ctypes.c_int32), ("d_model", ctypes.c_int32),
        ("d_ff", ctypes.c_int32), ("keep", ctypes.c_int32), ("w_gate", ctypes.c_void_p), ("w_up", ctypes.c_void_p),
        ("w_down", ctypes.c_void_p), ("out", ctypes.c_void_p), ("kept", ctypes.c_void_p), ("status", ctypes.c_void_p),
    ]


def load_library(path: str = _LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"librk.so not built at {path}; run python -m head_aware_paged_rope_b300.build")
    lib = ctypes.CDLL(path)
    lib.rk_rope_workspace_size.restype = ctypes.c_size_t
    lib.rk_rope_workspace_size.argtypes = [ctypes.c_int32, ctypes.c_int32]
    lib.rk_rope_reposition.restype = ctypes.c_int
    lib.rk_rope_reposition.argtypes = [ctypes.POINTER(RopeArgs), ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    for name in ("rk_segpaged_prefill_workspace_size", "rk_segpaged_decode_workspace_size"):
        f = getattr(lib, name)
        f.restype = ctypes.c_size_t
        f.argtypes = [ctypes.POINTER(AttnArgs)]
    for name in ("rk_segpaged_prefill", "rk_segpaged_decode"):
        f = getattr(lib, name)
        f.restype = ctypes.c_int
        f.argtypes = [ctypes.POINTER(AttnArgs), ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    lib.rk_rope_coefficients.restype = ctypes.c_int
    lib.rk_rope_coefficients.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_double,
                                         ctypes.c_void_p, ctypes.c_void_p]
    lib.rk_append_kv.restype = ctypes.c_int
    lib.rk_append_kv.argtypes = [ctypes.POINTER(AppendArgs), ctypes.c_void_p]
    lib.rk_ring_advance.restype = ctypes.c_int
    lib.rk_ring_advance.argtypes = [ctypes.POINTER(RingArgs), ctypes.c_void_p]
    lib.rk_sparse_ffn_workspace_size.restype = ctypes.c_size_t
    lib.rk_sparse_ffn_workspace_size.argtypes = [ctypes.POINTER(SparseFfnArgs)]
    lib.rk_sparse_ffn.restype = ctypes.c_int
    lib.rk_sparse_ffn.argtypes = [ctypes.POINTER(SparseFfnArgs), ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    lib.rk_status_string.restype = ctypes.c_char_p
    lib.rk_status_string.argtypes = [ctypes.c_int]
    lib.rk_version.restype = ctypes.c_int32
    lib.rk_version.argtypes = []
    return lib


LIB = load_library()


def status_string(code: int) -> str:
    return LIB.rk_status_string(int(code)).decode()


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("librk takes device tensors")
    if not t.is_contiguous():
        raise ValueError("librk takes contiguous tensors")
    return t.data_ptr()


def _keep(struct, *tensors):
    """The struct holds raw device pointers: keep the tensors they point into alive as long as
    the struct is (a temporary tensor would otherwise be freed and its memory reused)."""
    struct._tensors = tuple(t for t in tensors if t is not None)
    return struct


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _workspace(nbytes: int, device, workspace: Optional[torch.Tensor], zeroed: bool = False) -> Optional[torch.Tensor]:
    if nbytes == 0:
        return workspace
    if workspace is not None:
        return workspace
    return (torch.zeros if zeroed else torch.empty)(nbytes, dtype=torch.uint8, device=device)


def _check(code: int, where: str) -> None:
    if code != RK_OK:
        raise RkError(code, where)


def rope_coefficients(deltas: torch.Tensor, d: int, theta: float, stream=None) -> torch.Tensor:
    """fp32 [n][d/2][4] coefficient rows of the turns by `deltas` (int32 device tensor)."""
    coef = torch.empty((deltas.numel(), d // 2, 4), dtype=torch.float32, device=deltas.device)
    _check(LIB.rk_rope_coefficients(_ptr(deltas), deltas.numel(), d, float(theta), _ptr(coef), _stream(stream)),
           "rk_rope_coefficients")
    return coef


def rope_workspace_size(n_runs: int, d: int) -> int:
    return int(LIB.rk_rope_workspace_size(n_runs, d))


def rope_reposition(k_src: torch.Tensor, k_dst: torch.Tensor, src_tables: torch.Tensor, dst_tables: torch.Tensor,
                    runs: torch.Tensor, *, max_tok: int, theta: float, style: int = RK_ROPE_HALF_SPLIT,
                    status: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                    stream=None) -> None:
    """k_src/k_dst: [pages][P][d] bf16 pools; src/dst_tables: int32; runs: int32 [n_runs][8]."""
    n_pages_src, P, d = k_src.shape
    a = RopeArgs(k_src=_ptr(k_src), n_src_pages=n_pages_src, k_dst=_ptr(k_dst), n_dst_pages=k_dst.shape[0],
                 src_tables=_ptr(src_tables), n_src_entries=src_tables.numel(), dst_tables=_ptr(dst_tables),
                 n_dst_entries=dst_tables.numel(), runs=_ptr(runs), n_runs=runs.shape[0], max_tok=int(max_tok),
                 P=P, d=d, theta=float(theta), style=int(style), status=_ptr(status))
    ws = _workspace(rope_workspace_size(runs.shape[0], d), k_src.device, workspace)
    nbytes = ws.numel() if ws is not None else 0
    _check(LIB.rk_rope_reposition(ctypes.byref(a), _ptr(ws), nbytes, _stream(stream)), "rk_rope_reposition")


def attn_args(q, seq_len, k_pool, v_pool, page_table, page_logical, n_pages, head_class, window, sink, out,
              *, cu_seqlens_q=None, lse=None, status=None, total_q: int, max_q: int, scale: float = 0.0,
              flags: int = 0, k_new=None, v_new=None, k_rot=None, rot_coef=None, rot_style: int = 0) -> AttnArgs:
    B = seq_len.shape[0]
    Hq, d = q.shape[1], q.shape[2]
    Hkv = n_pages.shape[0] // max(B, 1)
    return _keep(AttnArgs(q=_ptr(q), cu_seqlens_q=_ptr(cu_seqlens_q), seq_len=_ptr(seq_len), k_pool=_ptr(k_pool),
                    v_pool=_ptr(v_pool), n_pool_pages=k_pool.shape[0], page_table=_ptr(page_table),
                    page_logical=_ptr(page_logical), n_pages=_ptr(n_pages), head_class=_ptr(head_class),
                    window=_ptr(window), sink=_ptr(sink), B=B, Hq=Hq, Hkv=Hkv, d=d, P=k_pool.shape[1],
                    max_pages=page_table.shape[1], total_q=int(total_q), max_q=int(max_q), scale=float(scale),
                    out=_ptr(out), lse=_ptr(lse), status=_ptr(status), flags=int(flags), k_new=_ptr(k_new),
                    v_new=_ptr(v_new), k_rot=_ptr(k_rot), rot_coef=_ptr(rot_coef),
                    n_rot=0 if rot_coef is None else int(rot_coef.shape[0]), rot_style=int(rot_style)),
                 q, seq_len, k_pool, v_pool, page_table, page_logical, n_pages, head_class, window, sink, out,
                 cu_seqlens_q, lse, status, k_new, v_new, k_rot, rot_coef)


def segpaged_prefill_workspace_size(args: AttnArgs) -> int:
    return int(LIB.rk_segpaged_prefill_workspace_size(ctypes.byref(args)))


def segpaged_decode_workspace_size(args: AttnArgs) -> int:
    return int(LIB.rk_segpaged_decode_workspace_size(ctypes.byref(args)))


def segpaged_prefill(args: AttnArgs, *, device=None, workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    n = segpaged_prefill_workspace_size(args)
    ws = _workspace(n, device or torch.device("cuda"), workspace)
    _check(LIB.rk_segpaged_prefill(ctypes.byref(args), _ptr(ws), ws.numel() if ws is not None else 0,
                                   _stream(stream)), "rk_segpaged_prefill")


def segpaged_decode(args: AttnArgs, *, device=None, workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """A caller-owned `workspace` must be zero-filled before its first decode call; each call
    leaves its split counters at zero, so it can be reused by later decode calls."""
    n = segpaged_decode_workspace_size(args)
    ws = _workspace(n, device or torch.device("cuda"), workspace, zeroed=True)
    _check(LIB.rk_segpaged_decode(ctypes.byref(args), _ptr(ws), ws.numel() if ws is not None else 0,
                                  _stream(stream)), "rk_segpaged_decode")


def append_args(k_new, v_new, pos, k_pool, v_pool, page_table, page_logical, n_pages, *, status=None) -> AppendArgs:
    """k_new/v_new: bf16 [B][Hkv][d]; pos: int32 [B]; tables as for attention."""
    B, Hkv, d = k_new.shape
    return _keep(AppendArgs(k_new=_ptr(k_new), v_new=_ptr(v_new), pos=_ptr(pos), k_pool=_ptr(k_pool),
                            v_pool=_ptr(v_pool), n_pool_pages=k_pool.shape[0], page_table=_ptr(page_table),
                            page_logical=_ptr(page_logical), n_pages=_ptr(n_pages), B=B, Hkv=Hkv, d=d,
                            P=k_pool.shape[1], max_pages=page_table.shape[1], status=_ptr(status)),
                 k_new, v_new, pos, k_pool, v_pool, page_table, page_logical, n_pages, status)


def append_kv(args: AppendArgs, stream=None) -> None:
    _check(LIB.rk_append_kv(ctypes.byref(args), _stream(stream)), "rk_append_kv")


def ring_args(pos, page_table, page_logical, n_pages, ring, window, sink, *, Hkv: int, P: int,
              status=None, src_page_table=None, src_page_logical=None) -> RingArgs:
    """Tables [B*Hkv][max_pages] (several layers may be stacked as extra sequences); pos: int32 [B].
    With src_page_table / src_page_logical the lists are advanced from those tables into
    page_table / page_logical (out of place) instead of in place."""
    B = pos.shape[0]
    return _keep(RingArgs(pos=_ptr(pos), page_table=_ptr(page_table), page_logical=_ptr(page_logical),
                    n_pages=_ptr(n_pages), ring=_ptr(ring), window=_ptr(window), sink=_ptr(sink), B=B, Hkv=Hkv,
                    P=P, max_pages=page_table.shape[1], status=_ptr(status),
                    src_page_table=_ptr(src_page_table), src_page_logical=_ptr(src_page_logical)),
                 pos, page_table, page_logical, n_pages, ring, window, sink, status, src_page_table, src_page_logical)


def ring_advance(args: RingArgs, stream=None) -> None:
    _check(LIB.rk_ring_advance(ctypes.byref(args), _stream(stream)), "rk_ring_advance")


def sparse_ffn_args(x, importance, w_gate, w_up, w_down, out, kept, *, keep: int, status=None) -> SparseFfnArgs:
    """x: bf16 [T][d_model]; importance: fp32 [T]; w_gate/w_up: bf16 [d_ff][d_model];
    w_down: bf16 [d_model][d_ff]; out: bf16 [T][d_model]; kept: int32 [keep]."""
    T, d_model = x.shape
    return _keep(SparseFfnArgs(x=_ptr(x), importance=_ptr(importance), T=T, d_model=d_model, d_ff=w_gate.shape[0],
                         keep=int(keep), w_gate=_ptr(w_gate), w_up=_ptr(w_up), w_down=_ptr(w_down), out=_ptr(out),
                         kept=_ptr(kept), status=_ptr(status)),
                 x, importance, w_gate, w_up, w_down, out, kept, status)


def sparse_ffn(args: SparseFfnArgs, *, device=None, workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    n = int(LIB.rk_sparse_ffn_workspace_size(ctypes.byref(args)))
    ws = _workspace(n, device or torch.device("cuda"), workspace)
    _check(LIB.rk_sparse_ffn(ctypes.byref(args), _ptr(ws), ws.numel() if ws is not None else 0, _stream(stream)),
           "rk_sparse_ffn")


def version() -> int:
    return int(LIB.rk_version())
