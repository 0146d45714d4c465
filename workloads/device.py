"""Upload synthetic workloads (workloads.synth) to device tensors.  Plumbing only."""
from __future__ import annotations

import dataclasses

import numpy as np
import torch


def to_device(a: np.ndarray, device) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


@dataclasses.dataclass
class DeviceAttn:
    q: torch.Tensor
    cu_seqlens_q: torch.Tensor
    seq_len: torch.Tensor
    k_pool: torch.Tensor
    v_pool: torch.Tensor
    page_table: torch.Tensor
    page_logical: torch.Tensor
    n_pages: torch.Tensor
    head_class: torch.Tensor
    window: torch.Tensor
    sink: torch.Tensor
    out: torch.Tensor
    lse: torch.Tensor
    total_q: int
    max_q: int

    def args(self, rk, decode: bool = False, status=None, use_logical: bool = True, flags: int = 0):
        return rk.attn_args(self.q, self.seq_len, self.k_pool, self.v_pool, self.page_table,
                            self.page_logical if use_logical else None, self.n_pages, self.head_class,
                            self.window, self.sink, self.out, cu_seqlens_q=None if decode else self.cu_seqlens_q,
                            lse=self.lse, status=status, total_q=self.total_q, max_q=1 if decode else self.max_q,
                            flags=flags)


def attn_to_device(batch, device, k_pool: torch.Tensor = None, v_pool: torch.Tensor = None) -> DeviceAttn:
    T, Hq, d = batch.q.shape
    return DeviceAttn(
        q=to_device(batch.q, device), cu_seqlens_q=to_device(batch.cu_seqlens_q, device),
        seq_len=to_device(batch.seq_len, device),
        k_pool=k_pool if k_pool is not None else to_device(batch.k_pool, device),
        v_pool=v_pool if v_pool is not None else to_device(batch.v_pool, device),
        page_table=to_device(batch.page_table, device), page_logical=to_device(batch.page_logical, device),
        n_pages=to_device(batch.n_pages, device), head_class=to_device(batch.head_class, device),
        window=to_device(batch.window, device), sink=to_device(batch.sink, device),
        out=torch.empty((T, Hq, d), dtype=torch.bfloat16, device=device),
        lse=torch.empty((T, Hq), dtype=torch.float32, device=device),
        total_q=int(batch.total_q), max_q=int(batch.max_q))


@dataclasses.dataclass
class DeviceRope:
    k_src: torch.Tensor
    src_tables: torch.Tensor
    dst_tables: torch.Tensor
    runs: torch.Tensor
    max_tok: int
    theta: float
    style: int

    def run(self, rk, k_dst: torch.Tensor, status=None, stream=None, workspace=None):
        rk.rope_reposition(self.k_src, k_dst, self.src_tables, self.dst_tables, self.runs, max_tok=self.max_tok,
                           theta=self.theta, style=self.style, status=status, stream=stream, workspace=workspace)


def rope_to_device(job, device) -> DeviceRope:
    return DeviceRope(k_src=to_device(job.k_src, device), src_tables=to_device(job.src_tables, device),
                      dst_tables=to_device(job.dst_tables, device), runs=to_device(job.runs, device),
                      max_tok=job.max_tok, theta=job.theta, style=job.style)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Device bf16 tensor -> numpy uint16 bit patterns."""
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)
