"""Algorithmic work of one launch, for roofline reporting.

Conventions (counted on visible pairs only; masked work inside partial tiles is not
credited, exp is not counted):
  * attention FLOPs = 4 * d * (query head, visible key) pairs   (Q.K^T and P.V)
  * decode KV bytes = 2 * d * 2 bytes per visible key per KV head (K and V read once
    for all query heads of the group)
  * RoPE bytes      = 2 * d * 2 bytes per repositioned token row (read + write)
Visible sets follow include/rk_api.h: listed page, j < seq_len, j <= p, and for local
heads j > p - W or j < S.
"""
from __future__ import annotations

import numpy as np

LOCAL = 1


def _visible_counts(batch, positions_of_seq):
    """Per (sequence, KV head): array of visible-key counts for the given query positions."""
    out = {}
    P = batch.P
    for b in range(batch.B):
        L = int(batch.seq_len[b])
        pos = np.asarray(positions_of_seq(b), dtype=np.int64)
        for h in range(batch.Hkv):
            s = b * batch.Hkv + h
            n = int(batch.n_pages[s])
            listed = np.zeros(max(L, 1), dtype=np.int64)
            lp = np.asarray(batch.page_logical[s, :n], dtype=np.int64)
            for x in lp:
                lo, hi = x * P, min((x + 1) * P, L)
                if lo < hi:
                    listed[lo:hi] = 1
            csum = np.concatenate([[0], np.cumsum(listed)])           # csum[k] = listed in [0, k)
            upto = csum[np.clip(pos + 1, 0, L)]                         # listed j <= p (and < L)
            if int(batch.head_class[s]) == LOCAL:
                W, S = int(batch.window[s]), int(batch.sink[s])
                lo = np.clip(pos - W + 1, 0, L)                         # window [p-W+1, p]
                win = upto - csum[lo]
                sink_hi = np.minimum(np.minimum(S, lo), L)              # sink part below the window
                cnt = win + csum[np.clip(sink_hi, 0, L)]
            else:
                cnt = upto
            out[(b, h)] = cnt
    return out


def visible_pairs(batch) -> int:
    """(query head, visible key) pairs of a prefill/decode launch."""
    cu = np.asarray(batch.cu_seqlens_q)
    G = batch.Hq // batch.Hkv

    def pos(b):
        nq = int(cu[b + 1] - cu[b])
        L = int(batch.seq_len[b])
        return L - nq + np.arange(nq)

    return int(G * sum(int(c.sum()) for c in _visible_counts(batch, pos).values()))


def attention_flops(batch) -> int:
    return 4 * batch.d * visible_pairs(batch)


def decode_kv_bytes(batch) -> int:
    """K+V bytes of the visible keys of a decode launch (one query at seq_len-1)."""
    cnt = _visible_counts(batch, lambda b: [int(batch.seq_len[b]) - 1])
    return int(sum(int(c.sum()) for c in cnt.values())) * 2 * batch.d * 2


def rope_bytes(job) -> int:
    return int(job.total_tok) * job.d * 2 * 2
