"""The masked-dense comparison path (a measurement, not a product path): dense K/V plus an
explicit attn_mask per KV head through torch's scaled_dot_product_attention.  It must
compute the same visible sets as SegPagedAttention -- checked against the fp64 oracle --
so that timing it against the mask-free kernel compares equal work ("小红书 RedKnot",
section 3, fourth component: a mask drops a prefix-cache kernel to its slow path)."""
import os
import sys

import numpy as np
import pytest
import torch

from oracle import rk_oracle as O
from workloads import synth

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402

pytestmark = pytest.mark.gpu


def _check(batch, out):
    ref = O.segpaged_attention(batch)
    G = batch.Hq // batch.Hkv
    go = np.concatenate([out[t, h * G:(h + 1) * G] for (t, h) in ref])
    ro = np.concatenate([v[0] for v in ref.values()])
    assert np.abs(go - ro).max() <= 3e-2
    assert np.linalg.norm(go - ro) <= 5e-3 * np.linalg.norm(ro)


def test_masked_dense_path_computes_the_visible_sets():
    w = synth.rag_prefill(n_segments=3, seg_tokens=700, n_suffix=60, Hq=16, Hkv=4)
    a = w.attn
    q, ks, vs, masks = bench.masked_dense_inputs(torch, a, torch.device("cuda"))
    out = bench.masked_dense_sdpa(torch, q, ks, vs, masks, a.Hq // a.Hkv)
    _check(a, out.float().cpu().numpy())


def test_unmasked_dense_path_is_causal_attention_over_every_key():
    w = synth.rag_prefill(n_segments=3, seg_tokens=700, n_suffix=60, Hq=16, Hkv=4)
    a = w.attn
    dense = synth.AttnBatch(**{**a.__dict__, "head_class": np.zeros_like(a.head_class)})
    q, ks, vs, masks = bench.masked_dense_inputs(torch, dense, torch.device("cuda"))
    out = bench.masked_dense_sdpa(torch, q, ks, vs, masks, a.Hq // a.Hkv, causal_only=True)
    _check(dense, out.float().cpu().numpy())
