"""The measurement counters used by bench.py agree with the oracle's explicit count."""
import dataclasses

import numpy as np

from head_aware_paged_rope_b300 import roofline
from oracle import rk_oracle as O
from workloads import synth


def test_pairs_match_oracle_tiny():
    a = synth.tiny_prefill().attn
    assert roofline.attention_flops(a) == O.attention_flops(a) == 9707520


def test_pairs_match_oracle_mixed_small():
    w = synth.mixed_classes(B=3, lengths=(512, 1024), suffix_range=(40, 90), seg_tokens=256)
    assert roofline.attention_flops(w.attn) == O.attention_flops(w.attn)


def test_pairs_match_oracle_local_sink():
    w = synth.decode_microbench(B=3, ctx=700, Hq=8, Hkv=4, window=50, sink=20)
    a = w.attn
    assert roofline.attention_flops(a) == O.attention_flops(a)
    # decode bytes: one query per sequence at seq_len - 1
    assert roofline.decode_kv_bytes(a) * 4 // 4 == O.attention_flops(a) // (4 * a.d * (a.Hq // a.Hkv)) * 2 * a.d * 2


def test_rope_bytes():
    w = synth.rag_prefill(n_segments=2, seg_tokens=100, n_suffix=10)
    assert roofline.rope_bytes(w.rope) == 2 * 8 * 100 * 128 * 4
