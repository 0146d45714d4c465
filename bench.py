#!/usr/bin/env python3
"""Benchmark of the RoPE-repositioning + SegPagedAttention hot path on B300.

Workload (default): the 128K long-context layer stack -- 8 layers of 64 query / 8 KV
heads, head dim 128, page 16; context of 131072 tokens made of 32 reusable segments of
4096 tokens whose cached K is repositioned (RoPE) to its online offsets; a 1024-token
suffix prefill per layer; then 64 decode steps over all 8 layers, each appending its
token.  (layer, KV head) classes: exactly 3 of 64 global, the rest local with window 512,
which store only their window and reuse a ring of pages during the decode.  All inputs are seeded
synthetic bf16 N(0, 1) data (workloads/synth.py).

One step = for every layer: rk_rope_reposition, rk_segpaged_prefill; then 64 decode steps,
each: rk_ring_advance (all layers' page rings), then per layer rk_segpaged_decode, which
also stores the layer's new token.  The step is captured once in a CUDA graph and replayed.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  See the design notes for the field definitions.
"""
from __future__ import annotations

import argparse
import ctypes
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "SegPaged prefill TFLOP/s & decode KV-read GB/s on 1 B300, % of roofline"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=8)
    ap.add_argument("--decode-steps", type=int, default=64)
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-cases", action="store_true", help="skip the decode-microbenchmark and layer-prefill parts")
    ap.add_argument("--case", choices=["rag_prefill", "stack_prefill", "decode_microbench", "stack_decode", "rag_rope",
                                       "sparse_ffn"],
                    help="run one call of one workload --steps times (for profiling) instead of the step")
    ap.add_argument("--layer", type=int, default=None,
                    help="with --case stack_*: the layer (default: the first layer holding a global head)")
    return ap.parse_args()


def profiled_traffic(kernel):
    """DRAM bytes per launch of `kernel` from the ncu capture summarised in profiles/, or None
    when the kernel's sources have changed since (their SHA-256 is recorded with the figure)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        entry = json.load(f).get(kernel)
    if not entry:
        return None
    return entry["dram_bytes_per_launch"] if sources_digest(entry["sources"]) == entry["sources_sha256"] else None


def sources_digest(paths):
    """SHA-256 of the code of `paths` with comments and blank space removed (comment edits
    leave a measurement valid, code edits do not)."""
    import hashlib
    import re
    h = hashlib.sha256()
    for rel in paths:
        with open(os.path.join(ROOT, rel)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update(re.sub(r"\s+", " ", text).strip().encode())
    return h.hexdigest()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def workload_config(args):
    return {
        "workload": "stack128k: %d layers x (64 q / 8 KV heads, d 128, page 16), context 131072 = 32 segments x 4096 "
                    "repositioned, 1024-token suffix prefill, %d decode steps each appending its token; 3 of 64 "
                    "(layer, KV head) global, rest local window 512 storing only their window (page ring of 33 "
                    "pages in decode)" % (args.layers, args.decode_steps),
        "layers": args.layers, "context": 131072, "segments": 32, "segment_tokens": 4096, "suffix": 1024,
        "decode_steps": args.decode_steps, "Hq": 64, "Hkv": 8, "head_dim": 128, "page": 16, "theta": 1e6,
        "l2": "inputs larger than L2: each replayed step reads about 0.47 GB of distinct K/V and offline K "
              "(the decode windows, re-read every decode step, stay in L2 as in serving)",
        "parallelism": "replicas",
    }


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- distributed
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(torch, value, device, world):
    """The largest of a per-rank time over all ranks (the job's time is its slowest rank)."""
    if world <= 1:
        return float(value)
    t = torch.tensor([float(value)], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(work_per_rank, world, ms):
    """Whole-job rate: every rank processes `work_per_rank` units (weak scaling) in `ms`."""
    return work_per_rank * world / (ms * 1e-3)


# ----------------------------------------------------------------------------- reference arm
def _oracle_sample(layer_wl, n_queries, seed):
    """Rows (query token, KV head) sampled from a layer: n_queries spread tokens x all KV heads."""
    a = layer_wl.attn
    rng = np.random.default_rng(seed)
    toks = np.sort(rng.choice(a.total_q, size=min(n_queries, a.total_q), replace=False))
    return [(int(t), h) for t in toks for h in range(a.Hkv)]


def _sample_flops(batch, rows):
    from head_aware_paged_rope_b300 import roofline
    import dataclasses
    G = batch.Hq // batch.Hkv
    tot = 0
    cnt = roofline._visible_counts(batch, lambda b: [int(batch.seq_len[b]) - batch.total_q + t for t in range(batch.total_q)])
    for t, h in rows:
        tot += int(cnt[(0, h)][t])
    return 4 * batch.d * G * tot


def _blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        return int(max(n)) if n else os.cpu_count()
    except Exception:
        return os.cpu_count()


CPU_SAMPLE_QUERIES = 8      # query tokens of the oracle sample (x 8 KV heads)
CPU_SAMPLE_ROPE = 1024      # RoPE tokens of the oracle sample


def oracle_step(layer_wl, rows, n_rope_tok):
    """One bounded oracle pass: RoPE of one run prefix plus attention of the sampled rows."""
    from oracle import rk_oracle as O
    r = layer_wl.rope
    run = r.runs[:1].copy()
    run[0, 6] = min(int(run[0, 6]), n_rope_tok)
    t0 = time.perf_counter()
    O.paged_rope_reposition(r.k_src, r.src_tables, r.dst_tables, run, layer_wl.theta, r.P, r.style)
    O.segpaged_attention(layer_wl.attn, rows)
    return time.perf_counter() - t0


def cpu_sample(args):
    """The oracle's bounded sample of the workload, the same for the CPU baseline and the
    reference arm: a layer holding a global head, attention of CPU_SAMPLE_QUERIES spread
    query tokens x every KV head (each with its 8 query heads) over their visible keys, plus
    RoPE of CPU_SAMPLE_ROPE tokens of one run."""
    from workloads import synth
    classes = synth.stack_classes(n_layers=args.layers)
    layer = next((l for l, c in enumerate(classes) if 0 in c), 0)
    wl = synth.stack_layer(layer, n_layers=args.layers, n_decode=0)
    rows = _oracle_sample(wl, CPU_SAMPLE_QUERIES, 17)
    flops = _sample_flops(wl.attn, rows)
    text = (f"layer {layer} (holds a global head): attention of {CPU_SAMPLE_QUERIES} query tokens x 8 KV heads "
            f"(x 8 query heads each) over their visible keys, plus RoPE of {CPU_SAMPLE_ROPE} tokens of one run, "
            f"per step; value = sample attention FLOPs / oracle time")
    return wl, rows, flops, text


def cpu_baseline(args, steps):
    wl, rows, flops, text = cpu_sample(args)
    secs = [oracle_step(wl, rows, CPU_SAMPLE_ROPE) for _ in range(steps)]
    return {"value": flops * steps / sum(secs) / 1e12, "unit": UNIT, "cores": _blas_threads(), "kind": "oracle",
            "sample": text + f"; {steps} steps, {sum(secs):.1f} s"}


def reference_main(args, world, rank):
    if rank != 0:
        return 0
    wl, rows, flops, text = cpu_sample(args)
    for _ in range(args.warmup):
        oracle_step(wl, rows, CPU_SAMPLE_ROPE)
    times = [oracle_step(wl, rows, CPU_SAMPLE_ROPE) for _ in range(args.steps)]
    total = sum(times)
    value = flops * args.steps / total / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(args),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": _blas_threads(), "kind": "oracle",
                             "sample": text},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- our arm
class LayerState:
    """Device inputs, outputs and prebuilt C-ABI argument structs of one layer.  The decode
    tables of all layers live in one stack (`dec`) so one rk_ring_advance call per decode
    step advances every layer's page rings."""

    def __init__(self, rk, wl, dev, n_dec, torch, dec, layer):
        from workloads.device import attn_to_device, rope_to_device, to_device
        self.wl = wl
        a = wl.attn
        self.rope = rope_to_device(wl.rope, dev)
        self.attn = attn_to_device(a, dev)
        self.rope_ws = torch.empty(rk.rope_workspace_size(wl.rope.n_runs, a.d), dtype=torch.uint8, device=dev)
        rr = self.rope
        self.rope_args = rk.RopeArgs(
            k_src=rr.k_src.data_ptr(), n_src_pages=rr.k_src.shape[0], k_dst=self.attn.k_pool.data_ptr(),
            n_dst_pages=self.attn.k_pool.shape[0], src_tables=rr.src_tables.data_ptr(),
            n_src_entries=rr.src_tables.numel(), dst_tables=rr.dst_tables.data_ptr(),
            n_dst_entries=rr.dst_tables.numel(), runs=rr.runs.data_ptr(), n_runs=rr.runs.shape[0],
            max_tok=rr.max_tok, P=a.P, d=a.d, theta=rr.theta, style=rr.style, status=None)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.prefill_args = self.attn.args(rk, status=self.status)
        self.prefill_ws = torch.empty(max(1, rk.segpaged_prefill_workspace_size(self.prefill_args)), dtype=torch.uint8,
                                      device=dev)
        # decode step s: append the token at position seq_len + s, then one query there
        self.n_dec = n_dec
        self.dec_q = to_device(wl.decode_q[:n_dec].reshape(n_dec, a.Hq, a.d), dev)
        self.dec_k = to_device(wl.decode_k[:n_dec], dev)           # [n_dec][1][Hkv][d]
        self.dec_v = to_device(wl.decode_v[:n_dec], dev)
        self.dec_out = torch.empty((n_dec, a.Hq, a.d), dtype=torch.bfloat16, device=dev)
        self.dec_lse = torch.empty((n_dec, a.Hq), dtype=torch.float32, device=dev)
        nn = dec.n[layer]
        self.dec_args = []
        for s in range(n_dec):
            da = self.attn
            tab, lg = dec.tab[s % 2][layer], dec.lg[s % 2][layer]
            self.dec_args.append(rk.AttnArgs(
                q=self.dec_q[s].data_ptr(), cu_seqlens_q=None, seq_len=dec.seq[s].data_ptr(),
                k_pool=da.k_pool.data_ptr(), v_pool=da.v_pool.data_ptr(), n_pool_pages=da.k_pool.shape[0],
                page_table=tab.data_ptr(), page_logical=lg.data_ptr(), n_pages=nn.data_ptr(),
                head_class=da.head_class.data_ptr(), window=da.window.data_ptr(), sink=da.sink.data_ptr(), B=1,
                Hq=a.Hq, Hkv=a.Hkv, d=a.d, P=a.P, max_pages=tab.shape[1], total_q=1, max_q=1, scale=0.0,
                out=self.dec_out[s].data_ptr(), lse=self.dec_lse[s].data_ptr(), status=self.status.data_ptr(),
                flags=rk.RK_ATTN_METADATA_STABLE | rk.RK_ATTN_POOLS_STABLE, k_new=self.dec_k[s].data_ptr(),
                v_new=self.dec_v[s].data_ptr()))
        self.dec_ws = torch.zeros(max(1, rk.segpaged_decode_workspace_size(self.dec_args[0])), dtype=torch.uint8,
                                  device=dev)

    def host_inputs(self):
        d = self.attn
        return [self.rope.k_src, self.rope.src_tables, self.rope.dst_tables, self.rope.runs, d.q, d.cu_seqlens_q,
                d.seq_len, d.k_pool, d.v_pool, d.page_table, d.page_logical, d.n_pages, d.head_class, d.window,
                d.sink, self.dec_q, self.dec_k, self.dec_v]

    def host_outputs(self):
        return [self.attn.out, self.attn.lse, self.dec_out, self.dec_lse]


class DecodeTables:
    """The decode page tables of all layers, stacked as [layers][B*Hkv][max_pages] (layers
    as extra sequences of one rk_ring_advance call), twice: step s decodes on buffer s % 2,
    and before it the rings of step s + 1 are advanced out of place into the other buffer,
    so that no decode call waits for a table update.  Also their starting state (restored at
    the start of every replayed decode phase), the ring sizes, and per-step positions."""

    def __init__(self, rk, wls, dev, n_dec, torch):
        from workloads.device import to_device
        L = len(wls)
        a0 = wls[0].attn
        nseg = a0.B * a0.Hkv
        mp = max(int(w.dec_page_table.shape[1]) for w in wls)
        tab = np.full((L, nseg, mp), -1, np.int32)
        lg = np.full((L, nseg, mp), -1, np.int32)
        for l, w in enumerate(wls):
            tab[l, :, :w.dec_page_table.shape[1]] = w.dec_page_table
            lg[l, :, :w.dec_page_logical.shape[1]] = w.dec_page_logical
        self.tab0, self.lg0 = to_device(tab, dev), to_device(lg, dev)
        self.tab = torch.stack([self.tab0, self.tab0])       # [2][layers][B*Hkv][max_pages]
        self.lg = torch.stack([self.lg0, self.lg0])
        self.n = to_device(np.stack([w.dec_n_pages for w in wls]), dev)
        self.ring = to_device(np.concatenate([w.ring for w in wls]), dev)
        self.window = to_device(np.concatenate([w.attn.window for w in wls]), dev)
        self.sink = to_device(np.concatenate([w.attn.sink for w in wls]), dev)
        base = int(a0.seq_len[0])
        self.pos = torch.tensor([[base + s] * L for s in range(n_dec)], dtype=torch.int32, device=dev)
        self.seq = torch.tensor([[base + s + 1] for s in range(n_dec)], dtype=torch.int32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        flat = lambda t, i: t[i].view(L * nseg, mp)
        # step 0's rings, in place on buffer 0; then before step s, step s + 1's out of place
        self.ring_first = rk.ring_args(self.pos[0], flat(self.tab, 0), flat(self.lg, 0), self.n.view(-1), self.ring,
                                       self.window, self.sink, Hkv=a0.Hkv, P=a0.P, status=self.status)
        self.ring_next = [rk.ring_args(self.pos[s + 1], flat(self.tab, (s + 1) % 2), flat(self.lg, (s + 1) % 2),
                                       self.n.view(-1), self.ring, self.window, self.sink, Hkv=a0.Hkv, P=a0.P,
                                       status=self.status, src_page_table=flat(self.tab, s % 2),
                                       src_page_logical=flat(self.lg, s % 2)) for s in range(n_dec - 1)]

    def host_inputs(self):
        return [self.tab0, self.lg0, self.n, self.ring, self.window, self.sink, self.pos, self.seq]


def _call(fn, args_struct, ws, stream_handle):
    code = fn(ctypes.byref(args_struct), ctypes.c_void_p(ws.data_ptr()), ws.numel(), ctypes.c_void_p(stream_handle))
    if code != 0:
        raise RuntimeError(f"librk call failed with status {code}")


def _call2(fn, args_struct, stream_handle):
    code = fn(ctypes.byref(args_struct), ctypes.c_void_p(stream_handle))
    if code != 0:
        raise RuntimeError(f"librk call failed with status {code}")


def enqueue(rk, layers, dec, stream_handle, phase):
    """Enqueue one phase (or the whole step) through the C ABI; returns the number of our
    kernels it launches."""
    n = 0
    if phase in ("step", "rope", "prefill"):
        for L in layers:
            if phase in ("step", "rope"):
                _call(rk.LIB.rk_rope_reposition, L.rope_args, L.rope_ws, stream_handle)
                n += 2
            if phase in ("step", "prefill"):
                _call(rk.LIB.rk_segpaged_prefill, L.prefill_args, L.prefill_ws, stream_handle)
                n += 3
    if phase in ("step", "decode"):
        dec.tab.copy_(dec.tab0.unsqueeze(0).expand_as(dec.tab))   # the rings start from the state after
        dec.lg.copy_(dec.lg0.unsqueeze(0).expand_as(dec.lg))      # the prefill, in both buffers
        _call2(rk.LIB.rk_ring_advance, dec.ring_first, stream_handle)
        n += 1
        for s in range(layers[0].n_dec):
            if s + 1 < layers[0].n_dec:   # the next step's tables, while this step decodes
                _call2(rk.LIB.rk_ring_advance, dec.ring_next[s], stream_handle)
                n += 1
            for L in layers:   # each decode call first stores its layer's new token (k_new / v_new)
                _call(rk.LIB.rk_segpaged_decode, L.dec_args[s], L.dec_ws, stream_handle)
                # one kernel for up to 512 head segments (B * Hkv), else planner + attention + merge
                n += 1 if L.dec_args[s].B * L.dec_args[s].Hkv <= 512 else 3
    return n


def capture(torch, rk, layers, dec, phase, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        enqueue(rk, layers, dec, stream.cuda_stream, phase)      # eager warm-up (sets kernel attributes)
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=stream):
        n = enqueue(rk, layers, dec, torch.cuda.current_stream().cuda_stream, phase)
    torch.cuda.synchronize()
    return g, n


def time_graph(torch, g, stream, steps, warmup):
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def masked_dense_inputs(torch, batch, dev):
    """Dense K/V and explicit masks of a prefill launch, for the masked comparison path:
    per KV head h, K[h] / V[h] hold keys 0..L-1 gathered from the head's pages (every head
    must list every page below L), and mask[h][i][j] is True when key j is visible to
    query i (causal, and for a local head inside its window or its sink).  This is the
    form a dense attention kernel takes: the visible set as an attn_mask tensor.  Plumbing
    only -- built once, outside any timed region."""
    from workloads.device import to_device
    assert batch.B == 1, "one sequence"
    L, P, nq = int(batch.seq_len[0]), batch.P, batch.total_q
    j = torch.arange(L, device=dev)
    pos = (L - nq + torch.arange(nq, device=dev))[:, None]
    kp, vp = to_device(batch.k_pool, dev), to_device(batch.v_pool, dev)
    ks, vs, masks = [], [], []
    for h in range(batch.Hkv):
        lg = batch.page_logical[h, :int(batch.n_pages[h])]
        assert np.array_equal(lg, np.arange(len(lg))) and len(lg) * P >= L, "full page lists"
        pages = to_device(batch.page_table[h, :len(lg)].astype(np.int64), dev)
        rows = pages[j // P] * P + j % P
        ks.append(kp.view(-1, batch.d)[rows])
        vs.append(vp.view(-1, batch.d)[rows])
        m = j[None, :] <= pos
        if int(batch.head_class[h]) == 1:
            W, S = int(batch.window[h]), int(batch.sink[h])
            m &= (j[None, :] > pos - W) | (j[None, :] < S)
        masks.append(m)
    q = to_device(batch.q, dev)                                     # [nq][Hq][d]
    return q, ks, vs, masks


def masked_dense_sdpa(torch, q, ks, vs, masks, G, causal_only=False):
    """One prefill over dense K/V through torch's scaled_dot_product_attention, one call per
    KV head (its G query heads): with the explicit boolean mask (the masked path), or with
    is_causal and no mask (the unmasked fast path, every head treated as global)."""
    F = torch.nn.functional
    outs = []
    for h in range(len(ks)):
        qh = q[:, h * G:(h + 1) * G].transpose(0, 1)[None]           # [1][G][nq][d]
        kh, vh = ks[h][None, None].expand(1, G, -1, -1), vs[h][None, None].expand(1, G, -1, -1)
        if causal_only:   # queries at the end of the keys: the causal mask aligned to the lower right
            from torch.nn.attention.bias import causal_lower_right
            o = F.scaled_dot_product_attention(qh, kh, vh, attn_mask=causal_lower_right(qh.shape[2], kh.shape[2]))
        else:
            o = F.scaled_dot_product_attention(qh, kh, vh, attn_mask=masks[h][None, None])
        outs.append(o[0].transpose(0, 1))
    return torch.cat(outs, dim=1)                                     # [nq][Hq][d]


def time_masked_comparison(torch, rk, dev, steps, warmup):
    """The RAG prefill layer three ways: SegPagedAttention (our prefill over the page lists),
    the masked path (dense K/V + an attn_mask tensor per head through torch's
    scaled_dot_product_attention), and the unmasked fast path on the same dense K/V
    (is_causal, no mask, every head dense) -- the comparison the pages make between their
    mask-free kernel and a prefix cache that must pass a mask."""
    from head_aware_paged_rope_b300 import roofline
    from workloads import synth
    from workloads.device import attn_to_device
    wl = synth.rag_prefill()
    a = wl.attn
    G = a.Hq // a.Hkv
    q, ks, vs, masks = masked_dense_inputs(torch, a, dev)
    da = attn_to_device(a, dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    args = da.args(rk, status=st)
    ws = torch.empty(rk.segpaged_prefill_workspace_size(args), dtype=torch.uint8, device=dev)

    def t(fn, n):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    ms_seg = t(lambda: rk.segpaged_prefill(args, workspace=ws), max(steps, 10))
    ms_mask = t(lambda: masked_dense_sdpa(torch, q, ks, vs, masks, G), max(3, steps // 3))
    ms_flash = t(lambda: masked_dense_sdpa(torch, q, ks, vs, masks, G, causal_only=True), max(3, steps // 3))
    assert int(st.item()) == 0
    flops = roofline.attention_flops(a)
    return {"workload": "RAG layer (6 x 5000 context, 512-query suffix, 64 q / 8 KV heads, 1 global + 7 local W 256)",
            "segpaged_ms": ms_seg, "masked_dense_ms": ms_mask, "unmasked_dense_causal_ms": ms_flash,
            "masked_over_segpaged": ms_mask / ms_seg, "masked_over_unmasked": ms_mask / ms_flash,
            "segpaged_TFLOP/s": flops / (ms_seg * 1e-3) / 1e12,
            "masked_path": "torch scaled_dot_product_attention with a boolean attn_mask per KV head",
            "unmasked_path": "torch scaled_dot_product_attention is_causal=True on the same dense K/V"}


def time_sparse_ffn(torch, rk, dev, steps, warmup):
    """The token-level sparse FFN on the Qwen3-32B feed-forward block (d_model 5120, d_ff
    25600) over a 4096-token segment, half the tokens kept: selection, gather, and the two
    GEMMs.  FLOPs = 2 * keep * d_model * 3 d_ff (the three weight matrices)."""
    from workloads import synth
    from workloads.device import to_device
    w = synth.sparse_ffn_workload()
    x = to_device(w.x, dev)
    out = torch.empty_like(x)
    kept = torch.empty(w.keep, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    args = rk.sparse_ffn_args(x, torch.from_numpy(w.importance).to(dev), to_device(w.w_gate, dev),
                              to_device(w.w_up, dev), to_device(w.w_down, dev), out, kept, keep=w.keep, status=st)
    ws = torch.empty(int(rk.LIB.rk_sparse_ffn_workspace_size(ctypes.byref(args))), dtype=torch.uint8, device=dev)
    for _ in range(max(warmup, 3)):
        rk.sparse_ffn(args, workspace=ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = max(5, steps // 5)
    e0.record()
    for _ in range(n):
        rk.sparse_ffn(args, workspace=ws)
    e1.record()
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ms = e0.elapsed_time(e1) / n
    flops = 2 * w.keep * w.x.shape[1] * 3 * w.w_gate.shape[0]
    return {"workload": f"Qwen3-32B FFN block (d_model 5120, d_ff 25600), {len(w.importance)} tokens, {w.keep} kept",
            "ms": ms, "TFLOP/s": flops / (ms * 1e-3) / 1e12, "flops": flops}


def time_cases(torch, rk, dev, steps, warmup):
    """The decode microbenchmark (one call) and the isolated 128K layer prefill, each timed
    like `--case` (calls captured in a graph, pools rotated past L2)."""
    out = {}
    for case in ("decode_microbench", "stack_prefill"):
        calls, work, unit, label = build_case(torch, rk, dev, case, None)
        ms = time_calls(torch, dev, calls, max(steps, 10), max(warmup, 3))
        out[case] = {"ms": ms, unit: work / (ms * 1e-3), "workload": label, "pool_copies": len(calls)}
    return out


def ours_main(args, world, rank, local):
    import torch
    import head_aware_paged_rope_b300 as rk
    from head_aware_paged_rope_b300 import roofline
    from workloads import synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    peaks, peaks_src = load_peaks()

    t_gen = time.time()
    wls = [synth.stack_layer(l, n_layers=args.layers, n_decode=args.decode_steps) for l in range(args.layers)]
    flops_prefill = flops_decode = 0
    bytes_rope = bytes_decode = 0
    for wl in wls:
        flops_prefill += roofline.attention_flops(wl.attn)
        bytes_rope += roofline.rope_bytes(wl.rope)
        a = wl.attn
        for s in range(args.decode_steps):
            n_tok = a.seq_len + s + 1
            d = synth.dense_listing(dataclasses.replace(a, seq_len=n_tok.astype(np.int32),
                                                        cu_seqlens_q=np.arange(a.B + 1, dtype=np.int32)), n_tok)
            flops_decode += roofline.attention_flops(d)
            bytes_decode += roofline.decode_kv_bytes(d)
    dec = DecodeTables(rk, wls, dev, args.decode_steps, torch)
    layers = [LayerState(rk, wl, dev, args.decode_steps, torch, dec, l) for l, wl in enumerate(wls)]
    del wls
    torch.cuda.synchronize()
    t_gen = time.time() - t_gen

    stream = torch.cuda.Stream(device=dev)
    g_step, launches_per_step = capture(torch, rk, layers, dec, "step", stream)
    for L in layers:
        L.status.zero_()
    dec.status.zero_()
    # correctness guard: the device status word of every call must stay clear
    g_step.replay()
    torch.cuda.synchronize()
    bad = [int(L.status.item()) for L in layers if int(L.status.item()) != 0] + \
        ([int(dec.status.item())] if int(dec.status.item()) else [])
    if bad:
        raise RuntimeError(f"device status {bad}")

    sampler = ClockSampler(local)
    for _ in range(args.warmup):
        g_step.replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    ms_step = time_graph(torch, g_step, stream, args.steps, 0)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms_step = max_over_ranks(torch, ms_step, dev, world)

    # per-phase timing (each phase captured alone and replayed)
    parts = {}
    for phase in ("rope", "prefill", "decode"):
        g, n = capture(torch, rk, layers, dec, phase, stream)
        ms = time_graph(torch, g, stream, max(3, args.steps // 2), args.warmup)
        parts[phase] = {"ms": ms, "launches": n}
        del g
    parts["rope"].update({"GB/s": bytes_rope / (parts["rope"]["ms"] * 1e-3) / 1e9, "bytes": bytes_rope,
                          "calls": args.layers})
    parts["prefill"].update({"TFLOP/s": flops_prefill / (parts["prefill"]["ms"] * 1e-3) / 1e12, "flops": flops_prefill,
                             "calls": args.layers})
    parts["decode"].update({"GB/s": bytes_decode / (parts["decode"]["ms"] * 1e-3) / 1e9, "bytes": bytes_decode,
                            "TFLOP/s": flops_decode / (parts["decode"]["ms"] * 1e-3) / 1e12,
                            "calls": args.layers * args.decode_steps,
                            "note": "per step: one rk_ring_advance (all layers) that prepares the next step's "
                                    "tables in the other buffer, then per layer one rk_segpaged_decode that also "
                                    "stores the layer's new token (k_new / v_new)"})
    parts["rope"]["frac_hbm"] = parts["rope"]["GB/s"] / peaks["hbm_gbs"]
    parts["decode"]["frac_hbm"] = parts["decode"]["GB/s"] / peaks["hbm_gbs"]
    parts["prefill"]["frac_bf16_burst"] = parts["prefill"]["TFLOP/s"] / peaks["bf16_tflops"]
    parts["prefill"]["frac_bf16_sustained"] = parts["prefill"]["TFLOP/s"] / peaks["bf16_tflops_sustained"]
    if not args.no_cases:
        parts["masked_comparison"] = time_masked_comparison(torch, rk, dev, args.steps, args.warmup)
        parts["sparse_ffn"] = time_sparse_ffn(torch, rk, dev, args.steps, args.warmup)
        parts["sparse_ffn"]["frac_bf16_burst"] = parts["sparse_ffn"]["TFLOP/s"] / peaks["bf16_tflops"]
        for name, v in time_cases(torch, rk, dev, args.steps, args.warmup).items():
            if "GB/s" in v:
                v["frac_hbm"] = v["GB/s"] / peaks["hbm_gbs"]
            else:
                v["frac_bf16_burst"] = v["TFLOP/s"] / peaks["bf16_tflops"]
            parts[name] = v

    dom = max(("rope", "prefill", "decode"), key=lambda k: parts[k]["ms"])
    if dom == "prefill":
        roof = {"kernel": "prefill_tc_kernel (with its planner)", "bound": "tensor",
                "achieved": parts["prefill"]["TFLOP/s"], "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"}
        roof["traffic"] = None
    elif dom == "decode":
        # one decode_tc_kernel launch per rk_segpaged_decode call (up to 512 head segments):
        # achieved = algorithmic bytes per launch / average launch time in the replayed phase
        n_launch = parts["decode"]["calls"]
        roof = {"kernel": "decode_tc_kernel", "bound": "hbm", "achieved": parts["decode"]["GB/s"],
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "bytes_per_launch": bytes_decode / n_launch,
                "avg_launch_us": parts["decode"]["ms"] * 1e3 / n_launch}
        roof["traffic"] = profiled_traffic("decode_tc_kernel")
    else:
        roof = {"kernel": "rope_apply_kernel", "bound": "hbm", "achieved": parts["rope"]["GB/s"],
                "peak": peaks["hbm_gbs"], "unit": "GB/s"}
        roof["traffic"] = None
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["peak_source"] = peaks_src + (" (burst)" if roof["bound"] == "tensor" else " (copy)")

    step_flops = flops_prefill + flops_decode
    value = job_throughput(step_flops, world, ms_step) / 1e12

    # end to end from pinned host buffers: every input copied in and every output copied out
    # each step; "e2e" enqueues the step through the C ABI call by call, "e2e_graph" replays
    # the captured step between the copies
    e2e = e2e_graph = None
    if not args.no_e2e:
        ins, outs = [], []
        for t in [x for L in layers for x in L.host_inputs()] + dec.host_inputs():
            h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
            h.copy_(t)
            ins.append((t, h))
        for t in [x for L in layers for x in L.host_outputs()]:
            outs.append((t, torch.empty(t.shape, dtype=t.dtype, pin_memory=True)))
        h2d = sum(h.numel() * h.element_size() for _, h in ins)
        d2h = sum(h.numel() * h.element_size() for _, h in outs)

        def run_e2e(replay):
            with torch.cuda.stream(stream):
                for dt, ht in ins:
                    dt.copy_(ht, non_blocking=True)
                if replay:
                    g_step.replay()
                else:
                    enqueue(rk, layers, dec, stream.cuda_stream, "step")
                for dt, ht in outs:
                    ht.copy_(dt, non_blocking=True)

        res = {}
        for replay in (False, True):
            run_e2e(replay)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(args.e2e_steps):
                run_e2e(replay)
            e1.record(stream)
            torch.cuda.synchronize()
            ms = max_over_ranks(torch, e0.elapsed_time(e1) / args.e2e_steps, dev, world)
            res[replay] = {"value": job_throughput(step_flops, world, ms) / 1e12, "unit": UNIT,
                           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms,
                           "steps": args.e2e_steps}
        e2e, e2e_graph = res[False], res[True]
        e2e["how"] = "every rk_* call of the step enqueued through the C ABI (ctypes) between the copies"
        e2e_graph["how"] = "the captured step replayed between the copies"
        del ins, outs

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args, steps=2)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded bf16 N(0,1) K/V/q, seeded page "
                "permutations and head classes; no dataset)", "config": workload_config(args),
                "parts": parts, "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "e2e_graph": e2e_graph,
                "gpu_launches": launches_per_step * args.steps, "clocks": clocks,
                "setup_s": round(t_gen, 1)}
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def build_case(torch, rk, dev, case, layer):
    """Calls (closures, each one library call) of one workload, cycling through enough
    copies of the K/V pools that the visible bytes of consecutive calls exceed three times
    the L2, so they are not served from L2; and the work of one call."""
    from head_aware_paged_rope_b300 import roofline
    from workloads import synth
    from workloads.device import attn_to_device, rope_to_device, to_device
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    if case == "sparse_ffn":
        w = synth.sparse_ffn_workload()
        x = to_device(w.x, dev)
        out = torch.empty_like(x)
        kept = torch.empty(w.keep, dtype=torch.int32, device=dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        args = rk.sparse_ffn_args(x, torch.from_numpy(w.importance).to(dev), to_device(w.w_gate, dev),
                                  to_device(w.w_up, dev), to_device(w.w_down, dev), out, kept, keep=w.keep, status=st)
        ws = torch.empty(int(rk.LIB.rk_sparse_ffn_workspace_size(ctypes.byref(args))), dtype=torch.uint8, device=dev)
        flops = 2 * w.keep * w.x.shape[1] * 3 * w.w_gate.shape[0]
        return ([lambda: rk.sparse_ffn(args, workspace=ws), st], flops / 1e12, "TFLOP/s",
                "Qwen3-32B FFN block (d_model 5120, d_ff 25600), 4096 tokens, 2048 kept")
    classes = synth.stack_classes()
    glob_layer = next(l for l, c in enumerate(classes) if 0 in c)
    if case == "rag_prefill" or case == "rag_rope":
        wl, label = synth.rag_prefill(), "RAG layer (6 x 5000 context, 512-query suffix, 64 q / 8 KV heads)"
    elif case == "stack_prefill":
        layer = glob_layer if layer is None else layer
        wl = synth.stack_layer(layer, n_decode=0)
        label = f"128K stack layer {layer} prefill (1024 queries over 131072 + 1024 keys)"
    elif case == "decode_microbench":
        wl, label = synth.decode_microbench(), "decode microbenchmark (32 x 8192, 32 q / 8 KV heads, page 16)"
    elif case == "stack_decode":
        layer = glob_layer if layer is None else layer
        w = synth.stack_layer(layer, n_decode=1)
        a = w.attn
        wl = dataclasses.replace(w, attn=dataclasses.replace(
            a, q=np.ascontiguousarray(w.decode_q[0]), cu_seqlens_q=np.arange(a.B + 1, dtype=np.int32),
            seq_len=(a.seq_len + 1).astype(np.int32), page_table=w.dec_page_table, page_logical=w.dec_page_logical,
            n_pages=w.dec_n_pages))
        label = f"128K stack layer {layer}, first decode step"
    else:
        raise ValueError(case)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    calls = []
    if case == "rag_rope":
        dr = rope_to_device(wl.rope, dev)
        kp = to_device(wl.attn.k_pool, dev)
        ws = torch.empty(rk.rope_workspace_size(wl.rope.n_runs, wl.attn.d), dtype=torch.uint8, device=dev)
        calls.append(lambda: dr.run(rk, kp, status=st, workspace=ws))
        return calls, roofline.rope_bytes(wl.rope) / 1e9, "GB/s", label + ", RoPE"
    decode = case in ("decode_microbench", "stack_decode")
    da = attn_to_device(wl.attn, dev)
    base = da.args(rk, decode=decode, status=st,
                   flags=(rk.RK_ATTN_METADATA_STABLE | rk.RK_ATTN_POOLS_STABLE) if decode else 0)
    n = (rk.segpaged_decode_workspace_size if decode else rk.segpaged_prefill_workspace_size)(base)
    ws = torch.zeros(n, dtype=torch.uint8, device=dev)
    fn = rk.segpaged_decode if decode else rk.segpaged_prefill
    if decode:
        work, unit = roofline.decode_kv_bytes(wl.attn) / 1e9, "GB/s"
    else:
        work, unit = roofline.attention_flops(wl.attn) / 1e12, "TFLOP/s"
    touched = max(1, roofline.decode_kv_bytes(wl.attn))
    copies = max(1, min(8, -(-3 * l2 // touched)))
    keep = [da]
    for c in range(copies):
        a = rk.AttnArgs.from_buffer_copy(base)
        if c:
            kc, vc = da.k_pool.clone(), da.v_pool.clone()
            keep += [kc, vc]
            a.k_pool, a.v_pool = kc.data_ptr(), vc.data_ptr()
        calls.append(lambda a=a, keep=keep: fn(a, workspace=ws))
    calls.append(st)      # the status word, checked after timing
    return calls, work, unit, label


def time_calls(torch, dev, calls, steps, warmup):
    """Average time of one call: `steps` calls captured in a CUDA graph, replayed `steps`
    times after `warmup` replays, CUDA events on the replay stream."""
    st = calls[-1]
    calls = calls[:-1] if isinstance(st, torch.Tensor) else calls
    for i in range(warmup):
        calls[i % len(calls)]()
    torch.cuda.synchronize()
    stream = torch.cuda.Stream(device=dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(steps):
            calls[i % len(calls)]()
    for _ in range(max(1, warmup)):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    if isinstance(st, torch.Tensor):
        assert int(st.item()) == 0, f"device status {int(st.item())}"
    return e0.elapsed_time(e1) / (steps * steps)


def case_main(args):
    """One library call of one workload, repeated: a small, self-contained target for ncu."""
    import torch
    import head_aware_paged_rope_b300 as rk
    dev = torch.device("cuda", 0)
    calls, work, unit, label = build_case(torch, rk, dev, args.case, args.layer)
    ms = time_calls(torch, dev, calls, args.steps, args.warmup)
    print(json.dumps({"case": args.case, "workload": label, "ms_per_call": ms, unit: work / (ms * 1e-3),
                      "pool_copies": len(calls) - 1}), flush=True)
    return 0


def main():
    args = parse_args()
    world, rank, local = dist_setup(args)
    if args.case:
        return case_main(args)
    if args.impl == "reference":
        return reference_main(args, world, rank)
    return ours_main(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
