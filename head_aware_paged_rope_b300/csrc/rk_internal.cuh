// Internal declarations shared by the librk CUDA sources (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "rk_api.h"

namespace rk {

// ------------------------------------------------------------------ device error word
__device__ __forceinline__ void report(int32_t* status, int32_t code) {
  if (status) atomicCAS(status, 0, code);
}

// ------------------------------------------------------------------ bf16 helpers
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float y;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
  return y;
}

__device__ __forceinline__ float fast_log2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------------------ RoPE turn of one channel pair
// (xa, xb) turned by the angle whose cos / sin are split into a head with 16 significant bits
// and an fp32 tail, cf = (c_hi, c_lo, s_hi, s_lo): for bf16 inputs the head products are exact
// in fp32, so the result carries only the final fp32 rounding even when the products cancel.
// Used by the RoPE kernel and by the attention kernels that turn K as they read it, so both
// produce the same bf16 values.
__device__ __forceinline__ void rotate_pair(float xa, float xb, const float4& cf, float& ya, float& yb) {
  const float hi_a = fmaf(xa, cf.x, -(xb * cf.z));   // xa*c_hi - xb*s_hi (both products exact)
  const float lo_a = fmaf(xa, cf.y, -(xb * cf.w));
  const float hi_b = fmaf(xa, cf.z, xb * cf.x);      // xa*s_hi + xb*c_hi
  const float lo_b = fmaf(xa, cf.w, xb * cf.y);
  ya = hi_a + lo_a;
  yb = hi_b + lo_b;
}

// ------------------------------------------------------------------ attention work list
// A unit is one (head segment, query tile): the queries [tok0, tok0+ntok) of one sequence
// against one KV head.  Its visible page-list entries form at most two ranges (sink pages
// [0, e_sink) and window/causal pages [e_w, e_w + n_vis - e_sink)); a virtual index v in
// [0, n_vis) walks both.  An item is a contiguous slice [v_begin, v_end) of one unit.
struct Unit {
  int32_t seg;        // b * Hkv + h
  int32_t tok0;       // first query token (row of q)
  int32_t ntok;       // queries in the tile
  int32_t pos0;       // position of query tok0
  int32_t e_sink;     // entries [0, e_sink) are the sink range
  int32_t e_w;        // first entry of the second range
  int32_t n_vis;      // entries to visit
  int32_t n_splits;   // items of this unit
  int32_t first_item; // index of its first full-size item (they are consecutive)
  int32_t b;          // sequence
  int32_t n_full;     // full-size chunks
  int32_t rem_item;   // planner scratch (-1 once planned)
};

struct Item {
  int32_t unit;
  int32_t v_begin;
  int32_t v_end;
  int32_t split;
};

struct PlanHeader {
  int32_t n_units;
  int32_t n_items;
  int32_t chunk;      // entries per split
  int32_t counter;    // dynamic work counter (reset by the planner)
  int32_t n_split;    // units with more than one item (listed in split_list)
  int32_t merge_counter;   // merge jobs taken (reset by the planner)
  int32_t pad[58];
};

// Item index of split s of a unit (the items of a unit are consecutive).
__device__ __forceinline__ int32_t unit_item(const Unit& u, int32_t s) { return u.first_item + s; }

__device__ __forceinline__ int32_t unit_entry(const Unit& u, int32_t v) {
  return v < u.e_sink ? v : u.e_w + (v - u.e_sink);
}

// Parameters common to the attention kernels (copied from rk_attn_args + derived values).
struct AttnParams {
  const __nv_bfloat16* q;
  const int32_t* cu_seqlens_q;
  const int32_t* seq_len;
  const __nv_bfloat16* k_pool;
  const __nv_bfloat16* v_pool;
  int64_t n_pool_pages;
  const int32_t* page_table;
  const int32_t* page_logical;
  const int32_t* n_pages;
  const int32_t* head_class;
  const int32_t* window;
  const int32_t* sink;
  int32_t B, Hq, Hkv, d, P, max_pages, total_q, max_q;
  int32_t G;           // Hq / Hkv
  int32_t tok_per_unit;
  float scale_log2;    // softmax scale * log2(e)
  __nv_bfloat16* out;
  float* lse;
  int32_t* status;
  int32_t flags;       // RK_ATTN_* bits
  const __nv_bfloat16* k_new;   // decode: the new token's K / V per head segment, or null
  const __nv_bfloat16* v_new;
  const int32_t* k_rot;         // per listed entry: coefficient row of its K turn, -1 none; or null
  const float4* rot_coef;       // [n_rot][d/2] (c_hi, c_lo, s_hi, s_lo)
  int32_t n_rot;
  int32_t rot_style;
};

// Workspace carve-up for the attention calls.
struct AttnWorkspace {
  PlanHeader* header;
  Unit* units;
  Item* items;
  float* part_lse;     // [max_items][rows]
  float* part_o;       // [max_items][rows][d]
  int32_t* unit_done;  // [max_units] softmax warps that stored their rows of a partial (8 per item)
  int32_t* split_list; // [max_units] the units with more than one item, in unit order
  int32_t max_units;
  int32_t max_items;
  int32_t rows;        // rows per unit (query tile rows)
};

constexpr int kTargetItems = 2048;   // upper bound on items beyond one per unit
// Prefill items: about kItemsPerCta per CTA, each at least kMinChunkTiles key tiles (finer
// items balance the CTAs; each item also costs a start, an epilogue and a partial to merge).
constexpr int kItemsPerCta = 8;
constexpr int kMinChunkTiles = 12;

// ------------------------------------------------------------------ decode work list
// Decode is scheduled stream-K style: the key tiles (128 keys) of all head segments are
// concatenated, segment after segment, and CTA c of the decode grid takes the equal share
// [c*T/gs, (c+1)*T/gs) of the T tiles (gs = min(grid, T); further CTAs get none).  A segment whose tiles fall to several CTAs is
// "split": each CTA writes a normalised partial result into its slot and
// combine_decode_tc_kernel merges them.  plan_decode_kernel (rk_plan.cu) writes:
struct DecSeg {
  int32_t e_sink, e_w, n_vis, n_tiles;      // visible entry ranges (see Unit) and key tiles
  int32_t tile0;                            // first tile of the segment in the global sequence
  int32_t slot0;                            // first partial slot (split segments only)
  int32_t cta0;                             // first CTA whose share touches the segment
  int32_t n_splits;                         // CTAs that touch it (1: written directly)
  int32_t b, tok, pos, cls;                 // sequence, query row, query position, head class
  int32_t W, S, L, pad;                     // window, sink, context length
};

struct DecCta {
  int32_t seg0;          // segment holding the first tile of the share (B*Hkv if none)
  int32_t tile_begin, tile_end, pad;
};

struct DecHeader {
  int32_t total_tiles;
  int32_t n_split;       // split segments, listed in DecWorkspace::split_segs
  int32_t grid;          // CTAs of the decode kernel the shares were cut for
  int32_t pad[61];
};

struct DecWorkspace {
  DecHeader* header;
  int32_t* counters;     // [7 * kDecMaxGrid], zero between calls (single-launch path): merge tickets
                         // per segment (by its first CTA) and per group of CTAs (by group slot),
                         // then ready flags per partial slot and per group slot
  DecSeg* segs;          // [B*Hkv]
  DecCta* ctas;          // [grid]
  int32_t* split_segs;   // [B*Hkv]
  float* part_lse;       // [max_slots][G], log2 domain
  float* part_o;         // [max_slots][G][d], normalised partial outputs
  float* grp_lse;        // [2 * grid][G]: merged groups of partials (single-launch path)
  float* grp_o;          // [2 * grid][G][d]
  int32_t max_slots;     // >= the slots any plan needs: max(B*Hkv + grid, 2 * grid)
  int32_t grid;
};

constexpr int kDecTileKeys = 128;
constexpr int kDecMaxSegs = 16384;   // B * Hkv of one decode call (the planner keeps 8 bytes per segment on chip)
constexpr int kDecFusedSegs = 512;   // up to this many segments every decode CTA plans for itself
constexpr int kDecMaxGrid = 1024;    // split counters kept at the start of the decode workspace
constexpr size_t kDecCounterBytes = 256 + sizeof(int32_t) * 7 * kDecMaxGrid;   // header + counters + flags

// Lower bound (first entry >= x) of an ascending logical-page list from its two ends: the
// answer when the ends decide it, else -1 and a guess g (1 <= g <= n-1) to verify with
// lb_verify after loading row[g-1] and row[g].  `hint` is where the answer lies if the
// list is contiguous near it.
__device__ __forceinline__ int lb_ends(const int32_t* row, int n, int first, int last, int x, int hint, int& g) {
  g = -1;
  if (!row) return min(max(x, 0), n);
  if (n <= 0 || x <= first) return 0;
  if (x > last) return n;
  if (last - first == n - 1) return x - first;
  g = min(max(hint, 1), n - 1);   // first < x <= last: the answer is in [1, n-1]
  return -1;
}

// below = row[g-1], at = row[g]
__device__ __forceinline__ int lb_verify(const int32_t* row, int n, int x, int g, int below, int at) {
  if (below < x && at >= x) return g;
  int lo = at < x ? g + 1 : 1, hi = at < x ? n : g - 1;   // row[0] < x; row[g-1] >= x in the second case
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(row + mid) < x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// Visible entry ranges of one decode segment (its query sits at position seq_len - 1),
// found in three rounds of loads -- the segment's scalars, the two ends of its logical-page
// list, one check of every bound the ends leave open -- so that a thread can interleave
// the rounds of several segments.  Result: e_sink, e_w, n_vis as in Unit.
struct DecRange {
  int b, L, n, cls, W, S, first, last;
  const int32_t* lrow;
  int x_hi, x_w, x_s, r_hi, r_w, r_s, g_hi, g_w, g_s;
  int a_hi, b_hi, a_w, b_w, a_s, b_s;
  int e_sink, e_w, n_vis;

  __device__ __forceinline__ void load1(const AttnParams& p, int seg) {
    b = seg / p.Hkv;
    L = __ldg(p.seq_len + b);
    n = __ldg(p.n_pages + seg);
    cls = __ldg(p.head_class + seg);
    const int Wr = __ldg(p.window + seg);
    const int Sr = p.sink ? __ldg(p.sink + seg) : 0;
    const bool local = cls == RK_CLASS_LOCAL;
    W = local ? Wr : 0;
    S = local ? Sr : 0;
    if (n < 0 || n > p.max_pages) { report(p.status, RK_ERR_DEVICE_BOUNDS); n = 0; }
    lrow = p.page_logical ? p.page_logical + int64_t(seg) * p.max_pages : nullptr;
  }
  __device__ __forceinline__ void load2() {
    first = last = 0;
    if (lrow && n > 0 && L > 0) {
      first = __ldg(lrow);
      last = __ldg(lrow + n - 1);
    }
  }
  __device__ __forceinline__ void load3(const AttnParams& p) {
    // n strictly ascending entries span at least n - 1 logical pages
    if (lrow && n > 1 && L > 0 && (long long)last - first < n - 1) report(p.status, RK_ERR_DEVICE_ORDER);
    g_hi = g_w = g_s = -1;
    r_hi = r_w = r_s = 0;
    if (L <= 0 || n <= 0) return;
    const bool local = cls == RK_CLASS_LOCAL;
    const int pos = L - 1;
    x_hi = pos / p.P + 1;                   // entries with logical page <= pos / P
    x_w = max(0, pos - W + 1) / p.P;        // first window page
    x_s = (S - 1) / p.P + 1;                // entries past the sink pages
    r_hi = lb_ends(lrow, n, first, last, x_hi, n - 1 - (last - x_hi), g_hi);
    if (local) r_w = lb_ends(lrow, n, first, last, x_w, n - 1 - (last - x_w), g_w);
    if (local && S > 0) r_s = lb_ends(lrow, n, first, last, x_s, x_s - first, g_s);
    if (g_hi >= 0) { a_hi = __ldg(lrow + g_hi - 1); b_hi = __ldg(lrow + g_hi); }
    if (g_w >= 0) { a_w = __ldg(lrow + g_w - 1); b_w = __ldg(lrow + g_w); }
    if (g_s >= 0) { a_s = __ldg(lrow + g_s - 1); b_s = __ldg(lrow + g_s); }
  }
  __device__ __forceinline__ void finish() {
    e_sink = e_w = n_vis = 0;
    if (L <= 0 || n <= 0) return;
    if (g_hi >= 0) r_hi = lb_verify(lrow, n, x_hi, g_hi, a_hi, b_hi);
    if (g_w >= 0) r_w = lb_verify(lrow, n, x_w, g_w, a_w, b_w);
    if (g_s >= 0) r_s = lb_verify(lrow, n, x_s, g_s, a_s, b_s);
    const int e_hi = r_hi;
    if (cls == RK_CLASS_LOCAL) {
      int ew = min(r_w, e_hi), es = S > 0 ? min(r_s, e_hi) : 0;
      if (es >= ew) { es = 0; ew = 0; }
      e_sink = es;
      e_w = ew;
      n_vis = es + (e_hi - ew);
    } else {
      n_vis = e_hi;
    }
  }
};

// Block-wide exclusive scan of one int per thread (blockDim.x a multiple of 32, at most
// 1024); returns the prefix, writes the total.  s_warp holds 32 ints.
__device__ __forceinline__ int block_exclusive_scan(int v, int* total, int* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < (blockDim.x >> 5) ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    s_warp[lane] = w;   // inclusive prefix of warp sums
  }
  __syncthreads();
  const int base = warp ? s_warp[warp - 1] : 0;
  *total = s_warp[(blockDim.x >> 5) - 1];
  __syncthreads();
  return base + x - v;
}

// The same for one 64-bit value per thread (several counts packed in bit fields, none of
// which may carry into the next); s_warp holds 32 values.
__device__ __forceinline__ unsigned long long block_exclusive_scan64(unsigned long long v, unsigned long long* total,
                                                                     unsigned long long* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    unsigned long long w = lane < (blockDim.x >> 5) ? s_warp[lane] : 0ull;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    s_warp[lane] = w;   // inclusive prefix of warp sums
  }
  __syncthreads();
  const unsigned long long base = warp ? s_warp[warp - 1] : 0ull;
  *total = s_warp[(blockDim.x >> 5) - 1];
  __syncthreads();
  return base + x - v;
}

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Launch configuration with programmatic dependent launch: the kernel may be scheduled
// before its predecessor in the stream has finished; it must execute
// griddepcontrol.wait before touching anything the predecessor writes.
inline cudaLaunchConfig_t pdl_config(dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                     cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// Launchers implemented in the .cu files.
cudaError_t launch_plan(const AttnParams& p, const AttnWorkspace& ws, int rows_per_unit,
                        int entries_per_tile, int target_items, int min_chunk_tiles, cudaStream_t stream);
cudaError_t launch_plan_decode(const AttnParams& p, const DecWorkspace& ws, cudaStream_t stream);
cudaError_t launch_decode_tc(const AttnParams& p, const DecWorkspace& ws, cudaStream_t stream);
// bf16 2-D / 3-D tensor map with 128-byte swizzle (rk_prefill_tc.cu)
bool encode_tmap_bf16(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                      const cuuint32_t* box);
cudaError_t launch_rope(const rk_rope_args& a, void* workspace, cudaStream_t stream);
cudaError_t launch_rope_coefficients(const int32_t* deltas, int n, int d, double theta, void* coef,
                                     cudaStream_t stream);
cudaError_t launch_append_kv(const rk_append_args& a, cudaStream_t stream);
size_t sparse_ffn_ws_bytes(int keep, int d_model, int d_ff);
cudaError_t launch_sparse_ffn(const rk_sparse_ffn_args& a, void* ws, cudaStream_t stream);
cudaError_t launch_ring_advance(const rk_ring_args& a, cudaStream_t stream);

int device_sm_count();

}  // namespace rk
