// Work planning for SegPagedAttention.
//
// The visible key set of a query tile against one KV head is read straight off that
// head's page list ("RedKnot" article, SegPagedAttention paragraph: the table records
// which pages the head reads).  The planner turns every (query tile, KV head) unit into
// at most two ranges of list entries -- sink pages and the causal / window pages -- by
// binary search on the ascending logical page numbers, then cuts the units into items
// of about equal size so that a persistent grid stays busy whatever the mix of head
// classes.  The attention kernel merges the items of a unit with the usual log-sum-exp rule.
#include "rk_internal.cuh"
#include "rk_sm100.cuh"

#include <algorithm>

namespace rk {

namespace {

constexpr int kPlanThreads = 1024;

// first entry e in [0, n) with logical(e) >= x
__device__ int lower_bound_lp(const int32_t* row, int n, int x) {
  if (!row) return min(max(x, 0), n);
  if (n <= 0) return 0;
  const int first = __ldg(row), last = __ldg(row + n - 1);
  if (x <= first) return 0;
  if (x > last) return n;
  if (last - first == n - 1) return x - first;    // contiguous run of logical pages
  // the list may end in a contiguous run (a window after sink pages): guess, then verify
  const int guess = n - 1 - (last - x);
  if (guess > 0 && guess < n) {
    const int at = __ldg(row + guess);
    if (at == x) return guess;
    if (at < x && __ldg(row + guess + 1) > x) return guess + 1;
  }
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(row + mid) < x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// first entry e in [0, n) with logical(e) > x
__device__ __forceinline__ int upper_bound_lp(const int32_t* row, int n, int x) {
  return lower_bound_lp(row, n, x + 1);
}

__global__ __launch_bounds__(kPlanThreads) void plan_kernel(AttnParams p, AttnWorkspace ws, int tok_per_unit,
                                                            int entries_per_tile, int target_items,
                                                            int min_chunk_tiles, int32_t* tile_prefix) {
  __shared__ int s_warp[32];
  __shared__ unsigned long long s_total_entries;
  __shared__ int s_chunk;
  sm100::grid_dependency_wait();      // inputs written by earlier kernels in the stream
  sm100::grid_launch_dependents();    // the attention kernel may start its prologue
  const int tid = threadIdx.x;
  if (tid == 0) s_total_entries = 0ull;

  // 1. query tiles per sequence and their prefix (units are enumerated as (tile, KV head))
  int carry = 0;
  for (int base = 0; base < p.B; base += kPlanThreads) {
    const int b = base + tid;
    int tiles = 0;
    if (b < p.B) {
      const int nq = __ldg(p.cu_seqlens_q + b + 1) - __ldg(p.cu_seqlens_q + b);
      tiles = nq > 0 ? (nq + tok_per_unit - 1) / tok_per_unit : 0;
    }
    int total;
    const int pre = block_exclusive_scan(tiles, &total, s_warp);
    if (b < p.B) tile_prefix[b] = carry + pre;
    carry += total;
  }
  if (tid == 0) tile_prefix[p.B] = carry;
  __syncthreads();
  const int n_tiles = carry;
  int n_units = n_tiles * p.Hkv;
  if (n_units > ws.max_units) {  // cannot happen with the sizes the host validated
    if (tid == 0) report(p.status, RK_ERR_DEVICE_BOUNDS);
    n_units = ws.max_units;
  }

  // 2. visible entry ranges of every unit
  unsigned long long my_entries = 0;
  for (int u = tid; u < n_units; u += kPlanThreads) {
    const int tile_g = u / p.Hkv, h = u - (u / p.Hkv) * p.Hkv;
    int lo = 0, hi = p.B;   // last b with tile_prefix[b] <= tile_g
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (tile_prefix[mid] <= tile_g) lo = mid; else hi = mid;
    }
    const int b = lo;
    const int tile = tile_g - tile_prefix[b];
    const int seg = b * p.Hkv + h;
    const int q0 = __ldg(p.cu_seqlens_q + b);
    const int nq = __ldg(p.cu_seqlens_q + b + 1) - q0;
    const int L = __ldg(p.seq_len + b);
    Unit un;
    un.seg = seg;
    un.b = b;
    un.tok0 = q0 + tile * tok_per_unit;
    un.ntok = min(tok_per_unit, nq - tile * tok_per_unit);
    un.pos0 = L - nq + tile * tok_per_unit;
    un.e_sink = 0;
    un.e_w = 0;
    un.n_vis = 0;
    int n = __ldg(p.n_pages + seg);
    if (n < 0 || n > p.max_pages) { report(p.status, RK_ERR_DEVICE_BOUNDS); n = 0; }
    if (q0 < 0 || nq < 0 || int64_t(q0) + nq > p.total_q) {   // queries outside q / out
      report(p.status, RK_ERR_DEVICE_BOUNDS);
      un.ntok = 0;
      n = 0;
    }
    const int p_first = un.pos0, p_last = un.pos0 + un.ntok - 1;
    if (L > 0 && p_last >= 0 && n > 0) {
      const int32_t* lrow = p.page_logical ? p.page_logical + int64_t(seg) * p.max_pages : nullptr;
      // n strictly ascending entries span at least n - 1 logical pages
      if (lrow && n > 1 && (long long)__ldg(lrow + n - 1) - __ldg(lrow) < n - 1) report(p.status, RK_ERR_DEVICE_ORDER);
      const int cap = min(p_last, L - 1);
      const int e_hi = upper_bound_lp(lrow, n, cap / p.P);
      const int cls = __ldg(p.head_class + seg);
      if (cls == RK_CLASS_LOCAL) {
        const int W = __ldg(p.window + seg);
        const int S = p.sink ? __ldg(p.sink + seg) : 0;
        const int start = max(0, p_first - W + 1);
        int e_w = min(lower_bound_lp(lrow, n, start / p.P), e_hi);
        int e_s = S > 0 ? min(upper_bound_lp(lrow, n, (S - 1) / p.P), e_hi) : 0;
        if (e_s >= e_w) { e_s = 0; e_w = 0; }
        un.e_sink = e_s;
        un.e_w = e_w;
        un.n_vis = e_s + (e_hi - e_w);
      } else {
        un.n_vis = e_hi;
      }
    }
    ws.units[u] = un;
    my_entries += (unsigned long long)un.n_vis;
  }
  atomicAdd(&s_total_entries, my_entries);
  __syncthreads();

  // 3. chunk size: about target_items items overall, whole key tiles, at least min_chunk_tiles
  if (tid == 0) {
    const unsigned long long total = s_total_entries;
    long long c = (long long)((total + target_items - 1) / (unsigned long long)max(target_items, 1));
    c = max(c, (long long)min_chunk_tiles * entries_per_tile);
    c = ((c + entries_per_tile - 1) / entries_per_tile) * entries_per_tile;
    s_chunk = (int)min(c, (long long)(1 << 30));
  }
  __syncthreads();
  const int chunk = s_chunk;

  // 4. items: a unit's entries are cut into full-size chunks, a remainder of more than half
  //    a chunk becoming an item of its own and a smaller one joining the last chunk.  The
  //    items of a unit are consecutive, and the units come in three classes: single items
  //    of at least a chunk (the longest, first), then the units cut into several items in
  //    unit order -- so that they complete one after another and the attention kernel can
  //    merge each while later ones run -- then the single items shorter than a chunk.  The
  //    split units are listed for that merge; their completion counters start at zero.
  int cls_items[3] = {0, 0, 0}, carry_split = 0;
  for (int base = 0; base < n_units; base += kPlanThreads) {
    const int u = base + tid;
    int ns = 0, cls = 0;
    if (u < n_units) {
      const int nv = ws.units[u].n_vis;
      const int r = nv % chunk, nf = nv / chunk;
      const int rm = (nv == 0 || (r != 0 && (nf == 0 || 2 * r > chunk))) ? 1 : 0;
      ns = nf + rm;
      cls = ns > 1 ? 1 : nf >= 1 ? 0 : 2;
      ws.units[u].n_full = nf;
      ws.units[u].n_splits = ns;
      ws.unit_done[u] = 0;
    }
    int tot[3], pre[3];
#pragma unroll
    for (int c = 0; c < 3; ++c) pre[c] = block_exclusive_scan(cls == c ? ns : 0, &tot[c], s_warp);
    int tot_s;
    const int pre_s = block_exclusive_scan(cls == 1 ? 1 : 0, &tot_s, s_warp);
    if (u < n_units) {
      const int base_c = cls == 0 ? cls_items[0] + pre[0] : cls == 1 ? cls_items[1] + pre[1] : cls_items[2] + pre[2];
      ws.units[u].first_item = base_c;   // within its class, made absolute below
      ws.units[u].rem_item = cls;
      if (cls == 1) ws.split_list[carry_split + pre_s] = u;
    }
#pragma unroll
    for (int c = 0; c < 3; ++c) cls_items[c] += tot[c];
    carry_split += tot_s;
  }
  __syncthreads();
  const int n_items_all = cls_items[0] + cls_items[1] + cls_items[2];
  for (int u = tid; u < n_units; u += kPlanThreads) {
    Unit& un = ws.units[u];
    const int cls = un.rem_item;
    un.first_item += cls == 0 ? 0 : cls == 1 ? cls_items[0] : cls_items[0] + cls_items[1];
    un.rem_item = -1;
    const int nv = un.n_vis;
    for (int s = 0; s < un.n_splits; ++s) {
      const int it = unit_item(un, s);
      if (it >= ws.max_items) { report(p.status, RK_ERR_DEVICE_BOUNDS); break; }
      Item item;
      item.unit = u;
      item.v_begin = s * chunk;
      item.v_end = s == un.n_splits - 1 ? nv : (s + 1) * chunk;
      item.split = s;
      ws.items[it] = item;
    }
  }
  if (tid == 0) {
    ws.header->n_units = n_units;
    ws.header->n_items = min(n_items_all, ws.max_items);
    ws.header->chunk = chunk;
    ws.header->counter = 0;
    ws.header->n_split = carry_split;
    ws.header->merge_counter = 0;
  }
}

// Decode plan: one query per sequence at position seq_len - 1.
//  1. each head segment's visible entry ranges (as plan_kernel), in three rounds of loads:
//     the segment's scalars, the two ends of its logical-page list, then one check of every
//     bound the ends do not settle; its key tiles; and, for a segment with nothing visible,
//     its output (zeros, lse = -inf), which no CTA writes;
//  2. the tile prefix over segments: T tiles in all; with gs = min(grid, T), CTA c < gs of
//     the decode grid takes tiles [c*T/gs, (c+1)*T/gs), so tile t belongs to CTA
//     ((t+1)*gs + T - 1) / T - 1 (the others get no tiles);
//  3. per segment the CTAs its tiles fall to; segments with more than one get consecutive
//     partial slots and are listed for combine_decode_tc_kernel;
//  4. per CTA the segment holding its first tile.
// Per-segment tile counts and prefixes stay in shared memory (8 bytes per segment).
__global__ __launch_bounds__(kPlanThreads) void plan_decode_kernel(AttnParams p, DecWorkspace ws) {
  // the decode kernel may start its prologue now; it reads this plan after griddepcontrol.wait
  sm100::grid_launch_dependents();
  extern __shared__ int s_seg[];            // [nseg] tiles, then [nseg] first tile
  __shared__ int s_warp[32];
  const int tid = threadIdx.x;
  const int nseg = p.B * p.Hkv;
  const int ept = kDecTileKeys / p.P;
  const int grid = ws.grid;
  int* s_nt = s_seg;
  int* s_t0 = s_seg + nseg;

  // 1. visible ranges
  for (int seg = tid; seg < nseg; seg += kPlanThreads) {
    DecRange r;
    r.load1(p, seg);
    r.load2();
    r.load3(p);
    r.finish();
    const int b = r.b, L = r.L, cls = r.cls, W = r.W, S = r.S, pos = L - 1;
    const int e_sink = r.e_sink, e_w = r.e_w, n_vis = r.n_vis;
    DecSeg& ds = ws.segs[seg];
    ds.e_sink = e_sink;
    ds.e_w = e_w;
    ds.n_vis = n_vis;
    const int nt = (n_vis + ept - 1) / ept;
    ds.n_tiles = nt;
    ds.b = b;
    ds.tok = b;
    ds.pos = pos;
    ds.cls = cls;
    ds.W = W;
    ds.S = S;
    ds.L = L;
    s_nt[seg] = nt;
    if (nt == 0) {   // nothing visible: out = 0, lse = -inf
      const int h = seg - b * p.Hkv;
      uint4* o = reinterpret_cast<uint4*>(p.out + (int64_t(b) * p.Hq + h * p.G) * p.d);
      for (int i = 0; i < p.G * p.d / 8; ++i) o[i] = make_uint4(0, 0, 0, 0);
      if (p.lse)
        for (int g = 0; g < p.G; ++g) p.lse[int64_t(b) * p.Hq + h * p.G + g] = -INFINITY;
    }
  }
  __syncthreads();

  // 2. tile prefix
  int carry = 0;
  for (int base = 0; base < nseg; base += kPlanThreads) {
    const int seg = base + tid;
    const int nt = seg < nseg ? s_nt[seg] : 0;
    int tot;
    const int pre = block_exclusive_scan(nt, &tot, s_warp);
    if (seg < nseg) s_t0[seg] = carry + pre;
    carry += tot;
  }
  const long long T = carry;
  // shares are cut over at most T CTAs, so that every share holds at least one tile and
  // the CTAs a segment's tiles fall to are exactly the ones that write its partials
  const int gs = (int)min((long long)grid, T);
  for (int c = tid; c < grid; c += kPlanThreads) {
    DecCta dc;
    dc.seg0 = nseg;
    dc.tile_begin = c < gs ? (int)((long long)c * T / gs) : (int)T;
    dc.tile_end = c < gs ? (int)((long long)(c + 1) * T / gs) : (int)T;
    dc.pad = 0;
    ws.ctas[c] = dc;
  }
  __syncthreads();

  // 3. owners, splits and slots;  4. first segment of each CTA's share
  auto owner = [&](long long t) { return (int)(((t + 1) * gs + T - 1) / T - 1); };
  int carry_slot = 0, carry_split = 0;
  for (int base = 0; base < nseg; base += kPlanThreads) {
    const int seg = base + tid;
    int ns = 0, t0 = 0, nt = 0, c0 = 0, c1 = -1;
    if (seg < nseg) {
      t0 = s_t0[seg];
      nt = s_nt[seg];
      if (nt > 0) {
        c0 = owner(t0);
        c1 = owner((long long)t0 + nt - 1);
        ns = c1 - c0 + 1;
      }
    }
    const int split = ns > 1 ? 1 : 0;
    int tot_slot, tot_split;
    const int pre_slot = block_exclusive_scan(split ? ns : 0, &tot_slot, s_warp);
    const int pre_split = block_exclusive_scan(split, &tot_split, s_warp);
    if (seg < nseg) {
      DecSeg& ds = ws.segs[seg];
      ds.tile0 = t0;
      ds.cta0 = c0;
      ds.n_splits = nt > 0 ? ns : 1;
      ds.slot0 = split ? carry_slot + pre_slot : -1;
      if (split) ws.split_segs[carry_split + pre_split] = seg;
      if (nt > 0) {
        // CTAs whose share starts inside this segment: all of c0..c1 except c0 when its share
        // began in an earlier segment
        const int cs = ((long long)c0 * T / gs < t0) ? c0 + 1 : c0;
        for (int c = cs; c <= c1; ++c) ws.ctas[c].seg0 = seg;
      }
    }
    carry_slot += tot_slot;
    carry_split += tot_split;
  }
  if (carry_slot > ws.max_slots) {   // cannot happen (slots <= segments + grid); nothing is scheduled
    if (tid == 0) report(p.status, RK_ERR_DEVICE_BOUNDS);
    for (int c = tid; c < grid; c += kPlanThreads) ws.ctas[c].tile_end = ws.ctas[c].tile_begin;
    carry_split = 0;
  }
  if (tid == 0) {
    ws.header->total_tiles = (int)T;
    ws.header->n_split = carry_split;
    ws.header->grid = grid;
  }
}

}  // namespace

cudaError_t launch_plan_decode(const AttnParams& p, const DecWorkspace& ws, cudaStream_t stream) {
  const size_t smem = size_t(8) * p.B * p.Hkv;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(plan_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         8 * kDecMaxSegs);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  plan_decode_kernel<<<1, kPlanThreads, smem, stream>>>(p, ws);
  return cudaGetLastError();
}

cudaError_t launch_plan(const AttnParams& p, const AttnWorkspace& ws, int tok_per_unit,
                        int entries_per_tile, int target_items, int min_chunk_tiles, cudaStream_t stream) {
  // the tile prefix lives right after the partial outputs (sized by the host)
  int32_t* tile_prefix = reinterpret_cast<int32_t*>(ws.part_o + int64_t(ws.max_items) * ws.rows * p.d);
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(1), dim3(kPlanThreads), 0, stream, attr);
  return cudaLaunchKernelEx(&cfg, plan_kernel, p, ws, tok_per_unit, entries_per_tile, target_items,
                            min_chunk_tiles, tile_prefix);
}


}  // namespace rk
