// Decode-time storage: writing a step's new K/V rows into their page slots, and the page
// ring of window-only local heads.
//
// "小红书 RedKnot", section 3, first and fourth components: a local head keeps only a
// window of KV, so the pages its window has left can hold new tokens -- this is where
// the gain in concurrent sessions comes from.  With window W and page size P, a local
// head needs at most ceil(W/P) + 1 window pages at any time (its window spans at most
// ceil(W/P) + 1 pages, and the page a new token opens is one of them), so a ring of that
// many pages serves the whole decode.
//
// Both kernels are memory-trivial (a few rows and table entries per head segment); they
// exist so that the whole decode step stays on the device (no host round trip, graph
// capturable).  One warp per head segment.
#include "rk_internal.cuh"
#include "rk_sm100.cuh"

namespace rk {

namespace {

constexpr int kWarps = 8;   // head segments per 256-thread block

// Entry of logical page lp in an ascending list of n entries, or -1.
__device__ __forceinline__ int find_entry(const int32_t* lrow, int n, int lp) {
  if (n <= 0) return -1;
  if (!lrow) return lp < n ? lp : -1;
  if (lrow[n - 1] == lp) return n - 1;   // the common case: the newest page
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (lrow[mid] < lp) lo = mid + 1; else hi = mid;
  }
  return lrow[lo] == lp ? lo : -1;
}

// k_pool[page][pos % P] = k_new[seg], v likewise: 16-byte lanes, K in the first half of the
// warp, V in the second.
template <int D>
__global__ __launch_bounds__(kWarps * 32) void append_kv_kernel(const rk_append_args a) {
  sm100::grid_dependency_wait();     // k_new / v_new / pos / the pools: earlier work is complete
  sm100::grid_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int seg = blockIdx.x * kWarps + warp;
  if (seg >= a.B * a.Hkv) return;
  const int b = seg / a.Hkv;
  const int pos = a.pos[b];
  int n = a.n_pages[seg];
  if (pos < 0 || n < 0 || n > a.max_pages) {
    if (lane == 0) report(a.status, RK_ERR_DEVICE_BOUNDS);
    return;
  }
  const int32_t* lrow = a.page_logical ? a.page_logical + int64_t(seg) * a.max_pages : nullptr;
  const int e = find_entry(lrow, n, pos / a.P);
  const int page = e >= 0 ? a.page_table[int64_t(seg) * a.max_pages + e] : -1;
  if (page < 0 || page >= a.n_pool_pages) {   // the slot's page is not listed, or outside the pool
    if (lane == 0) report(a.status, RK_ERR_DEVICE_BOUNDS);
    return;
  }
  constexpr int kLanes = D * 2 / 16;          // 16-byte pieces of one row
  const int half = lane / kLanes, piece = lane % kLanes;
  if (half < 2) {
    const int64_t row = int64_t(page) * a.P + pos % a.P;
    const uint4* src = reinterpret_cast<const uint4*>(half ? a.v_new : a.k_new) + int64_t(seg) * kLanes + piece;
    uint4* dst = reinterpret_cast<uint4*>(half ? a.v_pool : a.k_pool) + row * kLanes + piece;
    *dst = *src;
  }
}

// Ring advance of the window-only local heads (ring[s] = R > 0): when the new position
// opens a logical page the list does not hold, the oldest window entry (the first entry
// after the sink pages) gives its physical page to it -- the window entries move down by
// one and the new logical page takes the last entry.
__global__ __launch_bounds__(kWarps * 32) void ring_advance_kernel(const rk_ring_args a) {
  // In place, decode calls after this one may read the tables before their predecessor
  // completes (RK_ATTN_METADATA_STABLE), so nothing after it starts before these writes are
  // done.  Out of place, the destination is read only by later steps: the next kernels may
  // start at once.  Either way the earlier readers and writers of the tables are complete
  // before anything is written.
  const bool copy = a.src_page_table != nullptr;
  if (copy) sm100::grid_launch_dependents();
  sm100::grid_dependency_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int seg = blockIdx.x * kWarps + warp;
  if (seg >= a.B * a.Hkv) return;
  const int R = a.ring[seg];
  if (R <= 0) return;
  const int b = seg / a.Hkv;
  const int pos = a.pos[b];
  const int n = a.n_pages[seg];
  if (pos < 0 || n < 1 || n > a.max_pages) {
    if (lane == 0) report(a.status, RK_ERR_DEVICE_BOUNDS);
    return;
  }
  const int64_t off = int64_t(seg) * a.max_pages;
  int32_t* trow = a.page_table + off;
  int32_t* lrow = a.page_logical + off;
  const int32_t* st = copy ? a.src_page_table + off : trow;
  const int32_t* sl = copy ? a.src_page_logical + off : lrow;
  const int lp = pos / a.P;
  bool advance = sl[n - 1] < lp;              // else the page is listed already
  const int S = a.sink ? a.sink[seg] : 0;
  const int sink_pages = S > 0 ? (S - 1) / a.P + 1 : 0;
  int e_sink = 0;                             // leading entries that are sink pages
  while (e_sink < n && sl[e_sink] < sink_pages) ++e_sink;
  if (advance) {
    const int W = a.window[seg];
    // the ring is full and its oldest page lies wholly before the new token's window
    const bool ok = n - e_sink == R && (int64_t(sl[e_sink]) + 1) * a.P - 1 <= int64_t(pos) - W;
    if (!ok) {
      if (lane == 0) report(a.status, RK_ERR_DEVICE_BOUNDS);
      advance = false;                        // the list stays as it was
    }
  }
  if (!copy && !advance) return;
  const int phys = advance ? st[e_sink] : 0;
  // entry e of the new list: the window entries move down by one and the freed page takes
  // the new logical page (out of place, every entry is written); 32 entries at a time, all
  // reads of a round before its writes
  for (int base = copy ? 0 : e_sink; base < n; base += 32) {
    const int e = base + lane;
    int t = 0, l = 0;
    if (e < n) {
      if (!advance || e < e_sink) {
        t = st[e];
        l = sl[e];
      } else if (e < n - 1) {
        t = st[e + 1];
        l = sl[e + 1];
      } else {
        t = phys;
        l = lp;
      }
    }
    __syncwarp();
    if (e < n) {
      trow[e] = t;
      lrow[e] = l;
    }
    __syncwarp();
  }
}

}  // namespace

cudaError_t launch_append_kv(const rk_append_args& a, cudaStream_t stream) {
  const int nseg = a.B * a.Hkv;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3((nseg + kWarps - 1) / kWarps), dim3(kWarps * 32), 0, stream, attr);
  return a.d == 128 ? cudaLaunchKernelEx(&cfg, append_kv_kernel<128>, a)
                    : cudaLaunchKernelEx(&cfg, append_kv_kernel<64>, a);
}

cudaError_t launch_ring_advance(const rk_ring_args& a, cudaStream_t stream) {
  const int nseg = a.B * a.Hkv;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3((nseg + kWarps - 1) / kWarps), dim3(kWarps * 32), 0, stream, attr);
  return cudaLaunchKernelEx(&cfg, ring_advance_kernel, a);
}

}  // namespace rk
