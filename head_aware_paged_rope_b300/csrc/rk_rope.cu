// RoPE repositioning of cached K pages ("RedKnot" article, is96.com: the inverse
// rotation at the offline position followed by the forward rotation at the online
// position; "小红书 RedKnot", section 3, second component).
//
// Both positions of a run advance together, so R(pos_on) R(pos_off)^-1 is one turn by
// delta = pos_on0 - pos_off0 per channel pair.  Kernel 1 takes cos/sin of delta * w_i
// in double precision once per (run, pair) and splits each into a 16-significant-bit
// head plus an fp32 tail; kernel 2 streams the K rows: with bf16 inputs (8 significant
// bits) the head products are exact in fp32, so the rotated value carries only the
// final fp32 rounding even when the two products cancel, and the bf16 result stays
// within one ulp of the exact rotation.  Kernel 2 is HBM-bound: each token row is read
// once and written once with 16-byte vector accesses.
#include "rk_internal.cuh"
#include "rk_sm100.cuh"

#include <algorithm>

namespace rk {

namespace {

using namespace sm100;

// cos / sin of delta * theta^(-2i/d) in double precision, each split into a head with 16
// significant bits (so that head * bf16 is exact in fp32) and an fp32 tail.
__device__ __forceinline__ float4 rope_coeff(double delta, int i, int d, double theta) {
  const double w = pow(theta, -2.0 * double(i) / double(d));
  double s, c;
  sincos(delta * w, &s, &c);
  const float c_hi = __uint_as_float(__float_as_uint(__double2float_rn(c)) & 0xFFFFFF00u);
  const float s_hi = __uint_as_float(__float_as_uint(__double2float_rn(s)) & 0xFFFFFF00u);
  const float c_lo = __double2float_rn(c - double(c_hi));
  const float s_lo = __double2float_rn(s - double(s_hi));
  return make_float4(c_hi, c_lo, s_hi, s_lo);
}

__global__ void rope_coeff_kernel(const rk_rope_run* __restrict__ runs, int n_runs, int d,
                                  double theta, float4* __restrict__ coef) {
  const int run = blockIdx.x;
  const int i = threadIdx.x;
  if (run >= n_runs || i >= d / 2) return;
  const rk_rope_run r = runs[run];
  coef[size_t(run) * (d / 2) + i] = rope_coeff(double((long long)r.pos_on0 - (long long)r.pos_off0), i, d, theta);
}

__global__ void rope_coeff_delta_kernel(const int32_t* __restrict__ deltas, int n, int d, double theta,
                                        float4* __restrict__ coef) {
  const int r = blockIdx.x;
  const int i = threadIdx.x;
  if (r >= n || i >= d / 2) return;
  coef[size_t(r) * (d / 2) + i] = rope_coeff(double(deltas[r]), i, d, theta);
}

__device__ __forceinline__ void st_stream(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w) : "memory");
}

__device__ __forceinline__ float u32_elem(const uint4& v, int k) {
  const uint32_t w = (k >> 1) == 0 ? v.x : (k >> 1) == 1 ? v.y : (k >> 1) == 2 ? v.z : v.w;
  return (k & 1) ? bf16hi(w) : bf16lo(w);
}

// Kernel 2 is persistent (two CTAs per SM).  The runs' tokens are cut into blocks of kRows
// rows (32 KB of K); CTA c takes a contiguous range of blocks.  Its producer warp fetches
// the page ids of a group of blocks at once (one table entry per lane), then copies each
// block's source rows, one bulk copy per source page (one lane each), into a ring of
// kStages shared-memory stages.  Eight consumer warps rotate the rows (thread = row x 16
// channels, kRowsPerThread rows each) and store them to their destination pages with
// 16-byte streaming stores.  Every wait is bounded.
constexpr int kRopeConsumers = 256;
constexpr int kRopeThreads = kRopeConsumers + 32;
constexpr int kRopeStages = 3;
constexpr int kRowsPerThread = 4;
constexpr uint64_t kRopeWaitNs = 1000000000ull;

template <int D>
struct RopeCfg {
  static constexpr int kLanes = D / 16;                 // lanes per row (8 channel pairs each)
  static constexpr int kRowsPerPass = kRopeConsumers / kLanes;
  static constexpr int kRows = kRowsPerPass * kRowsPerThread;   // rows per block: 128 (d 128), 256 (d 64)
  static constexpr int kRowBytes = D * 2;
  static constexpr int kStageBytes = kRows * kRowBytes; // 32 KB
  static constexpr int kMaxPages = kRows / 16 + 1;      // pages one block touches (P >= 16): 9 or 17
  static constexpr int kSmem = kRopeStages * kStageBytes + 128;
};

struct RopeMeta {
  int32_t run, t0, n;           // n < 0: no more blocks
  int32_t pos_off0, pos_on0;
  int32_t src_p0, dst_p0;       // first table entry (logical page) the block touches
  uint32_t src_ok;              // bit i: the rows of source page src_p0 + i were copied
  int32_t dst_id[17];           // physical page of destination entry dst_p0 + i, -1 if invalid
  int32_t pad[7];
};

struct RopeShared {
  uint64_t full[kRopeStages], empty[kRopeStages];
  RopeMeta meta[kRopeStages];
  int abort;
};

__device__ __forceinline__ bool rope_wait(RopeShared& sh, uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*reinterpret_cast<volatile int*>(&sh.abort)) return false;
    if (globaltimer() - t0 > kRopeWaitNs) return false;
  }
}

template <int D, int STYLE>
__global__ __launch_bounds__(kRopeThreads) void rope_apply_kernel(
    const __nv_bfloat16* __restrict__ k_src, __nv_bfloat16* __restrict__ k_dst, int64_t n_src_pages,
    int64_t n_dst_pages, const int32_t* __restrict__ src_tables, int64_t n_src_entries,
    const int32_t* __restrict__ dst_tables, int64_t n_dst_entries, const rk_rope_run* __restrict__ runs,
    int n_runs, int P, int max_tok, const float4* __restrict__ coef, int32_t* status) {
  using C = RopeCfg<D>;
  constexpr int NS = kRopeStages;
  extern __shared__ __align__(128) uint8_t rope_smem[];
  __shared__ RopeShared sh;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sbase = smem_addr(rope_smem);
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_addr(&sh.full[s]), 1);
      mbar_init(smem_addr(&sh.empty[s]), kRopeConsumers / 32);
    }
    sh.abort = 0;
    mbar_fence_init();
  }
  __syncthreads();
  grid_dependency_wait();      // K pools and tables: everything before this call has completed
  grid_launch_dependents();

  const int tiles = (max_tok + C::kRows - 1) / C::kRows;
  const long long n_blocks = (long long)n_runs * tiles;
  const long long b_begin = (long long)blockIdx.x * n_blocks / gridDim.x;
  const long long b_end = (long long)(blockIdx.x + 1) * n_blocks / gridDim.x;

  if (warp == kRopeConsumers / 32) {
    // ---------------------------------------------------------------- producer warp
    const int kGroup = max(1, 31 * P / C::kRows);   // blocks whose pages fit in 32 table entries
    int cur_run = -1, n_tok = 0;
    bool run_ok = false;
    rk_rope_run rr{};
    int g_run = -1, g_idx = -1, g_src0 = 0, g_dst0 = 0, g_src_id = -1, g_dst_id = -1;
    uint32_t k = 0;
    bool ok = true;
    for (long long b = b_begin; b < b_end && ok; ++b) {
      const int run = int(b / tiles), tile = int(b - (long long)run * tiles);
      if (run != cur_run) {
        rr = runs[run];
        cur_run = run;
        run_ok = rr.n_tok >= 0 && rr.n_tok <= max_tok && rr.pos_off0 >= 0 && rr.pos_on0 >= 0 &&
                 rr.src_tab_off >= 0 && rr.dst_tab_off >= 0;
        if (!run_ok && lane == 0 && tile == 0) report(status, RK_ERR_DEVICE_BOUNDS);
        n_tok = min(rr.n_tok, max_tok);
      }
      const int t0 = tile * C::kRows;
      const int n = min(C::kRows, n_tok - t0);
      if (!run_ok || n <= 0) continue;
      // page ids of this block's group: lane j holds entry g_src0 + j (g_dst0 + j)
      const int grp = tile / kGroup;
      if (run != g_run || grp != g_idx) {
        const int tg0 = grp * kGroup * C::kRows;
        const int tg1 = min(n_tok, tg0 + kGroup * C::kRows) - 1;
        g_src0 = (rr.pos_off0 + tg0) / P;
        g_dst0 = (rr.pos_on0 + tg0) / P;
        const int se = g_src0 + lane, de = g_dst0 + lane;
        g_src_id = g_dst_id = -1;
        if (se <= (rr.pos_off0 + tg1) / P) {
          if (se < rr.src_tab_len && int64_t(rr.src_tab_off) + se < n_src_entries) {
            const int id = __ldg(src_tables + rr.src_tab_off + se);
            if (id >= 0 && id < n_src_pages) g_src_id = id; else report(status, RK_ERR_DEVICE_BOUNDS);
          } else {
            report(status, RK_ERR_DEVICE_BOUNDS);
          }
        }
        if (de <= (rr.pos_on0 + tg1) / P) {
          if (de < rr.dst_tab_len && int64_t(rr.dst_tab_off) + de < n_dst_entries) {
            const int id = __ldg(dst_tables + rr.dst_tab_off + de);
            if (id >= 0 && id < n_dst_pages) g_dst_id = id; else report(status, RK_ERR_DEVICE_BOUNDS);
          } else {
            report(status, RK_ERR_DEVICE_BOUNDS);
          }
        }
        g_run = run;
        g_idx = grp;
      }
      const int st = k % NS;
      bool got = true;
      if (lane == 0 && k >= NS) got = rope_wait(sh, smem_addr(&sh.empty[st]), ((k / NS) - 1) & 1);
      if (!__shfl_sync(0xffffffffu, got, 0)) { ok = false; break; }
      // source segments: lane i copies the block's rows on source entry sp0 + i
      const int sp0 = (rr.pos_off0 + t0) / P, sp1 = (rr.pos_off0 + t0 + n - 1) / P;
      const int dp0 = (rr.pos_on0 + t0) / P;
      const int src_id = __shfl_sync(0xffffffffu, g_src_id, min(31, sp0 - g_src0 + lane));
      int tok_lo = 0, rows = 0;
      bool seg = lane <= sp1 - sp0;
      if (seg) {
        tok_lo = max(t0, (sp0 + lane) * P - rr.pos_off0);
        const int tok_hi = min(t0 + n, (sp0 + lane + 1) * P - rr.pos_off0);
        rows = tok_hi - tok_lo;
        seg = rows > 0 && src_id >= 0;
      }
      const uint32_t okmask = __ballot_sync(0xffffffffu, seg);
      int bytes = seg ? rows * C::kRowBytes : 0;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) bytes += __shfl_xor_sync(0xffffffffu, bytes, o);
      int dids[C::kMaxPages];
#pragma unroll
      for (int i = 0; i < C::kMaxPages; ++i) dids[i] = __shfl_sync(0xffffffffu, g_dst_id, min(31, dp0 - g_dst0 + i));
      if (lane == 0) {
        RopeMeta& m = sh.meta[st];
        m.run = run;
        m.t0 = t0;
        m.n = n;
        m.pos_off0 = rr.pos_off0;
        m.pos_on0 = rr.pos_on0;
        m.src_p0 = sp0;
        m.dst_p0 = dp0;
        m.src_ok = okmask;
#pragma unroll
        for (int i = 0; i < C::kMaxPages; ++i) m.dst_id[i] = dids[i];
        mbar_arrive_expect_tx(smem_addr(&sh.full[st]), uint32_t(bytes));
      }
      __syncwarp();
      if (seg) {
        const int slot = rr.pos_off0 + tok_lo - (sp0 + lane) * P;
        bulk_copy_g2s(sbase + st * C::kStageBytes + (tok_lo - t0) * C::kRowBytes,
                      k_src + (int64_t(src_id) * P + slot) * D, uint32_t(rows * C::kRowBytes),
                      smem_addr(&sh.full[st]));
      }
      ++k;
    }
    if (ok) {   // end marker
      const int st = k % NS;
      bool got = true;
      if (lane == 0 && k >= NS) got = rope_wait(sh, smem_addr(&sh.empty[st]), ((k / NS) - 1) & 1);
      if (lane == 0 && got) {
        sh.meta[st].n = -1;
        mbar_arrive(smem_addr(&sh.full[st]));
      }
      ok = __shfl_sync(0xffffffffu, got, 0);
    }
    if (!ok && lane == 0) {
      report(status, RK_ERR_TIMEOUT);
      *reinterpret_cast<volatile int*>(&sh.abort) = 1;
      // copies still in flight land before the CTA exits (bounded)
      for (uint32_t j = k > NS ? k - NS : 0; j < k; ++j)
        mbar_wait(smem_addr(&sh.full[j % NS]), (j / NS) & 1);
    }
  } else {
    // ---------------------------------------------------------------- consumers
    const int ln = tid % C::kLanes;    // pairs 8*ln .. 8*ln+7
    const int row0 = tid / C::kLanes;
    const int ca = STYLE == RK_ROPE_HALF_SPLIT ? 8 * ln : 16 * ln;
    const int cb = STYLE == RK_ROPE_HALF_SPLIT ? D / 2 + 8 * ln : 16 * ln + 8;
    int cur_run = -1;
    float4 cf[8];
    for (uint32_t k = 0;; ++k) {
      const int st = k % NS;
      if (!rope_wait(sh, smem_addr(&sh.full[st]), (k / NS) & 1)) {
        report(status, RK_ERR_TIMEOUT);
        *reinterpret_cast<volatile int*>(&sh.abort) = 1;
        break;
      }
      const RopeMeta& m = sh.meta[st];
      const int n = m.n;
      if (n < 0) break;
      if (m.run != cur_run) {
        cur_run = m.run;
        const float4* cr = coef + size_t(cur_run) * (D / 2) + 8 * ln;
#pragma unroll
        for (int i = 0; i < 8; ++i) cf[i] = __ldg(cr + i);
      }
#pragma unroll
      for (int rr = 0; rr < kRowsPerThread; ++rr) {
        const int row = rr * C::kRowsPerPass + row0;
        if (row >= n) continue;
        const int t = m.t0 + row;
        const int spos = m.pos_off0 + t, opos = m.pos_on0 + t;
        const bool src_ok = (m.src_ok >> (spos / P - m.src_p0)) & 1u;
        const int did = m.dst_id[opos / P - m.dst_p0];
        if (src_ok && did >= 0) {
          const uint32_t rb = sbase + st * C::kStageBytes + row * C::kRowBytes;
          uint4 xa, xb;
          asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(xa.x), "=r"(xa.y), "=r"(xa.z), "=r"(xa.w)
                       : "r"(rb + ca * 2));
          asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(xb.x), "=r"(xb.y), "=r"(xb.z), "=r"(xb.w)
                       : "r"(rb + cb * 2));
          float ya[8], yb[8];
          uint4 oa, ob;
          if (STYLE == RK_ROPE_HALF_SPLIT) {
#pragma unroll
            for (int i = 0; i < 8; ++i) rotate_pair(u32_elem(xa, i), u32_elem(xb, i), cf[i], ya[i], yb[i]);
            oa.x = pack_bf16(ya[0], ya[1]); oa.y = pack_bf16(ya[2], ya[3]);
            oa.z = pack_bf16(ya[4], ya[5]); oa.w = pack_bf16(ya[6], ya[7]);
            ob.x = pack_bf16(yb[0], yb[1]); ob.y = pack_bf16(yb[2], yb[3]);
            ob.z = pack_bf16(yb[4], yb[5]); ob.w = pack_bf16(yb[6], yb[7]);
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              rotate_pair(u32_elem(xa, 2 * i), u32_elem(xa, 2 * i + 1), cf[i], ya[i], yb[i]);
              rotate_pair(u32_elem(xb, 2 * i), u32_elem(xb, 2 * i + 1), cf[4 + i], ya[4 + i], yb[4 + i]);
            }
            oa.x = pack_bf16(ya[0], yb[0]); oa.y = pack_bf16(ya[1], yb[1]);
            oa.z = pack_bf16(ya[2], yb[2]); oa.w = pack_bf16(ya[3], yb[3]);
            ob.x = pack_bf16(ya[4], yb[4]); ob.y = pack_bf16(ya[5], yb[5]);
            ob.z = pack_bf16(ya[6], yb[6]); ob.w = pack_bf16(ya[7], yb[7]);
          }
          __nv_bfloat16* dst = k_dst + (int64_t(did) * P + (opos - (opos / P) * P)) * D;
          st_stream(dst + ca, oa);
          st_stream(dst + cb, ob);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&sh.empty[st]));
    }
  }
}

template <int D, int STYLE>
cudaError_t launch_apply(const rk_rope_args& a, const float4* coef, cudaStream_t stream) {
  using C = RopeCfg<D>;
  const long long tiles = (a.max_tok + C::kRows - 1) / C::kRows;
  const long long blocks = tiles * a.n_runs;
  if (blocks == 0) return cudaSuccess;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(rope_apply_kernel<D, STYLE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  const int grid = int(std::min<long long>(blocks, 2LL * device_sm_count()));
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(grid), dim3(kRopeThreads), C::kSmem, stream, attr);
  return cudaLaunchKernelEx(&cfg, rope_apply_kernel<D, STYLE>, static_cast<const __nv_bfloat16*>(a.k_src),
                            static_cast<__nv_bfloat16*>(a.k_dst), a.n_src_pages, a.n_dst_pages, a.src_tables,
                            a.n_src_entries, a.dst_tables, a.n_dst_entries, a.runs, a.n_runs, a.P, a.max_tok, coef,
                            a.status);
}

}  // namespace


cudaError_t launch_rope_coefficients(const int32_t* deltas, int n, int d, double theta, void* coef,
                                     cudaStream_t stream) {
  rope_coeff_delta_kernel<<<n, d / 2, 0, stream>>>(deltas, n, d, theta, static_cast<float4*>(coef));
  return cudaGetLastError();
}

cudaError_t launch_rope(const rk_rope_args& a, void* workspace, cudaStream_t stream) {
  if (a.n_runs == 0) return cudaSuccess;
  float4* coef = static_cast<float4*>(workspace);
  rope_coeff_kernel<<<a.n_runs, a.d / 2, 0, stream>>>(a.runs, a.n_runs, a.d, a.theta, coef);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (a.d == 128)
    return a.style == RK_ROPE_HALF_SPLIT ? launch_apply<128, RK_ROPE_HALF_SPLIT>(a, coef, stream)
                                         : launch_apply<128, RK_ROPE_INTERLEAVED>(a, coef, stream);
  return a.style == RK_ROPE_HALF_SPLIT ? launch_apply<64, RK_ROPE_HALF_SPLIT>(a, coef, stream)
                                       : launch_apply<64, RK_ROPE_INTERLEAVED>(a, coef, stream);
}

}  // namespace rk
