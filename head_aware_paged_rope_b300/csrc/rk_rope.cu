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

namespace rk {

namespace {

__global__ void rope_coeff_kernel(const rk_rope_run* __restrict__ runs, int n_runs, int d,
                                  double theta, float4* __restrict__ coef) {
  const int run = blockIdx.x;
  const int i = threadIdx.x;
  if (run >= n_runs || i >= d / 2) return;
  const rk_rope_run r = runs[run];
  const double delta = double((long long)r.pos_on0 - (long long)r.pos_off0);
  const double w = pow(theta, -2.0 * double(i) / double(d));
  double s, c;
  sincos(delta * w, &s, &c);
  const float c_hi = __uint_as_float(__float_as_uint(__double2float_rn(c)) & 0xFFFFFF00u);
  const float s_hi = __uint_as_float(__float_as_uint(__double2float_rn(s)) & 0xFFFFFF00u);
  const float c_lo = __double2float_rn(c - double(c_hi));
  const float s_lo = __double2float_rn(s - double(s_hi));
  coef[size_t(run) * (d / 2) + i] = make_float4(c_hi, c_lo, s_hi, s_lo);
}

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ void st_stream(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w) : "memory");
}

__device__ __forceinline__ float u32_elem(const uint4& v, int k) {
  const uint32_t w = (k >> 1) == 0 ? v.x : (k >> 1) == 1 ? v.y : (k >> 1) == 2 ? v.z : v.w;
  return (k & 1) ? bf16hi(w) : bf16lo(w);
}

// Rotation of one pair with split coefficients; see the file comment.
__device__ __forceinline__ void rotate_pair(float xa, float xb, const float4& cf, float& ya, float& yb) {
  const float hi_a = fmaf(xa, cf.x, -(xb * cf.z));   // xa*c_hi - xb*s_hi (both products exact)
  const float lo_a = fmaf(xa, cf.y, -(xb * cf.w));
  const float hi_b = fmaf(xa, cf.z, xb * cf.x);      // xa*s_hi + xb*c_hi
  const float lo_b = fmaf(xa, cf.w, xb * cf.y);
  ya = hi_a + lo_a;
  yb = hi_b + lo_b;
}

constexpr int kRopeThreads = 256;
constexpr int kRopeUnroll = 4;

template <int D>
struct RopeShape {
  static constexpr int lanes_per_row = D / 16;                  // each lane: 16 channels (8 pairs)
  static constexpr int rows_per_pass = kRopeThreads / lanes_per_row;
  static constexpr int rows_per_cta = rows_per_pass * kRopeUnroll;
};

template <int D, int STYLE>
__global__ __launch_bounds__(kRopeThreads) void rope_apply_kernel(
    const __nv_bfloat16* __restrict__ k_src, __nv_bfloat16* __restrict__ k_dst, int64_t n_src_pages,
    int64_t n_dst_pages, const int32_t* __restrict__ src_tables, int64_t n_src_entries,
    const int32_t* __restrict__ dst_tables, int64_t n_dst_entries, const rk_rope_run* __restrict__ runs,
    int P, int max_tok, const float4* __restrict__ coef, int32_t* status) {
  using S = RopeShape<D>;
  const int run = blockIdx.x;
  const rk_rope_run r = runs[run];
  const int t0 = blockIdx.y * S::rows_per_cta;
  if (blockIdx.y == 0 && threadIdx.x == 0 &&
      (r.n_tok > max_tok || r.n_tok < 0 || r.pos_off0 < 0 || r.pos_on0 < 0))
    report(status, RK_ERR_DEVICE_BOUNDS);
  const int n_tok = min(r.n_tok, max_tok);
  if (t0 >= n_tok || r.pos_off0 < 0 || r.pos_on0 < 0) return;

  const int lane = threadIdx.x % S::lanes_per_row;   // pairs 8*lane .. 8*lane+7
  const int row = threadIdx.x / S::lanes_per_row;

  // channel offsets (elements) of the two 16-byte chunks this lane owns
  const int ca = STYLE == RK_ROPE_HALF_SPLIT ? 8 * lane : 16 * lane;
  const int cb = STYLE == RK_ROPE_HALF_SPLIT ? D / 2 + 8 * lane : 16 * lane + 8;

  uint4 xa[kRopeUnroll], xb[kRopeUnroll];
  int64_t dst_off[kRopeUnroll];
#pragma unroll
  for (int u = 0; u < kRopeUnroll; ++u) {
    dst_off[u] = -1;
    const int t = t0 + u * S::rows_per_pass + row;
    if (t >= n_tok) continue;
    const int s = r.pos_off0 + t;
    const int o = r.pos_on0 + t;
    const int si = s / P, oi = o / P;
    if (si >= r.src_tab_len || oi >= r.dst_tab_len || int64_t(r.src_tab_off) + si >= n_src_entries ||
        int64_t(r.dst_tab_off) + oi >= n_dst_entries || r.src_tab_off < 0 || r.dst_tab_off < 0) {
      report(status, RK_ERR_DEVICE_BOUNDS);
      continue;
    }
    const int sp = __ldg(src_tables + r.src_tab_off + si);
    const int dp = __ldg(dst_tables + r.dst_tab_off + oi);
    if (sp < 0 || sp >= n_src_pages || dp < 0 || dp >= n_dst_pages) {
      report(status, RK_ERR_DEVICE_BOUNDS);
      continue;
    }
    const __nv_bfloat16* src = k_src + (int64_t(sp) * P + (s - si * P)) * D;
    xa[u] = ld_stream(src + ca);
    xb[u] = ld_stream(src + cb);
    dst_off[u] = (int64_t(dp) * P + (o - oi * P)) * D;
  }

  float4 cf[8];
  const float4* cr = coef + size_t(run) * (D / 2) + 8 * lane;
#pragma unroll
  for (int m = 0; m < 8; ++m) cf[m] = __ldg(cr + m);

#pragma unroll
  for (int u = 0; u < kRopeUnroll; ++u) {
    if (dst_off[u] < 0) continue;
    float ya[8], yb[8];
    if (STYLE == RK_ROPE_HALF_SPLIT) {
#pragma unroll
      for (int m = 0; m < 8; ++m) rotate_pair(u32_elem(xa[u], m), u32_elem(xb[u], m), cf[m], ya[m], yb[m]);
      uint4 oa, ob;
      oa.x = pack_bf16(ya[0], ya[1]); oa.y = pack_bf16(ya[2], ya[3]);
      oa.z = pack_bf16(ya[4], ya[5]); oa.w = pack_bf16(ya[6], ya[7]);
      ob.x = pack_bf16(yb[0], yb[1]); ob.y = pack_bf16(yb[2], yb[3]);
      ob.z = pack_bf16(yb[4], yb[5]); ob.w = pack_bf16(yb[6], yb[7]);
      st_stream(k_dst + dst_off[u] + ca, oa);
      st_stream(k_dst + dst_off[u] + cb, ob);
    } else {
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        rotate_pair(u32_elem(xa[u], 2 * m), u32_elem(xa[u], 2 * m + 1), cf[m], ya[m], yb[m]);
        rotate_pair(u32_elem(xb[u], 2 * m), u32_elem(xb[u], 2 * m + 1), cf[4 + m], ya[4 + m], yb[4 + m]);
      }
      uint4 oa, ob;
      oa.x = pack_bf16(ya[0], yb[0]); oa.y = pack_bf16(ya[1], yb[1]);
      oa.z = pack_bf16(ya[2], yb[2]); oa.w = pack_bf16(ya[3], yb[3]);
      ob.x = pack_bf16(ya[4], yb[4]); ob.y = pack_bf16(ya[5], yb[5]);
      ob.z = pack_bf16(ya[6], yb[6]); ob.w = pack_bf16(ya[7], yb[7]);
      st_stream(k_dst + dst_off[u] + ca, oa);
      st_stream(k_dst + dst_off[u] + cb, ob);
    }
  }
}

template <int D, int STYLE>
cudaError_t launch_apply(const rk_rope_args& a, const float4* coef, cudaStream_t stream) {
  using S = RopeShape<D>;
  const int tiles = (a.max_tok + S::rows_per_cta - 1) / S::rows_per_cta;
  if (tiles == 0 || a.n_runs == 0) return cudaSuccess;
  dim3 grid(a.n_runs, tiles);
  rope_apply_kernel<D, STYLE><<<grid, kRopeThreads, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(a.k_src), static_cast<__nv_bfloat16*>(a.k_dst), a.n_src_pages,
      a.n_dst_pages, a.src_tables, a.n_src_entries, a.dst_tables, a.n_dst_entries, a.runs, a.P,
      a.max_tok, coef, a.status);
  return cudaGetLastError();
}

}  // namespace

int rope_rows_per_cta(int d) { return d == 64 ? RopeShape<64>::rows_per_cta : RopeShape<128>::rows_per_cta; }

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
