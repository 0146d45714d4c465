// SegPaged decode: one query per sequence, all query heads of a KV group at once.
//
// Decode reads every visible K/V row once and does little arithmetic per byte, so the
// kernel is bound by HBM bandwidth (the "LLM 推理原理详解" entry on the last page: decode is
// memory-bandwidth bound).  CTAs take items (a slice of one head segment's visible
// page-list entries, rk_plan.cu) from a shared counter.  Each of the four warps streams
// every fourth page of the slice through its own ring of shared-memory stages, filled by
// bulk asynchronous copies (one copy per K page and per V page: pages are contiguous
// P x d rows of the pool), so several pages per warp are in flight while it computes.
// Lane l owns channels [l*CH, l*CH + CH) of every row.  Scores of TG tokens x G heads are
// reduced across lanes with a transposing butterfly (NV - 1 shuffles for NV = TG*G sums),
// after which each lane owns one (head, token) score; online softmax runs per page and
// probabilities reach every lane through shared memory for the value product.  The four
// warps' states are merged at the end of an item; split items are merged by
// combine_decode_kernel.
#include "rk_internal.cuh"
#include "rk_sm100.cuh"

#include <algorithm>

namespace rk {

namespace {

using namespace sm100;

constexpr int kDecThreads = 128;
constexpr int kDecWarps = kDecThreads / 32;

template <int D>
struct RowChunk;
template <>
struct RowChunk<128> {
  using T = uint2;  // 4 bf16
  static __device__ __forceinline__ void to_f32(const T& v, float* f) {
    f[0] = bf16lo(v.x); f[1] = bf16hi(v.x); f[2] = bf16lo(v.y); f[3] = bf16hi(v.y);
  }
};
template <>
struct RowChunk<64> {
  using T = uint32_t;  // 2 bf16
  static __device__ __forceinline__ void to_f32(const T& v, float* f) { f[0] = bf16lo(v); f[1] = bf16hi(v); }
};

template <int D, int P>
struct DecShape {
  static constexpr int kPageBytes = P * D * 2;
  static constexpr int kStages = P == 16 ? 3 : 2;                         // ring depth per warp
  static constexpr int kWarpBytes = kStages * 2 * kPageBytes;            // K + V per stage
  static constexpr int kSmem = kDecWarps * kWarpBytes;
};

__device__ __forceinline__ void bulk_copy(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

template <int D, int G, int P>
__global__ __launch_bounds__(kDecThreads) void decode_kernel(AttnParams p, AttnWorkspace ws) {
  using SH = DecShape<D, P>;
  constexpr int NS = SH::kStages;
  constexpr int CH = D / 32;
  constexpr int TG = (32 / G < P) ? 32 / G : P;   // tokens per reduce group
  constexpr int NV = TG * G;                       // sums per group (power of two, <= 32)
  constexpr int LOGNV = NV == 32 ? 5 : NV == 16 ? 4 : NV == 8 ? 3 : NV == 4 ? 2 : NV == 2 ? 1 : 0;
  constexpr int LPI = 32 / NV;                     // lanes holding the same sum
  constexpr int NGRP = P / TG;
  using RC = RowChunk<D>;

  extern __shared__ __align__(128) uint8_t dsmem[];
  __shared__ float s_p[kDecWarps][P * G];          // probabilities of the current page, [token][head]
  __shared__ float s_m[kDecWarps][G];
  __shared__ float s_l[kDecWarps][G];
  __shared__ float s_o[kDecWarps][G][D];
  __shared__ uint64_t s_full[kDecWarps][NS];
  __shared__ int s_item;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int my_idx = lane / LPI;                   // (head, token) sum this lane ends up with
  const int my_g = my_idx / TG, my_t = my_idx % TG;
  const uint32_t ring = smem_addr(dsmem) + warp * SH::kWarpBytes;
  const uint8_t* ring_ptr = dsmem + warp * SH::kWarpBytes;

  if (lane == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(smem_addr(&s_full[warp][s]), 1);
    mbar_fence_init();
  }
  __syncwarp();

  uint32_t issued = 0, consumed = 0;    // pages this warp has requested / finished (across items)
  bool failed = false;

  while (true) {
    if (threadIdx.x == 0) s_item = atomicAdd(&ws.header->counter, 1);
    __syncthreads();
    const int it = s_item;
    const bool any_failed = __syncthreads_or(failed);
    if (it >= ws.header->n_items || any_failed) break;

    const Item item = ws.items[it];
    const Unit un = ws.units[item.unit];
    const int seg = un.seg;
    const int h = seg % p.Hkv;
    const int L = __ldg(p.seq_len + un.b);
    const int pq = un.pos0;
    const int cls = __ldg(p.head_class + seg);
    const bool local = cls == RK_CLASS_LOCAL;
    const int W = local ? __ldg(p.window + seg) : 0;
    const int S = (local && p.sink) ? __ldg(p.sink + seg) : 0;
    const int32_t* trow = p.page_table + int64_t(seg) * p.max_pages;
    const int32_t* lrow = p.page_logical ? p.page_logical + int64_t(seg) * p.max_pages : nullptr;

    float q[G][CH];
    {
      const __nv_bfloat16* qp = p.q + (int64_t(un.tok0) * p.Hq + h * G) * D + lane * CH;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        typename RC::T raw = *reinterpret_cast<const typename RC::T*>(qp + g * D);
        float f[CH];
        RC::to_f32(raw, f);
#pragma unroll
        for (int c = 0; c < CH; ++c) q[g][c] = f[c] * p.scale_log2;
      }
    }
    float m[G], o[G][CH];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m[g] = -INFINITY;
#pragma unroll
      for (int c = 0; c < CH; ++c) o[g][c] = 0.f;
    }
    float lsum = 0.f;           // own (head, token-slot) partial of the denominator
    float m_own = -INFINITY;    // running maximum of the own head (equals m[my_g])

    // this warp's pages of the item: v = v_begin + warp + k*4
    const int n_mine =
        item.v_end > item.v_begin + warp ? (item.v_end - item.v_begin - warp + kDecWarps - 1) / kDecWarps : 0;
    int next_issue = 0;
    // lane 0 only: request the k-th page of this warp into the next ring stage
    auto issue = [&](int k) {
      const int s = issued % NS;
      const uint32_t bar = smem_addr(&s_full[warp][s]);
      const int v = item.v_begin + warp + k * kDecWarps;
      const int pg = __ldg(trow + unit_entry(un, v));
      if (pg >= 0 && pg < p.n_pool_pages) {
        mbar_arrive_expect_tx(bar, 2 * SH::kPageBytes);
        bulk_copy(ring + s * 2 * SH::kPageBytes, p.k_pool + int64_t(pg) * P * D, SH::kPageBytes, bar);
        bulk_copy(ring + s * 2 * SH::kPageBytes + SH::kPageBytes, p.v_pool + int64_t(pg) * P * D,
                  SH::kPageBytes, bar);
      } else {
        report(p.status, RK_ERR_DEVICE_BOUNDS);
        mbar_arrive(bar);   // completes the phase without data; the page is masked below
      }
      ++issued;
    };
    if (lane == 0)
      for (; next_issue < n_mine && next_issue < NS; ++next_issue) issue(next_issue);
    issued = __shfl_sync(0xffffffffu, issued, 0);
    next_issue = __shfl_sync(0xffffffffu, next_issue, 0);

    for (int k = 0; k < n_mine; ++k) {
      const int v = item.v_begin + warp + k * kDecWarps;
      const int e = unit_entry(un, v);
      const int page = __ldg(trow + e);
      const bool page_ok = page >= 0 && page < p.n_pool_pages;
      const int lp = lrow ? __ldg(lrow + e) : e;
      const int s = consumed % NS;
      const bool got = mbar_wait(smem_addr(&s_full[warp][s]), (consumed / NS) & 1);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) report(p.status, RK_ERR_TIMEOUT);
        failed = true;
        break;
      }
      const uint8_t* kb = ring_ptr + s * 2 * SH::kPageBytes + lane * CH * 2;
      const uint8_t* vb = kb + SH::kPageBytes;

      // scores: one (head, token) value per lane and group
      float sc[NGRP];
#pragma unroll
      for (int grp = 0; grp < NGRP; ++grp) {
        float part[NV];
#pragma unroll
        for (int t = 0; t < TG; ++t) {
          float kf[CH];
          RC::to_f32(*reinterpret_cast<const typename RC::T*>(kb + (grp * TG + t) * D * 2), kf);
#pragma unroll
          for (int g = 0; g < G; ++g) {
            float acc = 0.f;
#pragma unroll
            for (int c = 0; c < CH; ++c) acc = fmaf(q[g][c], kf[c], acc);
            part[g * TG + t] = acc;
          }
        }
        // transposing butterfly: at each of the first LOGNV levels a lane keeps the half
        // of its sums selected by its lane bit and adds the partner's copy of that half
        int cnt = NV;
#pragma unroll
        for (int lvl = 0; lvl < 5; ++lvl) {
          const int off = 16 >> lvl;
          if (lvl < LOGNV) {
            const int half = cnt >> 1;
            const bool upper = (lane & off) != 0;
#pragma unroll
            for (int i = 0; i < NV / 2; ++i) {
              if (i < half) {
                const float send = upper ? part[i] : part[i + half];
                const float keep = upper ? part[i + half] : part[i];
                part[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
              }
            }
            cnt = half;
          } else {
            part[0] += __shfl_xor_sync(0xffffffffu, part[0], off);
          }
        }
        const int j = lp * P + grp * TG + my_t;
        const bool vis = page_ok && j < L && j <= pq && (!local || j > pq - W || j < S);
        sc[grp] = vis ? part[0] : -INFINITY;
      }

      // online softmax over the page
      float mx = sc[0];
#pragma unroll
      for (int grp = 1; grp < NGRP; ++grp) mx = fmaxf(mx, sc[grp]);
#pragma unroll
      for (int off = 1; off < TG * LPI; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      // mx is the page maximum of this lane's own head; every lane also needs the new
      // maxima of all heads to rescale its accumulators
      float alpha[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float mg = __shfl_sync(0xffffffffu, mx, g * TG * LPI);
        const float mn = fmaxf(m[g], mg);
        alpha[g] = (mn == -INFINITY) ? 1.f : fast_exp2(m[g] - mn);
        m[g] = mn;
      }
      const float m_new_own = fmaxf(m_own, mx);
      const float alpha_own = (m_new_own == -INFINITY) ? 1.f : fast_exp2(m_own - m_new_own);
      m_own = m_new_own;
      float psum = 0.f;
#pragma unroll
      for (int grp = 0; grp < NGRP; ++grp) {
        const float pv = (m_own == -INFINITY) ? 0.f : fast_exp2(sc[grp] - m_own);
        psum += pv;
        if (lane % LPI == 0) s_p[warp][(grp * TG + my_t) * G + my_g] = pv;
      }
      lsum = lsum * alpha_own + psum;
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int c = 0; c < CH; ++c) o[g][c] *= alpha[g];
      __syncwarp();
#pragma unroll
      for (int t = 0; t < P; ++t) {
        float vf[CH];
        RC::to_f32(*reinterpret_cast<const typename RC::T*>(vb + t * D * 2), vf);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float pg = s_p[warp][t * G + g];
#pragma unroll
          for (int c = 0; c < CH; ++c) o[g][c] = fmaf(pg, vf[c], o[g][c]);
        }
      }
      __syncwarp();   // stage s and s_p fully read before they are refilled
      ++consumed;
      if (lane == 0 && next_issue < n_mine) issue(next_issue++);
      issued = __shfl_sync(0xffffffffu, issued, 0);
      next_issue = __shfl_sync(0xffffffffu, next_issue, 0);
    }

    // merge the four warps
#pragma unroll
    for (int off = LPI; off < TG * LPI; off <<= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
    if (lane % (TG * LPI) == 0) s_l[warp][my_g] = lsum;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      if (lane == 0) s_m[warp][g] = m[g];
#pragma unroll
      for (int c = 0; c < CH; ++c) s_o[warp][g][lane * CH + c] = o[g][c];
    }
    __syncthreads();

    const bool split = un.n_splits > 1;
    for (int x = threadIdx.x; x < G * D; x += kDecThreads) {
      const int g = x / D, ch = x % D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, s_m[w][g]);
      float den = 0.f, num = 0.f;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) {
        const float wt = (M == -INFINITY) ? 0.f : fast_exp2(s_m[w][g] - M);
        den += wt * s_l[w][g];
        num += wt * s_o[w][g][ch];
      }
      const float val = den > 0.f ? num / den : 0.f;
      const float lse_nat = den > 0.f ? (M + fast_log2(den)) * 0.69314718055994531f : -INFINITY;
      const int hq = h * G + g;
      if (!split) {
        p.out[(int64_t(un.tok0) * p.Hq + hq) * D + ch] = __float2bfloat16_rn(val);
        if (p.lse && ch == 0) p.lse[int64_t(un.tok0) * p.Hq + hq] = lse_nat;
      } else {
        ws.part_o[(int64_t(it) * ws.rows + g) * D + ch] = val;
        if (ch == 0) ws.part_lse[int64_t(it) * ws.rows + g] = lse_nat;
      }
    }
  }
  // copies still in flight (only after a failure): let them land before the CTA exits
  if (lane == 0 && issued > consumed)
    for (uint32_t k = consumed; k < issued; ++k) mbar_wait(smem_addr(&s_full[warp][k % NS]), (k / NS) & 1);
  __syncwarp();
}

// Merge the split partials of decode units: one block per (unit, query head of the group);
// the four warps take every fourth split, lanes cover the head dimension.
template <int D>
__global__ __launch_bounds__(128) void combine_decode_kernel(AttnParams p, AttnWorkspace ws) {
  constexpr int CH = D / 32;
  __shared__ float s_m[4], s_den[4], s_num[4][D];
  const int u = blockIdx.x, g = blockIdx.y;
  if (u >= ws.header->n_units) return;
  const Unit un = ws.units[u];
  if (un.n_splits <= 1) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float M = -INFINITY;
  for (int s = threadIdx.x; s < un.n_splits; s += 128) M = fmaxf(M, ws.part_lse[int64_t(unit_item(un, s)) * ws.rows + g]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  if (lane == 0) s_m[warp] = M;
  __syncthreads();
  M = fmaxf(fmaxf(s_m[0], s_m[1]), fmaxf(s_m[2], s_m[3]));
  float den = 0.f, num[CH];
#pragma unroll
  for (int c = 0; c < CH; ++c) num[c] = 0.f;
#pragma unroll 4
  for (int s = warp; s < un.n_splits; s += 4) {
    const int64_t it = unit_item(un, s);
    const float l = ws.part_lse[it * ws.rows + g];
    const float w = (M == -INFINITY) ? 0.f : __expf(l - M);
    den += w;
    const float* po = ws.part_o + (it * ws.rows + g) * D + lane * CH;
#pragma unroll
    for (int c = 0; c < CH; ++c) num[c] += w * po[c];
  }
  if (lane == 0) s_den[warp] = den;
#pragma unroll
  for (int c = 0; c < CH; ++c) s_num[warp][lane * CH + c] = num[c];
  __syncthreads();
  if (warp == 0) {
    const float dsum = s_den[0] + s_den[1] + s_den[2] + s_den[3];
    const float inv = dsum > 0.f ? 1.f / dsum : 0.f;
    const int hq = (un.seg % p.Hkv) * p.G + g;
    __nv_bfloat16* o = p.out + (int64_t(un.tok0) * p.Hq + hq) * D;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int ch = lane * CH + c;
      o[ch] = __float2bfloat16_rn((s_num[0][ch] + s_num[1][ch] + s_num[2][ch] + s_num[3][ch]) * inv);
    }
    if (p.lse && lane == 0) p.lse[int64_t(un.tok0) * p.Hq + hq] = dsum > 0.f ? M + logf(dsum) : -INFINITY;
  }
}

template <int D, int G, int P>
cudaError_t launch_t(const AttnParams& p, const AttnWorkspace& ws, int grid, cudaStream_t stream) {
  using SH = DecShape<D, P>;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, G, P>, cudaFuncAttributeMaxDynamicSharedMemorySize, SH::kSmem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  decode_kernel<D, G, P><<<grid, kDecThreads, SH::kSmem, stream>>>(p, ws);
  return cudaGetLastError();
}

template <int D, int G>
cudaError_t launch_p(const AttnParams& p, const AttnWorkspace& ws, int grid, cudaStream_t stream) {
  return p.P == 16 ? launch_t<D, G, 16>(p, ws, grid, stream) : launch_t<D, G, 32>(p, ws, grid, stream);
}

template <int D>
cudaError_t launch_g(const AttnParams& p, const AttnWorkspace& ws, int grid, cudaStream_t stream) {
  switch (p.G) {
    case 1: return launch_p<D, 1>(p, ws, grid, stream);
    case 2: return launch_p<D, 2>(p, ws, grid, stream);
    case 4: return launch_p<D, 4>(p, ws, grid, stream);
    case 8: return launch_p<D, 8>(p, ws, grid, stream);
    case 16: return launch_p<D, 16>(p, ws, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int decode_ctas_per_sm(int P) { return P == 16 ? 2 : 1; }

cudaError_t launch_decode(const AttnParams& p, const AttnWorkspace& ws, int grid, cudaStream_t stream) {
  return p.d == 128 ? launch_g<128>(p, ws, grid, stream) : launch_g<64>(p, ws, grid, stream);
}

cudaError_t launch_combine_decode(const AttnParams& p, const AttnWorkspace& ws, cudaStream_t stream) {
  dim3 grid(std::max(1, ws.max_units), p.G);
  if (p.d == 128) combine_decode_kernel<128><<<grid, 128, 0, stream>>>(p, ws);
  else combine_decode_kernel<64><<<grid, 128, 0, stream>>>(p, ws);
  return cudaGetLastError();
}

}  // namespace rk
