// SegPaged decode: one query per sequence, all query heads of a KV group at once.
//
// Decode reads every visible K/V row once and does little arithmetic per byte, so the
// kernel is bound by HBM bandwidth (the "LLM 推理原理详解" entry on the last page: decode is
// memory-bandwidth bound).  Each CTA takes items (a slice of one head segment's visible
// page-list entries, see rk_plan.cu); each warp streams whole pages of that slice.
// Inside a warp lane l owns channels [l*CH, l*CH + CH) of every row, so a K or V row is
// one coalesced 256-byte (d = 128) warp access.  Scores of a group of TG tokens x G heads
// are reduced across lanes with a transposing butterfly (TG*G - 1 shuffles for 32 sums),
// after which each lane owns one (head, token) score.  Online softmax runs per page;
// probabilities reach every lane through shared memory for the value product.  The four
// warps' states are merged at the end of an item, and split items are merged by the
// combine kernel.
#include "rk_internal.cuh"

#include <algorithm>

namespace rk {

namespace {

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

template <int D, int G, int P>
__global__ __launch_bounds__(kDecThreads) void decode_kernel(AttnParams p, AttnWorkspace ws) {
  constexpr int CH = D / 32;
  constexpr int TG = (32 / G < P) ? 32 / G : P;   // tokens per reduce group
  constexpr int NV = TG * G;                       // sums per group (power of two, <= 32)
  constexpr int LOGNV = NV == 32 ? 5 : NV == 16 ? 4 : NV == 8 ? 3 : NV == 4 ? 2 : NV == 2 ? 1 : 0;
  constexpr int LPI = 32 / NV;                     // lanes holding the same sum
  constexpr int NGRP = P / TG;
  using RC = RowChunk<D>;

  __shared__ float s_p[kDecWarps][P * G];          // probabilities of the current page, [token][head]
  __shared__ float s_m[kDecWarps][G];
  __shared__ float s_l[kDecWarps][G];
  __shared__ float s_o[kDecWarps][G][D];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int my_idx = lane / LPI;                   // (head, token) sum this lane ends up with
  const int my_g = my_idx / TG, my_t = my_idx % TG;
  const int n_items = ws.header->n_items;

  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    const Item item = ws.items[it];
    const Unit un = ws.units[item.unit];
    const int seg = un.seg;
    const int h = seg % p.Hkv;
    const int L = __ldg(p.seq_len + un.b);
    const int pq = un.pos0;
    const int cls = __ldg(p.head_class + seg);
    const int W = cls == RK_CLASS_LOCAL ? __ldg(p.window + seg) : 0;
    const int S = (cls == RK_CLASS_LOCAL && p.sink) ? __ldg(p.sink + seg) : 0;
    const bool local = cls == RK_CLASS_LOCAL;

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
    float lsum = 0.f;   // own (head, token-slot) partial of the denominator
    float m_own = -INFINITY;  // running maximum of the own head (equals m[my_g])

    const int32_t* trow = p.page_table + int64_t(seg) * p.max_pages;
    const int32_t* lrow = p.page_logical ? p.page_logical + int64_t(seg) * p.max_pages : nullptr;

    for (int v = item.v_begin + warp; v < item.v_end; v += kDecWarps) {
      const int e = unit_entry(un, v);
      const int page = __ldg(trow + e);
      const int lp = lrow ? __ldg(lrow + e) : e;
      if (page < 0 || page >= p.n_pool_pages) {
        if (lane == 0) report(p.status, RK_ERR_DEVICE_BOUNDS);
        continue;
      }
      const __nv_bfloat16* kb = p.k_pool + int64_t(page) * P * D + lane * CH;
      const __nv_bfloat16* vb = p.v_pool + int64_t(page) * P * D + lane * CH;
      typename RC::T kr[P], vr[P];
#pragma unroll
      for (int t = 0; t < P; ++t) kr[t] = __ldg(reinterpret_cast<const typename RC::T*>(kb + t * D));
#pragma unroll
      for (int t = 0; t < P; ++t) vr[t] = __ldg(reinterpret_cast<const typename RC::T*>(vb + t * D));

      // scores: one (head, token) value per lane and group
      float sc[NGRP];
#pragma unroll
      for (int grp = 0; grp < NGRP; ++grp) {
        float part[NV];
#pragma unroll
        for (int t = 0; t < TG; ++t) {
          float kf[CH];
          RC::to_f32(kr[grp * TG + t], kf);
#pragma unroll
          for (int g = 0; g < G; ++g) {
            float acc = 0.f;
#pragma unroll
            for (int c = 0; c < CH; ++c) acc = fmaf(q[g][c], kf[c], acc);
            part[g * TG + t] = acc;
          }
        }
        // transposing butterfly: after level k the lane keeps the half of the sums
        // selected by its lane bit; sums are complete after all five levels
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
        const bool vis = j < L && j <= pq && (!local || j > pq - W || j < S);
        sc[grp] = vis ? part[0] : -INFINITY;
      }

      // online softmax over the page
      float mx = sc[0];
#pragma unroll
      for (int grp = 1; grp < NGRP; ++grp) mx = fmaxf(mx, sc[grp]);
#pragma unroll
      for (int off = 1; off < TG * LPI; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      // mx is now the page maximum of this lane's own head; every lane also needs the
      // new maxima of all heads to rescale its accumulators
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
        RC::to_f32(vr[t], vf);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float pg = s_p[warp][t * G + g];
#pragma unroll
          for (int c = 0; c < CH; ++c) o[g][c] = fmaf(pg, vf[c], o[g][c]);
        }
      }
      __syncwarp();
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
    __syncthreads();
  }
}

template <int D, int G, int P>
cudaError_t launch_t(const AttnParams& p, const AttnWorkspace& ws, int grid, cudaStream_t stream) {
  decode_kernel<D, G, P><<<grid, kDecThreads, 0, stream>>>(p, ws);
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

cudaError_t launch_decode(const AttnParams& p, const AttnWorkspace& ws, int grid, cudaStream_t stream) {
  return p.d == 128 ? launch_g<128>(p, ws, grid, stream) : launch_g<64>(p, ws, grid, stream);
}

}  // namespace rk
