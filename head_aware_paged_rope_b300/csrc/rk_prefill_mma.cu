// SegPaged prefill, warp-level tensor-core version (mma.sync m16n8k16, bf16 -> fp32).
//
// Each item (rk_plan.cu) is one slice of the visible page-list entries of one
// (query tile, KV head) unit.  The query tile packs ROWS = 64 rows as (token, head of
// the KV group), so all G query heads sharing a KV head read each K/V tile once.  K/V
// tiles of KEYS = 64 keys are gathered page by page straight from the pool through the
// head's page table with 16-byte cp.async (no attention mask anywhere: the visible set is
// the list of entries plus an in-register predicate for the causal / window edge,
// "小红书 RedKnot" section 3, fourth component).  Softmax is the usual online
// (running max, running sum) form; probabilities are fed to the value product as bf16.
//
// This kernel is the legacy-tensor-core baseline of the prefill path.
#include "rk_internal.cuh"

#include <algorithm>

namespace rk {

namespace {

constexpr int kRows = 64;
constexpr int kKeys = 64;
constexpr int kThreads = 128;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" :: "r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
               : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
               : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// 16-byte chunk ch of row r in a [rows][D] bf16 tile, XOR-swizzled against ldmatrix bank conflicts
template <int D>
__device__ __forceinline__ uint32_t swz(uint32_t base, int r, int ch) {
  return base + r * (D * 2) + ((ch ^ (r & 7)) << 4);
}

template <int D, int P>
struct PrefillSmem {
  static constexpr int kEPT = kKeys / P;        // page-list entries per key tile
  static constexpr int kTile = kKeys * D * 2;   // bytes of one K (or V) tile
  static constexpr int kQ = kRows * D * 2;
  static constexpr int kBytes = kQ + 4 * kTile + 2 * kEPT * 4;
};

template <int D, int P>
__global__ __launch_bounds__(kThreads) void prefill_mma_kernel(AttnParams p, AttnWorkspace ws) {
  using SM = PrefillSmem<D, P>;
  constexpr int EPT = SM::kEPT;
  constexpr int CHUNKS = D / 8;       // 16-byte chunks per row
  constexpr int KS = D / 16;          // k-steps of Q.K^T
  constexpr int NT = kKeys / 8;       // n-tiles of S
  constexpr int DT = D / 8;           // n-tiles of O

  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sK0 = sQ + SM::kQ;
  const uint32_t sV0 = sK0 + 2 * SM::kTile;
  int* s_lp = reinterpret_cast<int*>(smem + SM::kQ + 4 * SM::kTile);   // [2][EPT]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.G;
  const int n_items = ws.header->n_items;

  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    const Item item = ws.items[it];
    const Unit un = ws.units[item.unit];
    const int seg = un.seg;
    const int h = seg % p.Hkv;
    const int L = __ldg(p.seq_len + un.b);
    const int cls = __ldg(p.head_class + seg);
    const bool local = cls == RK_CLASS_LOCAL;
    const int W = local ? __ldg(p.window + seg) : 0;
    const int S = (local && p.sink) ? __ldg(p.sink + seg) : 0;
    const int rows_valid = un.ntok * G;
    const int32_t* trow = p.page_table + int64_t(seg) * p.max_pages;
    const int32_t* lrow = p.page_logical ? p.page_logical + int64_t(seg) * p.max_pages : nullptr;
    const int n_kt = (item.v_end - item.v_begin + EPT - 1) / EPT;

    // Q tile: rows (token t, head g) -> q[tok0 + t][h*G + g]
    for (int c = tid; c < kRows * CHUNKS; c += kThreads) {
      const int r = c / CHUNKS, ch = c % CHUNKS;
      const bool valid = r < rows_valid;
      const int t = valid ? r / G : 0, g = valid ? r % G : 0;
      const __nv_bfloat16* src = valid ? p.q + (int64_t(un.tok0 + t) * p.Hq + h * G + g) * D + ch * 8 : p.q;
      cp_async16(swz<D>(sQ, r, ch), src, valid);
    }

    auto load_tile = [&](int kt, int stage) {
      const int v0 = item.v_begin + kt * EPT;
      const uint32_t dK = sK0 + stage * SM::kTile, dV = sV0 + stage * SM::kTile;
      for (int c = tid; c < kKeys * CHUNKS; c += kThreads) {
        const int r = c / CHUNKS, ch = c % CHUNKS;
        const int v = v0 + r / P;
        int page = -1;
        if (v < item.v_end) {
          page = __ldg(trow + unit_entry(un, v));
          if (page < 0 || page >= p.n_pool_pages) {
            report(p.status, RK_ERR_DEVICE_BOUNDS);
            page = -1;
          }
        }
        const int64_t off = page >= 0 ? (int64_t(page) * P + (r % P)) * D + ch * 8 : 0;
        cp_async16(swz<D>(dK, r, ch), p.k_pool + off, page >= 0);
        cp_async16(swz<D>(dV, r, ch), p.v_pool + off, page >= 0);
      }
      if (tid < EPT) {
        const int v = v0 + tid;
        int lp = -1;
        if (v < item.v_end) {
          const int e = unit_entry(un, v);
          const int page = __ldg(trow + e);
          lp = (page >= 0 && page < p.n_pool_pages) ? (lrow ? __ldg(lrow + e) : e) : -1;
        }
        s_lp[stage * EPT + tid] = lp;
      }
    };

    if (n_kt > 0) load_tile(0, 0);
    cp_async_commit();

    // per-thread rows: r0 = 16*warp + lane/4 and r0 + 8
    const int r0 = warp * 16 + (lane >> 2);
    const int pos_r0 = un.pos0 + r0 / G, pos_r1 = un.pos0 + (r0 + 8) / G;
    const int wrow_lo = warp * 16, wrow_hi = min(warp * 16 + 15, max(rows_valid - 1, 0));
    const int wpos_lo = un.pos0 + wrow_lo / G, wpos_hi = un.pos0 + wrow_hi / G;

    float o[DT][4];
#pragma unroll
    for (int i = 0; i < DT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    uint32_t qf[KS][4];

    for (int kt = 0; kt < n_kt; ++kt) {
      const int stage = kt & 1;
      if (kt + 1 < n_kt) load_tile(kt + 1, stage ^ 1);
      cp_async_commit();
      cp_async_wait<1>();
      __syncthreads();
      if (kt == 0) {
#pragma unroll
        for (int ks = 0; ks < KS; ++ks)
          ldsm_x4(swz<D>(sQ, warp * 16 + (lane & 15), 2 * ks + (lane >> 4)), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
      }
      const uint32_t sK = sK0 + stage * SM::kTile, sV = sV0 + stage * SM::kTile;

      float s[NT][4];
#pragma unroll
      for (int i = 0; i < NT; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
      for (int np = 0; np < NT / 2; ++np) {
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          uint32_t b0, b1, b2, b3;
          const int krow = np * 16 + (lane & 7) + ((lane >> 4) << 3);
          ldsm_x4(swz<D>(sK, krow, 2 * ks + ((lane >> 3) & 1)), b0, b1, b2, b3);
          mma16816(s[2 * np], qf[ks], b0, b1);
          mma16816(s[2 * np + 1], qf[ks], b2, b3);
        }
      }

      // visibility: whole tile visible to all rows of this warp, or per element
      const int* lps = s_lp + stage * EPT;
      bool full = true;
      int lp_first = lps[0], lp_last = lps[0];
#pragma unroll
      for (int i = 0; i < EPT; ++i) {
        full = full && lps[i] >= 0;
        lp_last = lps[i] >= 0 ? lps[i] : lp_last;
      }
      const int j_min = lp_first * P, j_max = lp_last * P + P - 1;
      full = full && j_max <= wpos_lo && j_max < L && (!local || j_min > wpos_hi - W || j_max < S);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float x = s[nt][c] * p.scale_log2;
          if (!full) {
            const int col = nt * 8 + 2 * (lane & 3) + (c & 1);
            const int lp = lps[col / P];
            const int j = lp * P + (col % P);
            const int pos = (c < 2) ? pos_r0 : pos_r1;
            const bool vis = lp >= 0 && j < L && j <= pos && (!local || j > pos - W || j < S);
            if (!vis) x = -INFINITY;
          }
          s[nt][c] = x;
        }
      }

      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
        mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float a0 = mn0 == -INFINITY ? 1.f : fast_exp2(m0 - mn0);
      const float a1 = mn1 == -INFINITY ? 1.f : fast_exp2(m1 - mn1);
      const float ref0 = mn0 == -INFINITY ? 0.f : mn0, ref1 = mn1 == -INFINITY ? 0.f : mn1;
      m0 = mn0;
      m1 = mn1;
      float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        s[nt][0] = fast_exp2(s[nt][0] - ref0);
        s[nt][1] = fast_exp2(s[nt][1] - ref0);
        s[nt][2] = fast_exp2(s[nt][2] - ref1);
        s[nt][3] = fast_exp2(s[nt][3] - ref1);
        ps0 += s[nt][0] + s[nt][1];
        ps1 += s[nt][2] + s[nt][3];
      }
      l0 = l0 * a0 + ps0;
      l1 = l1 * a1 + ps1;
#pragma unroll
      for (int dt = 0; dt < DT; ++dt) {
        o[dt][0] *= a0; o[dt][1] *= a0;
        o[dt][2] *= a1; o[dt][3] *= a1;
      }

#pragma unroll
      for (int kk = 0; kk < kKeys / 16; ++kk) {
        uint32_t a[4];
        a[0] = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
        a[1] = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
        a[2] = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
        a[3] = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
        for (int dp = 0; dp < DT / 2; ++dp) {
          uint32_t b0, b1, b2, b3;
          const int vrow = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
          ldsm_x4_t(swz<D>(sV, vrow, 2 * dp + (lane >> 4)), b0, b1, b2, b3);
          mma16816(o[2 * dp], a, b0, b1);
          mma16816(o[2 * dp + 1], a, b2, b3);
        }
      }
      __syncthreads();
    }
    cp_async_wait<0>();

    // epilogue
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
    const float ln2 = 0.69314718055994531f;
    const float lse0 = l0 > 0.f ? (m0 + fast_log2(l0)) * ln2 : -INFINITY;
    const float lse1 = l1 > 0.f ? (m1 + fast_log2(l1)) * ln2 : -INFINITY;
    const bool split = un.n_splits > 1;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int r = r0 + half * 8;
      if (r >= rows_valid) continue;
      const float inv = half ? inv1 : inv0;
      const float lse = half ? lse1 : lse0;
      const int t = un.tok0 + r / G, hq = h * G + r % G;
      if (!split) {
        __nv_bfloat16* orow = p.out + (int64_t(t) * p.Hq + hq) * D;
#pragma unroll
        for (int dt = 0; dt < DT; ++dt) {
          const int col = dt * 8 + 2 * (lane & 3);
          *reinterpret_cast<uint32_t*>(orow + col) = pack_bf16(o[dt][2 * half] * inv, o[dt][2 * half + 1] * inv);
        }
        if (p.lse && (lane & 3) == 0) p.lse[int64_t(t) * p.Hq + hq] = lse;
      } else {
        float* prow = ws.part_o + (int64_t(it) * ws.rows + r) * D;
#pragma unroll
        for (int dt = 0; dt < DT; ++dt) {
          const int col = dt * 8 + 2 * (lane & 3);
          *reinterpret_cast<float2*>(prow + col) = make_float2(o[dt][2 * half] * inv, o[dt][2 * half + 1] * inv);
        }
        if ((lane & 3) == 0) ws.part_lse[int64_t(it) * ws.rows + r] = lse;
      }
    }
    __syncthreads();
  }
}

template <int D, int P>
cudaError_t launch_dp(const AttnParams& p, const AttnWorkspace& ws, int grid, cudaStream_t stream) {
  const int smem = PrefillSmem<D, P>::kBytes;
  static bool attr_set[64] = {false};   // per device; set once, outside any later graph capture
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(prefill_mma_kernel<D, P>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  prefill_mma_kernel<D, P><<<grid, kThreads, smem, stream>>>(p, ws);
  return cudaGetLastError();
}

}  // namespace

int prefill_mma_rows() { return kRows; }
int prefill_mma_keys() { return kKeys; }

cudaError_t launch_prefill_mma(const AttnParams& p, const AttnWorkspace& ws, int grid, cudaStream_t stream) {
  if (p.d == 128) return p.P == 16 ? launch_dp<128, 16>(p, ws, grid, stream) : launch_dp<128, 32>(p, ws, grid, stream);
  return p.P == 16 ? launch_dp<64, 16>(p, ws, grid, stream) : launch_dp<64, 32>(p, ws, grid, stream);
}

}  // namespace rk
