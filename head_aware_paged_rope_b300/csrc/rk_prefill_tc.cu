// SegPaged prefill on the 5th-generation tensor cores (tcgen05 + TMEM), sm_103a.
//
// What it computes is stated in include/rk_api.h: attention of each query over the keys
// its KV head lists in its own page table, with the causal / window edge applied as a
// predicate, never as an attn_mask tensor ("小红书 RedKnot" section 3, fourth component;
// "RedKnot" article, SegPagedAttention paragraph).
//
// One CTA = 6 warps working on items (rk_plan.cu) of 128 query rows (GQA-packed: 128/G
// tokens x the G query heads of one KV head) against a slice of that head's page list:
//   warp 4   producer: TMA loads the Q tile once per item, then for every 128-key tile
//            gathers its pages (8 of 16 tokens or 4 of 32) from the shared pool through the
//            page table, each page as one or two 64-column boxes, into a 2-stage ring;
//   warp 5   MMA issuer: S = Q K^T into one of two TMEM buffers (128 columns each), then
//            O += P V into a third TMEM region, one elected thread issuing tcgen05.mma;
//   warps 0-3 softmax: thread r owns query row r = TMEM lane r; loads its S row, masks the
//            edge, keeps a running maximum that is only moved when it grows by more than
//            2^8 (so O needs rescaling rarely; then the thread rescales its O row in TMEM),
//            writes P = 2^(S - m) as bf16 into shared memory (SW128 K-major, the MMA's A
//            operand), and finally normalises O and stores it.
// S of tile j+1 is computed while the softmax of tile j runs.  All waits are bounded.
#include "rk_internal.cuh"
#include "rk_sm100.cuh"

#include <algorithm>
#include <cudaTypedefs.h>

namespace rk {

namespace {

using namespace sm100;

constexpr int kTcThreads = 192;
constexpr int kRowsTc = 128;
constexpr int kKeysTc = 128;
constexpr int kStages = 2;
constexpr float kRescaleThreshold = 8.0f;   // log2 units

template <int D>
struct TcLayout {
  static constexpr int kHalf = kRowsTc * 128;          // bytes of one [128 rows][64] bf16 block
  static constexpr int kTile = kRowsTc * D * 2;        // Q, K or V tile
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTile;
  static constexpr int kV = kK + kStages * kTile;
  static constexpr int kP = kV + kStages * kTile;
  static constexpr int kBytes = kP + kRowsTc * kKeysTc * 2;
  static constexpr int kSmem = kBytes + 1024;          // slack for 1024-byte alignment
};

struct TcBarriers {
  uint64_t q_full;
  uint64_t kv_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t s_full[2];
  uint64_t s_empty[2];
  uint64_t p_full;
  uint64_t o_done;
  uint32_t tmem_slot;
  int abort;
};

__device__ __forceinline__ void fail(TcBarriers& b, int32_t* status) {
  report(status, RK_ERR_TIMEOUT);
  *reinterpret_cast<volatile int*>(&b.abort) = 1;
}

__device__ __forceinline__ bool aborted(TcBarriers& b) { return *reinterpret_cast<volatile int*>(&b.abort) != 0; }

template <int D, int P>
__global__ __launch_bounds__(kTcThreads, 1) void prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                                                                   const __grid_constant__ CUtensorMap tmK,
                                                                   const __grid_constant__ CUtensorMap tmV,
                                                                   AttnParams p, AttnWorkspace ws) {
  using LY = TcLayout<D>;
  constexpr int EPT = kKeysTc / P;       // pages per key tile
  constexpr int HALVES = D / 64;
  constexpr int KSTEPS = D / 16;         // MMA k-steps of Q.K^T
  constexpr uint32_t kIdescQK = idesc_bf16(kRowsTc, kKeysTc, 0);
  constexpr uint32_t kIdescPV = idesc_bf16(kRowsTc, D, 1);
  constexpr uint32_t kTmemCols = 512;
  constexpr uint32_t kColO = 256;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ TcBarriers bars;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sbase = smem_addr(smem);
  const uint32_t sQ = sbase + LY::kQ, sK = sbase + LY::kK, sV = sbase + LY::kV, sP = sbase + LY::kP;
  const uint32_t b_q = smem_addr(&bars.q_full), b_p = smem_addr(&bars.p_full), b_o = smem_addr(&bars.o_done);

  if (tid == 0) {
    mbar_init(b_q, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_addr(&bars.kv_full[s]), 1);
      mbar_init(smem_addr(&bars.kv_empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_addr(&bars.s_full[s]), 1);
      mbar_init(smem_addr(&bars.s_empty[s]), 128);
    }
    mbar_init(b_p, 128);
    mbar_init(b_o, 1);
    bars.abort = 0;
    mbar_fence_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_addr(&bars.tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_slot;

  const int G = p.G;
  const int n_items = ws.header->n_items;
  const int64_t oob_row = p.n_pool_pages * P;      // a row index past the pool: TMA fills zeros
  uint32_t g = 0;            // tiles processed by this CTA so far (all roles count alike)
  uint32_t q_uses = 0;       // items with at least one tile
  // last phase each role may still have in flight (for the bounded teardown)
  int last_kv_stage = -1;
  uint32_t last_kv_parity = 0;
  bool mma_pending = false;
  uint32_t mma_pending_parity = 0;

  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    const Item item = ws.items[it];
    const Unit un = ws.units[item.unit];
    const int seg = un.seg;
    const int h = seg % p.Hkv;
    const int n_kt = (item.v_end - item.v_begin + EPT - 1) / EPT;
    const int32_t* trow = p.page_table + int64_t(seg) * p.max_pages;
    const int32_t* lrow = p.page_logical ? p.page_logical + int64_t(seg) * p.max_pages : nullptr;

    if (warp == 4 && lane == 0 && n_kt > 0 && !aborted(bars)) {
      // ---------------------------------------------------------------- producer
      mbar_arrive_expect_tx(b_q, LY::kTile);
#pragma unroll
      for (int hf = 0; hf < HALVES; ++hf) tma_load_3d(sQ + hf * LY::kHalf, &tmQ, hf * 64, h * G, un.tok0, b_q);
      for (int j = 0; j < n_kt; ++j) {
        const uint32_t gg = g + j;
        const int st = gg % kStages;
        const uint32_t full = smem_addr(&bars.kv_full[st]), empty = smem_addr(&bars.kv_empty[st]);
        if (gg >= kStages && !mbar_wait(empty, ((gg / kStages) - 1) & 1)) { fail(bars, p.status); break; }
        mbar_arrive_expect_tx(full, 2 * LY::kTile);
        last_kv_stage = st;
        last_kv_parity = (gg / kStages) & 1;
        const int v0 = item.v_begin + j * EPT;
#pragma unroll
        for (int pg = 0; pg < EPT; ++pg) {
          const int v = v0 + pg;
          int64_t row = oob_row;
          if (v < item.v_end) {
            const int page = __ldg(trow + unit_entry(un, v));
            if (page >= 0 && page < p.n_pool_pages) row = int64_t(page) * P;
            else report(p.status, RK_ERR_DEVICE_BOUNDS);
          }
#pragma unroll
          for (int hf = 0; hf < HALVES; ++hf) {
            const uint32_t off = st * LY::kTile + hf * LY::kHalf + pg * P * 128;
            tma_load_2d(sK + off, &tmK, hf * 64, int(row), full);
            tma_load_2d(sV + off, &tmV, hf * 64, int(row), full);
          }
        }
      }
    } else if (warp == 5 && lane == 0 && n_kt > 0 && !aborted(bars)) {
      // ---------------------------------------------------------------- MMA issuer
      bool ok = mbar_wait(b_q, q_uses & 1);
      tc_fence_after();
      auto issue_pv = [&](int jj) -> bool {
        const uint32_t gg = g + jj;
        const int st = gg % kStages;
        if (!mbar_wait(b_p, gg & 1)) return false;
        tc_fence_after();
        const uint32_t vbase = sV + st * LY::kTile;
#pragma unroll
        for (int k = 0; k < kKeysTc / 16; ++k) {
          const uint64_t a = desc_sw128(sP + (k >> 2) * LY::kHalf + (k & 3) * 32, 16, 1024);
          const uint64_t b = desc_sw128(vbase + k * 2048, LY::kHalf, 1024);
          tc_mma_f16(tmem + kColO, a, b, kIdescPV, (jj > 0 || k > 0) ? 1u : 0u);
        }
        tc_commit(b_o);
        tc_commit(smem_addr(&bars.kv_empty[st]));
        mma_pending = true;
        mma_pending_parity = gg & 1;
        return true;
      };
      for (int j = 0; ok && j < n_kt; ++j) {
        const uint32_t gg = g + j;
        const int st = gg % kStages, sb = gg & 1;
        if (!mbar_wait(smem_addr(&bars.kv_full[st]), (gg / kStages) & 1)) { ok = false; break; }
        if (gg >= 2 && !mbar_wait(smem_addr(&bars.s_empty[sb]), ((gg >> 1) - 1) & 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t kbase = sK + st * LY::kTile;
#pragma unroll
        for (int k = 0; k < KSTEPS; ++k) {
          const uint64_t a = desc_sw128(sQ + (k >> 2) * LY::kHalf + (k & 3) * 32, 16, 1024);
          const uint64_t b = desc_sw128(kbase + (k >> 2) * LY::kHalf + (k & 3) * 32, 16, 1024);
          tc_mma_f16(tmem + sb * kKeysTc, a, b, kIdescQK, k > 0 ? 1u : 0u);
        }
        tc_commit(smem_addr(&bars.s_full[sb]));
        if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
      }
      if (ok) ok = issue_pv(n_kt - 1);
      if (!ok) fail(bars, p.status);
    } else if (warp < 4) {
      // ---------------------------------------------------------------- softmax + epilogue
      const int r = tid;                       // query row = TMEM lane
      const int rows_valid = un.ntok * G;
      const int pos = un.pos0 + r / G;
      const int L = __ldg(p.seq_len + un.b);
      const int cls = __ldg(p.head_class + seg);
      const bool local = cls == RK_CLASS_LOCAL;
      const int W = local ? __ldg(p.window + seg) : 0;
      const int S = (local && p.sink) ? __ldg(p.sink + seg) : 0;
      const uint32_t lane_base = uint32_t(warp * 32) << 16;
      float m_ref = -INFINITY, l_sum = 0.f;
      bool ok = true;
      for (int j = 0; j < n_kt; ++j) {
        const uint32_t gg = g + j;
        const int sb = gg & 1;
        // waits are made warp-uniform: tcgen05.ld/st below are warp-collective
        const bool got = !aborted(bars) && mbar_wait(smem_addr(&bars.s_full[sb]), (gg >> 1) & 1);
        if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
        tc_fence_after();
        float x[kKeysTc];
#pragma unroll
        for (int c = 0; c < kKeysTc / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + sb * kKeysTc + c * 32, v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) x[c * 32 + i] = __uint_as_float(v[i]) * p.scale_log2;
        }
        tc_fence_before();
        mbar_arrive(smem_addr(&bars.s_empty[sb]));

        // visibility of this tile's keys for this row
        const int v0 = item.v_begin + j * EPT;
        int lp[EPT];
        bool all_valid = true;
#pragma unroll
        for (int pg = 0; pg < EPT; ++pg) {
          const int v = v0 + pg;
          if (v < item.v_end) {
            const int e = unit_entry(un, v);
            lp[pg] = lrow ? __ldg(lrow + e) : e;
          } else {
            lp[pg] = -1;
            all_valid = false;
          }
        }
        const int j_min = lp[0] * P;
        int lp_last = lp[0];
#pragma unroll
        for (int pg = 0; pg < EPT; ++pg) lp_last = lp[pg] >= 0 ? lp[pg] : lp_last;
        const int j_max = lp_last * P + P - 1;
        const bool full = all_valid && j_max <= pos && j_max < L && (!local || j_min > pos - W || j_max < S);
        if (!full) {
#pragma unroll
          for (int c = 0; c < kKeysTc; ++c) {
            const int lpc = lp[c / P];
            const int jj = lpc * P + (c % P);
            const bool vis = lpc >= 0 && jj < L && jj <= pos && (!local || jj > pos - W || jj < S);
            if (!vis) x[c] = -INFINITY;
          }
        }
        float mx = x[0];
#pragma unroll
        for (int c = 1; c < kKeysTc; ++c) mx = fmaxf(mx, x[c]);
        const float m_new = fmaxf(m_ref, mx);
        const bool rescale = m_new > m_ref + kRescaleThreshold;   // false while both are -inf

        if (j > 0) {
          const bool got_o = mbar_wait(b_o, (gg - 1) & 1);
          if (!__all_sync(0xffffffffu, got_o)) { ok = false; break; }
          tc_fence_after();
          if (__any_sync(0xffffffffu, rescale)) {
            const float alpha = rescale ? fast_exp2(m_ref - m_new) : 1.f;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t v[32];
              tmem_ld32(tmem + lane_base + kColO + c * 32, v);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
              tmem_st32(tmem + lane_base + kColO + c * 32, v);
            }
            tmem_wait_st();
          }
        }
        if (rescale) {
          l_sum = (m_ref == -INFINITY) ? 0.f : l_sum * fast_exp2(m_ref - m_new);
          m_ref = m_new;
        }
        const float ref = m_ref == -INFINITY ? 0.f : m_ref;
        // P row -> shared memory, SW128 K-major: 16-byte chunk c of row r at
        // half (c / 8), row offset r * 128, chunk slot (c % 8) ^ (r % 8)
        float psum = 0.f;
#pragma unroll
        for (int c = 0; c < kKeysTc / 8; ++c) {
          float e[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            e[i] = fast_exp2(x[c * 8 + i] - ref);
            psum += e[i];
          }
          uint4 w;
          w.x = pack_bf16(e[0], e[1]);
          w.y = pack_bf16(e[2], e[3]);
          w.z = pack_bf16(e[4], e[5]);
          w.w = pack_bf16(e[6], e[7]);
          const uint32_t addr = sP + (c >> 3) * LY::kHalf + r * 128 + (((c & 7) ^ (r & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" :: "r"(addr), "r"(w.x), "r"(w.y), "r"(w.z),
                       "r"(w.w) : "memory");
        }
        l_sum += psum;
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(b_p);
      }
      // epilogue: O / l -> output (or split partial)
      if (ok && n_kt > 0) {
        const bool got_o = mbar_wait(b_o, (g + n_kt - 1) & 1);
        if (!__all_sync(0xffffffffu, got_o)) ok = false;
        tc_fence_after();
      }
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) fail(bars, p.status);
      const bool split = un.n_splits > 1;
      const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
      const float lse = l_sum > 0.f ? (m_ref + fast_log2(l_sum)) * 0.69314718055994531f : -INFINITY;
      const bool row_ok = r < rows_valid;
      const int t = un.tok0 + r / G, hq = h * G + r % G;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        if (ok && n_kt > 0) {
          tmem_ld32(tmem + lane_base + kColO + c * 32, v);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0u;
        }
        if (!row_ok) continue;
        if (!split) {
          __nv_bfloat16* orow = p.out + (int64_t(t) * p.Hq + hq) * D + c * 32;
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint4 w;
            w.x = pack_bf16(__uint_as_float(v[i]) * inv, __uint_as_float(v[i + 1]) * inv);
            w.y = pack_bf16(__uint_as_float(v[i + 2]) * inv, __uint_as_float(v[i + 3]) * inv);
            w.z = pack_bf16(__uint_as_float(v[i + 4]) * inv, __uint_as_float(v[i + 5]) * inv);
            w.w = pack_bf16(__uint_as_float(v[i + 6]) * inv, __uint_as_float(v[i + 7]) * inv);
            *reinterpret_cast<uint4*>(orow + i) = w;
          }
        } else {
          float* prow = ws.part_o + (int64_t(it) * ws.rows + r) * D + c * 32;
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(prow + i) =
                make_float4(__uint_as_float(v[i]) * inv, __uint_as_float(v[i + 1]) * inv,
                            __uint_as_float(v[i + 2]) * inv, __uint_as_float(v[i + 3]) * inv);
        }
      }
      if (row_ok) {
        if (!split) {
          if (p.lse) p.lse[int64_t(t) * p.Hq + hq] = lse;
        } else {
          ws.part_lse[int64_t(it) * ws.rows + r] = lse;
        }
      }
      tc_fence_before();
    }
    if (n_kt > 0) {
      g += n_kt;
      ++q_uses;
    }
    __syncthreads();
    if (aborted(bars)) break;
  }

  // teardown: let this CTA's own copies and MMAs land (bounded), then free TMEM
  if (warp == 4 && lane == 0 && last_kv_stage >= 0 && aborted(bars))
    mbar_wait(smem_addr(&bars.kv_full[last_kv_stage]), last_kv_parity);
  if (warp == 5 && lane == 0 && mma_pending && aborted(bars)) mbar_wait(b_o, mma_pending_parity);
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ host side
template <int D, int P>
cudaError_t launch_tc(const AttnParams& p, const AttnWorkspace& ws, int grid, cudaStream_t stream) {
  using LY = TcLayout<D>;
  CUtensorMap mq, mk, mv;
  const cuuint64_t qdims[3] = {cuuint64_t(D), cuuint64_t(p.Hq), cuuint64_t(p.total_q)};
  const cuuint64_t qstr[2] = {cuuint64_t(D) * 2, cuuint64_t(p.Hq) * D * 2};
  const cuuint32_t qbox[3] = {64, cuuint32_t(p.G), cuuint32_t(kRowsTc / p.G)};
  const cuuint64_t kdims[2] = {cuuint64_t(D), cuuint64_t(p.n_pool_pages) * P};
  const cuuint64_t kstr[1] = {cuuint64_t(D) * 2};
  const cuuint32_t kbox[2] = {64, cuuint32_t(P)};
  if (!encode_tmap_bf16(&mq, p.q, 3, qdims, qstr, qbox) || !encode_tmap_bf16(&mk, p.k_pool, 2, kdims, kstr, kbox) ||
      !encode_tmap_bf16(&mv, p.v_pool, 2, kdims, kstr, kbox))
    return cudaErrorInvalidValue;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<D, P>, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::kSmem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  prefill_tc_kernel<D, P><<<grid, kTcThreads, LY::kSmem, stream>>>(mq, mk, mv, p, ws);
  return cudaGetLastError();
}

}  // namespace

// ------------------------------------------------------------------ tensor maps
static PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* ptr = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

bool encode_tmap_bf16(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
            const cuuint32_t* box) {
  auto fn = get_encoder();
  if (!fn) return false;
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int prefill_tc_rows() { return kRowsTc; }
int prefill_tc_keys() { return kKeysTc; }

cudaError_t launch_prefill_tc(const AttnParams& p, const AttnWorkspace& ws, int grid, cudaStream_t stream) {
  if (p.d == 128) return p.P == 16 ? launch_tc<128, 16>(p, ws, grid, stream) : launch_tc<128, 32>(p, ws, grid, stream);
  return p.P == 16 ? launch_tc<64, 16>(p, ws, grid, stream) : launch_tc<64, 32>(p, ws, grid, stream);
}

}  // namespace rk
