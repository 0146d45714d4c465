// Token-level sparse FFN ("小红书 RedKnot", section 3, third component: elastic / sparse FFN
// chooses, token by token, which tokens go through the feed-forward network according to
// their attention importance, and skips the low-contribution ones -- at 2K-8K tokens the FFN
// is most of the prefill time).
//
//   1. select_kernel       the `keep` tokens with the highest importance (ties: lower token
//                          index first), listed in ascending order -- one CTA, radix select
//                          on the order-preserving integer image of the fp32 scores;
//   2. gather_kernel       their rows of x into a contiguous [keep][d_model] buffer;
//   3. ffn_gemm_kernel<0>  act = silu(x_sel W_gate^T) * (x_sel W_up^T)      [keep][d_ff]
//   4. ffn_gemm_kernel<1>  out[kept[m]] = act[m] W_down^T                    scattered rows
// Rows of skipped tokens are zero (their FFN is skipped; a residual add leaves them as they
// were).
//
// The GEMMs run on the 5th-generation tensor cores: C[M][N] = A[M][K] . B[N][K]^T with A and B
// K-major bf16, fp32 accumulation in TMEM.  Persistent CTAs (one per SM) walk 128 x 256 output
// tiles, N-major with M fastest so that consecutive tiles share their weight tile through L2.
// Per CTA, 6 warps:
//   warp 0    TMA producer: A tile [128][64] and B tile [256][64] per K step into a 4-stage
//             ring (128-byte swizzle); for the SwiGLU GEMM the B tile is 128 rows of W_gate
//             followed by the same 128 rows of W_up;
//   warp 1    MMA issuer (one thread): 4 x tcgen05.mma (M 128, N 256, K 16) per K step into one
//             of two TMEM accumulators of 256 columns, so the epilogue of one tile overlaps the
//             main loop of the next;
//   warps 2-5 epilogue: thread = TMEM lane = output row; silu(g) * u, or the scatter to kept[m].
// Every wait is bounded; a timeout sets RK_ERR_TIMEOUT and all roles leave.
#include "rk_internal.cuh"
#include "rk_sm100.cuh"

#include <algorithm>
#include <cmath>

namespace rk {

namespace {

using namespace sm100;

// ------------------------------------------------------------------ selection
constexpr int kSelThreads = 1024;

__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  if (f != f) return 0u;                         // NaN: below every number
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__global__ __launch_bounds__(kSelThreads) void select_kernel(const float* __restrict__ importance, int T, int keep,
                                                             int32_t* __restrict__ kept) {
  __shared__ int hist[256];
  __shared__ int s_warp[32];
  __shared__ uint32_t s_prefix;
  __shared__ int s_need;
  grid_dependency_wait();
  grid_launch_dependents();
  const int tid = threadIdx.x;
  if (keep <= 0) return;
  // k-th largest key, 8 bits at a time from the top: prefix of the answer and how many keys
  // equal to it are still to be taken
  if (tid == 0) { s_prefix = 0u; s_need = keep; }
  __syncthreads();
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += kSelThreads) hist[i] = 0;
    __syncthreads();
    const uint32_t prefix = s_prefix;
    const uint32_t hi_mask = shift == 24 ? 0u : (0xFFFFFFFFu << (shift + 8));
    for (int t = tid; t < T; t += kSelThreads) {
      const uint32_t k = order_key(importance[t]);
      if ((k & hi_mask) == (prefix & hi_mask)) atomicAdd(&hist[(k >> shift) & 255u], 1);
    }
    __syncthreads();
    if (tid == 0) {
      int need = s_need, digit = 255;
      for (; digit > 0; --digit) {                // from the largest digit down
        if (hist[digit] >= need) break;
        need -= hist[digit];
      }
      s_prefix = prefix | (uint32_t(digit) << shift);
      s_need = need;
    }
    __syncthreads();
  }
  const uint32_t kth = s_prefix;                 // the key of the k-th largest score
  const int ties = s_need;                       // keys equal to it that are kept (lowest indices)
  // kept: key > kth, or key == kth among the first `ties` such tokens; positions in index
  // order by two block scans over contiguous chunks of tokens
  const int per = (T + kSelThreads - 1) / kSelThreads;
  const int t0 = tid * per, t1 = min(T, t0 + per);
  int n_eq = 0;
  for (int t = t0; t < t1; ++t) n_eq += order_key(importance[t]) == kth;
  int tot;
  const int eq_before = block_exclusive_scan(n_eq, &tot, s_warp);
  int n_keep = 0, eq = eq_before;
  for (int t = t0; t < t1; ++t) {
    const uint32_t k = order_key(importance[t]);
    n_keep += k > kth || (k == kth && eq++ < ties);
  }
  int pos = block_exclusive_scan(n_keep, &tot, s_warp);
  eq = eq_before;
  for (int t = t0; t < t1; ++t) {
    const uint32_t k = order_key(importance[t]);
    if (k > kth || (k == kth && eq++ < ties)) kept[pos++] = t;
  }
}

// x_sel[i] = x[kept[i]], 16 bytes per thread
__global__ void gather_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ kept, int keep, int row16,
                              uint4* __restrict__ x_sel) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int64_t n = int64_t(keep) * row16;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n; i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t r = i / row16, c = i - r * row16;
    x_sel[i] = x[int64_t(__ldg(kept + r)) * row16 + c];
  }
}

// ------------------------------------------------------------------ GEMM
constexpr int kGThreads = 192;
constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr int kDownN = 256;                      // output columns of a down-projection tile
constexpr int kStages = 4;
constexpr int kATile = kBM * kBK * 2;            // 16 KB
constexpr int kBTile = kBN * kBK * 2;            // 32 KB
constexpr int kStageBytes = kATile + kBTile;
constexpr int kGSmem = kStages * kStageBytes + 1024;
constexpr uint64_t kGWaitNs = 1000000000ull;

struct GemmShared {
  uint64_t full[kStages], empty[kStages];
  uint64_t acc_full[2], acc_empty[2];
  uint32_t tmem_slot;
  int abort;
  int last;   // this CTA holds the last piece of a split tile
};

__device__ __forceinline__ bool g_aborted(GemmShared& sh) { return *reinterpret_cast<volatile int*>(&sh.abort) != 0; }
__device__ __forceinline__ bool g_wait(GemmShared& sh, uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (g_aborted(sh)) return false;
    if (globaltimer() - t0 > kGWaitNs) return false;
  }
}
__device__ __forceinline__ void g_fail(GemmShared& sh, int32_t* status) {
  report(status, RK_ERR_TIMEOUT);
  *reinterpret_cast<volatile int*>(&sh.abort) = 1;
}

struct GemmParams {
  int M, N, K;              // C[M][N] = A[M][K] . B[N][K]^T (MODE 0: N counts act columns, B holds 2N rows)
  __nv_bfloat16* c;         // MODE 0: act [M][N]; MODE 1: out rows, [*][N]
  const int32_t* rows;      // MODE 1: output row of each M row (the kept tokens)
  int ldc;
  int32_t* status;
  // MODE 1, last wave split along K: tiles [n_full, tiles) are cut into `split` pieces each;
  // every piece adds its fp32 tile into part[tail tile] (laid out [kDownN / 4][kBM] float4,
  // zero at the start), and the piece that takes the last ticket of its tile (tickets[tail
  // tile], zero at the start) converts the sum and scatters the rows
  int n_full, split;
  float* part;
  int32_t* tickets;
};

__device__ __forceinline__ float silu(float g) {
  // g * sigmoid(g), sigmoid via the ex2 instruction and a reciprocal
  return g * __frcp_rn(1.f + fast_exp2(-g * 1.4426950408889634f));
}

template <int MODE>
__global__ __launch_bounds__(kGThreads, 1) void ffn_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                                                                const __grid_constant__ CUtensorMap tmB0,
                                                                const __grid_constant__ CUtensorMap tmB1,
                                                                GemmParams g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ GemmShared sh;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sbase = smem_addr(smem);
  // MODE 0 covers 128 act columns per tile (256 accumulator columns: gate | up)
  constexpr int kMmaN = MODE == 0 ? kBN : kDownN;
  constexpr uint32_t kIdesc = idesc_bf16(kBM, kMmaN, 0, 0);
  constexpr int kTileN = MODE == 0 ? kBN / 2 : kDownN;
  constexpr int kLoadBytes = kATile + kMmaN * kBK * 2;
  const int m_tiles = (g.M + kBM - 1) / kBM, n_tiles = g.N / kTileN, k_steps = g.K / kBK;
  const int n_work = m_tiles * n_tiles;
  const bool split = MODE == 1 && g.split > 1;
  const int n_units = split ? g.n_full + (n_work - g.n_full) * g.split : n_work;
  // unit w: output tile `tile` (its row and column blocks m, n), K steps [kb, ke), and its
  // piece index (-1: the whole tile)
  auto unit = [&](int w, int& tile, int& m, int& n, int& kb, int& ke, int& piece) {
    tile = w;
    piece = -1;
    kb = 0;
    ke = k_steps;
    if (split && w >= g.n_full) {
      const int q = (w - g.n_full) / g.split;
      piece = (w - g.n_full) - q * g.split;
      tile = g.n_full + q;
      kb = int((long long)piece * k_steps / g.split);
      ke = int((long long)(piece + 1) * k_steps / g.split);
    }
    n = tile / m_tiles;
    m = tile - n * m_tiles;
  };

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_addr(&sh.full[s]), 1);
      mbar_init(smem_addr(&sh.empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_addr(&sh.acc_full[a]), 1);
      mbar_init(smem_addr(&sh.acc_empty[a]), 128);
    }
    sh.abort = 0;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" :: "l"(&tmA) : "memory");
    asm volatile("prefetch.tensormap [%0];" :: "l"(&tmB0) : "memory");
    if (MODE == 0) asm volatile("prefetch.tensormap [%0];" :: "l"(&tmB1) : "memory");
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(&sh.tmem_slot), 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_slot;
  grid_dependency_wait();
  grid_launch_dependents();

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      int last = -1;
      uint32_t last_par = 0;
      for (int w = blockIdx.x; ok && w < n_units; w += gridDim.x) {
        int tile, m, n, kb, ke, piece;
        unit(w, tile, m, n, kb, ke, piece);
        for (int ks = kb; ks < ke; ++ks, ++it) {
          const int s = it % kStages;
          if (it >= kStages && !g_wait(sh, smem_addr(&sh.empty[s]), ((it / kStages) - 1) & 1)) { ok = false; break; }
          const uint32_t bar = smem_addr(&sh.full[s]);
          mbar_arrive_expect_tx(bar, kLoadBytes);
          const uint32_t sa = sbase + s * kStageBytes, sb = sa + kATile;
          tma_load_2d(sa, &tmA, ks * kBK, m * kBM, bar);
          if (MODE == 0) {
            tma_load_2d(sb, &tmB0, ks * kBK, n * kTileN, bar);                     // gate rows
            tma_load_2d(sb + kBTile / 2, &tmB1, ks * kBK, n * kTileN, bar);        // up rows
          } else {
            tma_load_2d(sb, &tmB0, ks * kBK, n * kTileN, bar);
          }
          last = s;
          last_par = (it / kStages) & 1;
        }
      }
      if (!ok) g_fail(sh, g.status);
      if (g_aborted(sh) && last >= 0) mbar_wait(smem_addr(&sh.full[last]), last_par);   // copies land before exit
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t it = 0, tcount = 0;
      bool ok = true;
      for (int w = blockIdx.x; ok && w < n_units; w += gridDim.x, ++tcount) {
        const int a = tcount & 1;
        int tile, m, n, kb, ke, piece;
        unit(w, tile, m, n, kb, ke, piece);
        if (tcount >= 2 && !g_wait(sh, smem_addr(&sh.acc_empty[a]), ((tcount >> 1) - 1) & 1)) { ok = false; break; }
        tc_fence_after();
        for (int ks = kb; ks < ke; ++ks, ++it) {
          const int s = it % kStages;
          if (!g_wait(sh, smem_addr(&sh.full[s]), (it / kStages) & 1)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = sbase + s * kStageBytes, sb = sa + kATile;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t da = desc_sw128(sa + kk * 32, 16, 1024);
            const uint64_t db = desc_sw128(sb + kk * 32, 16, 1024);
            tc_mma_f16(tmem + a * kBN, da, db, kIdesc, (ks > kb || kk > 0) ? 1u : 0u);
          }
          tc_commit(smem_addr(&sh.empty[s]));
        }
        if (ok) tc_commit(smem_addr(&sh.acc_full[a]));
      }
      if (!ok) g_fail(sh, g.status);
    }
  } else {
    // ---------------------------------------------------------------- epilogue (warps 2-5)
    const int q = warp & 3;                      // TMEM lane quarter this warp may access
    const int r = q * 32 + lane;                 // row of the tile
    const uint32_t lane_base = uint32_t(q * 32) << 16;
    uint32_t tcount = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < n_units; w += gridDim.x, ++tcount) {
      int tile, m, n, kb, ke, piece;
      unit(w, tile, m, n, kb, ke, piece);
      const int a = tcount & 1;
      const bool got = g_wait(sh, smem_addr(&sh.acc_full[a]), (tcount >> 1) & 1);
      if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
      tc_fence_after();
      const int row = m * kBM + r;
      const bool live = row < g.M;
      if (MODE == 0) {
        __nv_bfloat16* dst = g.c + int64_t(row) * g.ldc + n * kTileN;
#pragma unroll 1
        for (int c = 0; c < kTileN; c += 32) {
          uint32_t gv[32], uv[32];
          tmem_ld32(tmem + lane_base + a * kBN + c, gv);
          tmem_ld32(tmem + lane_base + a * kBN + kTileN + c, uv);
          tmem_wait_ld();
          if (live) {
#pragma unroll
            for (int i = 0; i < 32; i += 8) {
              uint4 o;
              o.x = pack_bf16(silu(__uint_as_float(gv[i])) * __uint_as_float(uv[i]),
                              silu(__uint_as_float(gv[i + 1])) * __uint_as_float(uv[i + 1]));
              o.y = pack_bf16(silu(__uint_as_float(gv[i + 2])) * __uint_as_float(uv[i + 2]),
                              silu(__uint_as_float(gv[i + 3])) * __uint_as_float(uv[i + 3]));
              o.z = pack_bf16(silu(__uint_as_float(gv[i + 4])) * __uint_as_float(uv[i + 4]),
                              silu(__uint_as_float(gv[i + 5])) * __uint_as_float(uv[i + 5]));
              o.w = pack_bf16(silu(__uint_as_float(gv[i + 6])) * __uint_as_float(uv[i + 6]),
                              silu(__uint_as_float(gv[i + 7])) * __uint_as_float(uv[i + 7]));
              *reinterpret_cast<uint4*>(dst + c + i) = o;
            }
          }
        }
      } else if (piece >= 0) {
        // a piece of a split tile: added into the tile's fp32 sum, column blocks of 4 with the
        // rows adjacent, so that a warp's 32 rows touch 512 contiguous bytes
        const int q = tile - g.n_full;
        float4* acc = reinterpret_cast<float4*>(g.part) + int64_t(q) * (kDownN / 4) * kBM + r;
#pragma unroll 1
        for (int c = 0; c < kTileN; c += 32) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + a * kBN + c, v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            atomicAdd(acc + ((c + i) / 4) * kBM, make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]),
                                                               __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3])));
        }
        tc_fence_before();
        mbar_arrive(smem_addr(&sh.acc_empty[a]));   // the accumulator is free; the sum is in memory
        __threadfence();                              // the additions are visible before the ticket
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (r == 0) sh.last = atomicAdd(g.tickets + q, 1) == g.split - 1;
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (sh.last) {   // every piece is added: convert the sum and scatter the rows
          __threadfence();
          if (live) {
            const int orow = __ldg(g.rows + row);
            __nv_bfloat16* dst = g.c + int64_t(orow) * g.ldc + n * kTileN;
#pragma unroll 1
            for (int c4 = 0; c4 < kTileN / 4; c4 += 16) {   // 16 loads in flight
              float4 x[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) x[i] = __ldcg(acc + (c4 + i) * kBM);
#pragma unroll
              for (int i = 0; i < 16; i += 2) {
                uint4 o;
                o.x = pack_bf16(x[i].x, x[i].y);
                o.y = pack_bf16(x[i].z, x[i].w);
                o.z = pack_bf16(x[i + 1].x, x[i + 1].y);
                o.w = pack_bf16(x[i + 1].z, x[i + 1].w);
                *reinterpret_cast<uint4*>(dst + (c4 + i) * 4) = o;
              }
            }
          }
          if (r == 0) g.tickets[q] = 0;   // for the next call
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");   // sh.last is rewritten by the next piece
        continue;
      } else {
        const int orow = live ? __ldg(g.rows + row) : 0;
        __nv_bfloat16* dst = g.c + int64_t(orow) * g.ldc + n * kTileN;
#pragma unroll 1
        for (int c = 0; c < kTileN; c += 32) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + a * kBN + c, v);
          tmem_wait_ld();
          if (live) {
#pragma unroll
            for (int i = 0; i < 32; i += 8) {
              uint4 o;
              o.x = pack_bf16(__uint_as_float(v[i]), __uint_as_float(v[i + 1]));
              o.y = pack_bf16(__uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
              o.z = pack_bf16(__uint_as_float(v[i + 4]), __uint_as_float(v[i + 5]));
              o.w = pack_bf16(__uint_as_float(v[i + 6]), __uint_as_float(v[i + 7]));
              *reinterpret_cast<uint4*>(dst + c + i) = o;
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(smem_addr(&sh.acc_empty[a]));
    }
    if (!ok && lane == 0) g_fail(sh, g.status);
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int MODE>
cudaError_t launch_gemm(const void* A, int lda_rows, const void* B0, const void* B1, int b_rows, GemmParams g,
                        cudaStream_t stream) {
  CUtensorMap ma, mb0, mb1;
  const cuuint64_t adims[2] = {cuuint64_t(g.K), cuuint64_t(lda_rows)};
  const cuuint64_t astr[1] = {cuuint64_t(g.K) * 2};
  const cuuint32_t abox[2] = {kBK, kBM};
  const cuuint64_t bdims[2] = {cuuint64_t(g.K), cuuint64_t(b_rows)};
  const cuuint32_t bbox[2] = {kBK, MODE == 0 ? uint32_t(kBN / 2) : uint32_t(kDownN)};
  if (!encode_tmap_bf16(&ma, A, 2, adims, astr, abox) || !encode_tmap_bf16(&mb0, B0, 2, bdims, astr, bbox) ||
      !encode_tmap_bf16(&mb1, MODE == 0 ? B1 : B0, 2, bdims, astr, bbox))
    return cudaErrorInvalidValue;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(ffn_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGSmem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  const int tiles = ((g.M + kBM - 1) / kBM) * (g.N / (MODE == 0 ? kBN / 2 : kDownN));
  const int sms = device_sm_count();
  int units = tiles;
  g.n_full = tiles;
  g.split = 0;
  if (MODE == 1 && g.part) {
    // the tiles of an incomplete last wave are cut along K so that it fills the SMs (each
    // piece at least 4 K steps): R tiles x S pieces <= the SMs, partials in part / tickets
    const int R = tiles % sms, S = R > 0 ? std::min(sms / R, (g.K / kBK) / 4) : 0;
    if (S >= 2) {
      g.n_full = tiles - R;
      g.split = S;
      units = g.n_full + R * S;
      const cudaError_t e = cudaMemsetAsync(g.part, 0, size_t(R) * kBM * kDownN * sizeof(float), stream);
      if (e != cudaSuccess) return e;
    }
  }
  const int grid = std::max(1, std::min(units, sms));
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(grid), dim3(kGThreads), kGSmem, stream, attr);
  return cudaLaunchKernelEx(&cfg, ffn_gemm_kernel<MODE>, ma, mb0, mb1, g);
}

}  // namespace

// Workspace: gathered rows [keep][d_model] and activation [keep][d_ff] (bf16), then the fp32
// partial tiles of a split last wave of the down projection (at most one per SM) and their
// tickets.
size_t sparse_ffn_ws_bytes(int keep, int d_model, int d_ff) {
  const size_t sms = size_t(device_sm_count());
  return align256(size_t(keep) * d_model * 2) + align256(size_t(keep) * d_ff * 2) +
         align256(sms * kBM * kDownN * sizeof(float)) + align256(sms * sizeof(int32_t));
}

cudaError_t launch_sparse_ffn(const rk_sparse_ffn_args& a, void* ws, cudaStream_t stream) {
  uint8_t* base = static_cast<uint8_t*>(ws);
  const size_t sms = size_t(device_sm_count());
  const size_t off_act = align256(size_t(a.keep) * a.d_model * 2);
  const size_t off_part = off_act + align256(size_t(a.keep) * a.d_ff * 2);
  const size_t off_tick = off_part + align256(sms * kBM * kDownN * sizeof(float));
  __nv_bfloat16* x_sel = reinterpret_cast<__nv_bfloat16*>(base);
  __nv_bfloat16* act = reinterpret_cast<__nv_bfloat16*>(base + off_act);
  float* part = reinterpret_cast<float*>(base + off_part);
  int32_t* tickets = reinterpret_cast<int32_t*>(base + off_tick);
  cudaError_t e = cudaMemsetAsync(a.out, 0, size_t(a.T) * a.d_model * 2, stream);   // skipped tokens: zero
  if (e != cudaSuccess || a.keep == 0) return e;
  e = cudaMemsetAsync(tickets, 0, sms * sizeof(int32_t), stream);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(1), dim3(kSelThreads), 0, stream, attr);
  e = cudaLaunchKernelEx(&cfg, select_kernel, a.importance, a.T, a.keep, a.kept);
  if (e != cudaSuccess) return e;
  const int row16 = a.d_model / 8;
  const int64_t n16 = int64_t(a.keep) * row16;
  cudaLaunchAttribute attr2[1];
  cudaLaunchConfig_t cfg2 = pdl_config(dim3(unsigned(std::min<int64_t>((n16 + 255) / 256, 8LL * device_sm_count()))),
                                       dim3(256), 0, stream, attr2);
  e = cudaLaunchKernelEx(&cfg2, gather_kernel, static_cast<const uint4*>(a.x), static_cast<const int32_t*>(a.kept),
                         a.keep, row16, reinterpret_cast<uint4*>(x_sel));
  if (e != cudaSuccess) return e;
  GemmParams g1{a.keep, a.d_ff, a.d_model, act, nullptr, a.d_ff, a.status, 0, 0, nullptr, nullptr};
  e = launch_gemm<0>(x_sel, a.keep, a.w_gate, a.w_up, a.d_ff, g1, stream);
  if (e != cudaSuccess) return e;
  GemmParams g2{a.keep, a.d_model, a.d_ff, static_cast<__nv_bfloat16*>(a.out), a.kept, a.d_model, a.status,
                0, 0, part, tickets};
  return launch_gemm<1>(act, a.keep, a.w_down, nullptr, a.d_model, g2, stream);
}

}  // namespace rk
