// SegPaged prefill on the 5th-generation tensor cores (tcgen05 + TMEM), sm_103a.
//
// What it computes is stated in include/rk_api.h: attention of each query over the keys
// its KV head lists in its own page table, with the causal / window edge applied as a
// predicate, never as an attn_mask tensor ("小红书 RedKnot" section 3, fourth component;
// "RedKnot" article, SegPagedAttention paragraph).
//
// Work items (rk_plan.cu, longest first) are taken from a counter; they are slices of the
// page list of one unit: 256 query rows of one
// KV head (GQA-packed: 256/G tokens x the G query heads), processed as two 128-row tiles
// A and B that share every K/V tile loaded, which halves the K/V traffic per FLOP.
// One CTA per SM, 12 warps (three warpgroups):
//   warp 8   producer: TMA loads the two Q tiles once per item, then for every 128-key
//            tile gathers its pages (8 of 16 tokens or 4 of 32) from the shared pools
//            through the page table, one box per page and 64 channels, into separate K
//            and V rings (a K stage is freed as soon as both S tiles are computed);
//   warp 9   MMA issuer (one thread): S_A = Q_A K^T and S_B = Q_B K^T into TMEM, then
//            O_A += P_A V and O_B += P_B V with P read straight from TMEM;
//   warps 10-11 merge the units cut into several items as they complete (the softmax warps
//            join them once the item queue is empty), so no separate combine kernel runs;
//   warps 0-3 / 4-7  softmax of tile A / B: thread r owns row r (TMEM lane r), loads its S
//            row once into registers, masks the edge, keeps a running maximum that moves
//            only when it grows by more than 2^8 (then the row of O is rescaled in TMEM),
//            writes P = 2^(S - m) as bf16 pairs over the first half of its S columns, and at
//            the end of the item normalises its O row and stores it (or a split partial).
// Registers: the block is launched with 168 per thread (12 warps x 168 = the 64K file); the
// producer / MMA warpgroup drops to kRegsLow and the two softmax warpgroups rise to kRegsHigh
// (2 x 128 x kRegsHigh + 128 x kRegsLow = 384 x 168), which holds a whole 128-score row.
// TMEM: S_A cols 0-127, S_B 128-255, O_A 256-383, O_B 384-511.  The two softmax groups
// work on S_A and S_B while the tensor core computes the other tile.  All waits are bounded.
#include "rk_internal.cuh"
#include "rk_sm100.cuh"

#include <algorithm>
#include <cudaTypedefs.h>

namespace rk {

namespace {

using namespace sm100;

constexpr int kTcThreads = 384;
constexpr int kRegsLaunch = 168;             // 65536 / 384, rounded down to a multiple of 8
constexpr int kRegsHigh = 208;               // softmax warpgroups
constexpr int kRegsLow = 88;                 // producer + MMA warpgroup
static_assert(2 * 128 * kRegsHigh + 128 * kRegsLow == kTcThreads * kRegsLaunch, "register split must match the launch");
constexpr int kTileRows = 128;
constexpr int kUnitRows = 256;
constexpr int kKeysTc = 128;
constexpr float kRescaleThreshold = 8.0f;   // log2 units
constexpr int kHalf = kTileRows * 128;      // bytes of one [128 rows][64] bf16 block
constexpr uint64_t kWaitNs = 1000000000ull;

template <int D>
struct TcLayout {
  static constexpr int kTile = (D / 64) * kHalf;      // Q, K or V tile
  static constexpr int kNK = D == 128 ? 2 : 4;        // K stages (freed once both S are computed)
  static constexpr int kNV = D == 128 ? 3 : 4;        // V stages (held until the second value product)
  static constexpr int kQ = 0;                        // Q_A, Q_B
  static constexpr int kK = kQ + 2 * kTile;
  static constexpr int kV = kK + kNK * kTile;
  static constexpr int kBytes = kV + kNV * kTile;
  static constexpr int kSmem = kBytes + 1024;         // slack for 1024-byte alignment
};

struct TcBarriers {
  uint64_t q_full, q_empty;
  uint64_t k_full[4], k_empty[4];
  uint64_t v_full[4], v_empty[4];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_done[2];
  uint64_t iq_full[2], iq_empty[2];   // item ring: producer -> MMA issuer and softmax warps
  int ring[2];
  int job[2][2];                      // merge jobs of the two workers (softmax warps, warps 10-11)
  uint32_t tmem_slot;
  int abort;
};

__device__ __forceinline__ bool aborted(TcBarriers& b) { return *reinterpret_cast<volatile int*>(&b.abort) != 0; }
__device__ __forceinline__ void fail(TcBarriers& b, int32_t* status) {
  report(status, RK_ERR_TIMEOUT);
  *reinterpret_cast<volatile int*>(&b.abort) = 1;
}
// Bounded wait that also gives up as soon as another role has aborted.
__device__ __forceinline__ bool wait_or_abort(TcBarriers& b, uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (aborted(b)) return false;
    if (globaltimer() - t0 > kWaitNs) return false;
  }
}

// Wait (acquire) until a unit's completion counter reaches `target`.  Gives up after 1 s in
// which neither that counter nor the item counter moved, or when another role aborted.
__device__ __forceinline__ bool wait_count(TcBarriers& b, const int32_t* c, int target, const int32_t* items) {
  int v;
  asm volatile("ld.acquire.gpu.s32 %0, [%1];" : "=r"(v) : "l"(c) : "memory");
  if (v >= target) return true;
  int last = v, last_items = -1;
  uint64_t t0 = globaltimer();
  while (true) {
    __nanosleep(128);
    asm volatile("ld.acquire.gpu.s32 %0, [%1];" : "=r"(v) : "l"(c) : "memory");
    if (v >= target) return true;
    const int it = *reinterpret_cast<const volatile int32_t*>(items);
    const uint64_t now = globaltimer();
    if (v != last || it != last_items) {
      last = v;
      last_items = it;
      t0 = now;
    } else if (now - t0 > kWaitNs || aborted(b)) {
      return false;
    }
  }
}

// Merge of the units cut into several items.  Two workers in each CTA take jobs -- one split
// unit and kJobRows of its rows -- from a common counter, in the order the planner lists the
// split units, which is the order their items are handed out, so units complete one after
// another and most merges run while later items are computed:
//  - warps 10-11 (BACKGROUND), from the start, but only while items remain and only a job
//    whose unit is already complete (they look at the next job and claim it with a
//    compare-and-swap), so that they never hold a merge the tail waits for;
//  - the eight softmax warps once their items are done: they claim the next job outright and
//    wait until its unit is complete (each item of it is held by a running CTA whose softmax
//    warps take no job before their items are done).
// A unit is complete when the 8 softmax warps of every item of it have stored their rows of
// the partial.  The merge is the log-sum-exp rule: lse = log sum_s e^(lse_s),
// o = sum_s e^(lse_s - lse) o_s.  Warp w of the worker takes rows w, w + nwarps, ... of the
// job; lane l channels [l C, l C + C), with 8 items' partials of the row in flight.
template <int D, bool BACKGROUND>
__device__ __forceinline__ bool merge_split_units(const AttnParams& p, const AttnWorkspace& ws, TcBarriers& b,
                                                  int* job_slot, uint32_t bar, int nthreads, int wtid, int n_items) {
  constexpr int kJobRows = 8, C = D / 32, SPL = 8;
  const int wl = wtid >> 5, lane = wtid & 31, nwarps = nthreads >> 5;
  const int rb = ws.rows / kJobRows;
  const int n_jobs = ws.header->n_split * rb;
  const int G = p.G;
  volatile int32_t* vcounter = &ws.header->merge_counter;
  // diagnostic: wait for one stored piece more than there are, so that the bounded wait runs out
  const int extra = (p.flags & RK_ATTN_DIAG_EXPIRE_WAIT) ? 1 : 0;
  for (int k = 0;; ++k) {
    if (wtid == 0) {
      int job;
      if constexpr (BACKGROUND) {
        // the next job, if its unit is complete and items remain; else -1 (stop)
        job = -1;
        uint64_t t0 = globaltimer();
        int last_items = -1;
        while (true) {
          const int items = *reinterpret_cast<volatile int32_t*>(&ws.header->counter);
          if (items + int(gridDim.x) >= n_items || aborted(b)) break;
          const int j = *vcounter;
          if (j >= n_jobs) break;
          const int u = ws.split_list[j / rb];
          int done;
          asm volatile("ld.acquire.gpu.s32 %0, [%1];" : "=r"(done) : "l"(ws.unit_done + u) : "memory");
          if (done >= 8 * ws.units[u].n_splits + extra) {
            if (atomicCAS(&ws.header->merge_counter, j, j + 1) == j) { job = j; break; }
            continue;
          }
          const uint64_t now = globaltimer();
          if (items != last_items) { last_items = items; t0 = now; }
          else if (now - t0 > kWaitNs) break;   // no item taken for 1 s: leave it to the tail
          __nanosleep(256);
        }
      } else {
        job = atomicAdd(&ws.header->merge_counter, 1);
      }
      job_slot[k & 1] = job;
    }
    named_bar_sync(bar, nthreads);
    const int job = job_slot[k & 1];
    if (job < 0 || job >= n_jobs) return true;
    const int u = ws.split_list[job / rb];
    const Unit un = ws.units[u];
    const bool got =
        (BACKGROUND || wtid != 0) ? true : wait_count(b, ws.unit_done + u, 8 * un.n_splits + extra, &ws.header->counter);
    if (!named_bar_and(bar, nthreads, got)) return false;
    const int ns = un.n_splits;
    for (int r = (job % rb) * kJobRows + wl; r < (job % rb + 1) * kJobRows; r += nwarps) {
      float M = -INFINITY, den = 0.f, acc[C];
#pragma unroll
      for (int c = 0; c < C; ++c) acc[c] = 0.f;
      for (int s0 = 0; s0 < ns; s0 += SPL) {
        float lv[SPL], ov[SPL][C];
#pragma unroll
        for (int q = 0; q < SPL; ++q) {
          lv[q] = -INFINITY;
#pragma unroll
          for (int c = 0; c < C; ++c) ov[q][c] = 0.f;
          if (s0 + q < ns) {
            const int64_t row = int64_t(unit_item(un, s0 + q)) * ws.rows + r;
            lv[q] = __ldcg(ws.part_lse + row);
            const float* po = ws.part_o + row * D + lane * C;
            if constexpr (C == 4) {
              const float4 v = __ldcg(reinterpret_cast<const float4*>(po));
              ov[q][0] = v.x; ov[q][1] = v.y; ov[q][2] = v.z; ov[q][3] = v.w;
            } else {
              const float2 v = __ldcg(reinterpret_cast<const float2*>(po));
              ov[q][0] = v.x; ov[q][1] = v.y;
            }
          }
        }
        float mc = M;
#pragma unroll
        for (int q = 0; q < SPL; ++q) mc = fmaxf(mc, lv[q]);
        if (mc == -INFINITY) continue;
        const float f = M == -INFINITY ? 0.f : expf(M - mc);
        den *= f;
#pragma unroll
        for (int c = 0; c < C; ++c) acc[c] *= f;
        M = mc;
#pragma unroll
        for (int q = 0; q < SPL; ++q) {
          const float w = lv[q] == -INFINITY ? 0.f : expf(lv[q] - mc);
          den += w;
#pragma unroll
          for (int c = 0; c < C; ++c) acc[c] = fmaf(w, ov[q][c], acc[c]);
        }
      }
      if (r >= un.ntok * G) continue;
      const int t = un.tok0 + r / G;
      const int hq = (un.seg % p.Hkv) * G + (r % G);
      const float inv = den > 0.f ? 1.f / den : 0.f;
      __nv_bfloat16* o = p.out + (int64_t(t) * p.Hq + hq) * D + lane * C;
      if constexpr (C == 4) {
        uint2 w;
        w.x = pack_bf16(acc[0] * inv, acc[1] * inv);
        w.y = pack_bf16(acc[2] * inv, acc[3] * inv);
        *reinterpret_cast<uint2*>(o) = w;
      } else {
        *reinterpret_cast<uint32_t*>(o) = pack_bf16(acc[0] * inv, acc[1] * inv);
      }
      if (p.lse && lane == 0) p.lse[int64_t(t) * p.Hq + hq] = den > 0.f ? M + logf(den) : -INFINITY;
    }
  }
}

template <int D, int P>
__global__ __launch_bounds__(kTcThreads, 1) void prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                                                                   const __grid_constant__ CUtensorMap tmK,
                                                                   const __grid_constant__ CUtensorMap tmV,
                                                                   AttnParams p, AttnWorkspace ws) {
  using LY = TcLayout<D>;
  constexpr int EPT = kKeysTc / P;       // pages per key tile
  constexpr int HALVES = D / 64;
  constexpr int NK = LY::kNK, NV = LY::kNV;
  constexpr uint32_t kIdescQK = idesc_bf16(kTileRows, kKeysTc, 0);
  constexpr uint32_t kIdescPV = idesc_bf16(kTileRows, D, 1);
  constexpr uint32_t kTmemCols = 512;
  constexpr uint32_t kColO = 256;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ TcBarriers bars;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sbase = smem_addr(smem);
  const uint32_t sQ = sbase + LY::kQ, sK = sbase + LY::kK, sV = sbase + LY::kV;

  if (tid == 0) {
    mbar_init(smem_addr(&bars.q_full), 1);
    mbar_init(smem_addr(&bars.q_empty), 1);
    for (int s = 0; s < NK; ++s) {
      mbar_init(smem_addr(&bars.k_full[s]), 1);
      mbar_init(smem_addr(&bars.k_empty[s]), 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(smem_addr(&bars.v_full[s]), 1);
      mbar_init(smem_addr(&bars.v_empty[s]), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(smem_addr(&bars.s_full[x]), 1);
      mbar_init(smem_addr(&bars.p_full[x]), 128);
      mbar_init(smem_addr(&bars.o_done[x]), 1);
      mbar_init(smem_addr(&bars.iq_full[x]), 1);
      mbar_init(smem_addr(&bars.iq_empty[x]), 257);
    }
    bars.abort = 0;
    mbar_fence_init();
  }
  if (warp == 8 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" :: "l"(&tmQ) : "memory");
    asm volatile("prefetch.tensormap [%0];" :: "l"(&tmK) : "memory");
    asm volatile("prefetch.tensormap [%0];" :: "l"(&tmV) : "memory");
  }
  if (warp == 9) {
    tmem_alloc(smem_addr(&bars.tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_slot;
  grid_dependency_wait();      // the plan (and everything before it in the stream) is complete
  grid_launch_dependents();    // the next kernel may be scheduled as CTAs of this one finish

  const int G = p.G;
  const int n_items = ws.header->n_items;
  const int64_t oob_row = p.n_pool_pages * P;      // a row index past the pool: TMA fills zeros

  // each warpgroup changes its register budget inside its own branch, so that the compiler
  // allocates every role's code against that role's budget
  if (warp >= 8) {
    regs_decrease<kRegsLow>();
    if (warp == 8) {
      // ---------------------------------------------------------------- producer
      uint32_t gg = 0, qn = 0;
      int last_k = -1, last_v = -1;
      uint32_t last_k_par = 0, last_v_par = 0, last_q_par = 0;
      bool q_pending = false, ok = true;
      // items: blockIdx.x first, then from the counter (the next ticket is requested one item
      // ahead); each is handed to the other roles through the 2-entry ring
      int it = blockIdx.x, ticket = 0;
      for (int k = 0; ok; ++k) {
        if (k > 0) it = int(gridDim.x) + __shfl_sync(0xffffffffu, ticket, 0);   // requested one item ago
        const int slot = k & 1;
        bool gotr = true;
        if (lane == 0 && k >= 2) gotr = wait_or_abort(bars, smem_addr(&bars.iq_empty[slot]), ((k >> 1) - 1) & 1);
        if (!__shfl_sync(0xffffffffu, gotr, 0)) { ok = false; break; }
        const bool valid = it < n_items;
        if (lane == 0) {
          bars.ring[slot] = valid ? it : -1;
          mbar_arrive(smem_addr(&bars.iq_full[slot]));
          if (valid) ticket = atomicAdd(&ws.header->counter, 1);
        }
        if (!valid) break;
        const Item item = ws.items[it];
        const Unit un = ws.units[item.unit];
        const int n_kt = (item.v_end - item.v_begin + EPT - 1) / EPT;
        if (n_kt == 0) continue;
        const int h = un.seg % p.Hkv;
        const int32_t* trow = p.page_table + int64_t(un.seg) * p.max_pages;
        bool got = true;
        if (lane == 0) {   // both Q tiles; the buffer is free once the previous item's S are computed
          if (qn > 0) got = wait_or_abort(bars, smem_addr(&bars.q_empty), (qn - 1) & 1);
          if (got) {
            const uint32_t bar = smem_addr(&bars.q_full);
            mbar_arrive_expect_tx(bar, 2 * LY::kTile);
  #pragma unroll
            for (int x = 0; x < 2; ++x)
  #pragma unroll
              for (int hf = 0; hf < HALVES; ++hf)
                tma_load_3d(sQ + x * LY::kTile + hf * kHalf, &tmQ, hf * 64, h * G, un.tok0 + x * (kTileRows / G), bar);
            q_pending = true;
            last_q_par = qn & 1;
          }
        }
        if (!__shfl_sync(0xffffffffu, got, 0)) { ok = false; break; }
        ++qn;
        // page ids of 32 list entries at a time, the next group requested one group ahead
        constexpr int TPG = 32 / EPT;
        const int n_grp = (n_kt + TPG - 1) / TPG;
        auto fetch = [&](int grp, int& raw, bool& present) {
          const int v = item.v_begin + grp * 32 + lane;
          present = v < item.v_end;
          raw = present ? __ldg(trow + unit_entry(un, v)) : -1;
        };
        int raw;
        bool present;
        fetch(0, raw, present);
        for (int grp = 0; ok && grp < n_grp; ++grp) {
          int raw_n = -1;
          bool present_n = false;
          if (grp + 1 < n_grp) fetch(grp + 1, raw_n, present_n);
          const bool page_ok = present && raw >= 0 && raw < p.n_pool_pages;
          if (present && !page_ok) report(p.status, RK_ERR_DEVICE_BOUNDS);
          const int64_t row = page_ok ? int64_t(raw) * P : oob_row;
          const int tiles = min(TPG, n_kt - grp * TPG);
          for (int jt = 0; jt < tiles; ++jt, ++gg) {
            const int sk = gg % NK, sv = gg % NV;
            const int pg = lane - jt * EPT;
            got = true;
            if (lane == 0) {
              if (gg >= NK) got = wait_or_abort(bars, smem_addr(&bars.k_empty[sk]), ((gg / NK) - 1) & 1);
              if (got) {
                mbar_arrive_expect_tx(smem_addr(&bars.k_full[sk]), LY::kTile);
                last_k = sk;
                last_k_par = (gg / NK) & 1;
              }
            }
            if (!__shfl_sync(0xffffffffu, got, 0)) { ok = false; break; }
            if (pg >= 0 && pg < EPT)
  #pragma unroll
              for (int hf = 0; hf < HALVES; ++hf)
                tma_load_2d(sK + sk * LY::kTile + hf * kHalf + pg * P * 128, &tmK, hf * 64, int(row),
                            smem_addr(&bars.k_full[sk]));
            if (lane == 0) {
              if (gg >= NV) got = wait_or_abort(bars, smem_addr(&bars.v_empty[sv]), ((gg / NV) - 1) & 1);
              if (got) {
                mbar_arrive_expect_tx(smem_addr(&bars.v_full[sv]), LY::kTile);
                last_v = sv;
                last_v_par = (gg / NV) & 1;
              }
            }
            if (!__shfl_sync(0xffffffffu, got, 0)) { ok = false; break; }
            if (pg >= 0 && pg < EPT)
  #pragma unroll
              for (int hf = 0; hf < HALVES; ++hf)
                tma_load_2d(sV + sv * LY::kTile + hf * kHalf + pg * P * 128, &tmV, hf * 64, int(row),
                            smem_addr(&bars.v_full[sv]));
          }
          raw = raw_n;
          present = present_n;
        }
      }
      if (!ok && lane == 0) fail(bars, p.status);
      // copies still in flight after an abort: let them land before the CTA exits (bounded)
      if (lane == 0 && aborted(bars)) {
        if (last_k >= 0) mbar_wait(smem_addr(&bars.k_full[last_k]), last_k_par);
        if (last_v >= 0) mbar_wait(smem_addr(&bars.v_full[last_v]), last_v_par);
        if (q_pending) mbar_wait(smem_addr(&bars.q_full), last_q_par);
      }
    } else if (warp == 9) {
      // ---------------------------------------------------------------- MMA issuer
      if (lane == 0) {
        uint32_t gg = 0, qn = 0;
        bool ok = true, pending = false;
        uint32_t pend_bar = 0, pend_par = 0;
        for (int k = 0; ok; ++k) {
          if (!wait_or_abort(bars, smem_addr(&bars.iq_full[k & 1]), (k >> 1) & 1)) { ok = false; break; }
          const int it = bars.ring[k & 1];
          mbar_arrive(smem_addr(&bars.iq_empty[k & 1]));
          if (it < 0) break;
          const Item item = ws.items[it];
          const int n_kt = (item.v_end - item.v_begin + EPT - 1) / EPT;
          if (n_kt == 0) continue;
          if (!wait_or_abort(bars, smem_addr(&bars.q_full), qn & 1)) { ok = false; break; }
          ++qn;
          tc_fence_after();
          // order per tile j: S_A(j), O_B += P_B V (j-1), S_B(j), O_A += P_A V (j): the softmax of
          // one tile runs while the tensor core works for the other
          auto qk = [&](int x, uint32_t g1, uint32_t kb) -> bool {
            // S_x holds P_x of the previous tile, which that tile's value product reads.  That
            // product was issued before this one (after P_x was written), and the tensor pipe
            // runs the MMAs one thread issues in that order, so P_x is read before this S_x
            // overwrites it: no wait for the value product to complete.  (The softmax still
            // finds O_x complete when S_x arrives: the commit of S_x tracks every earlier MMA.)
            tc_fence_after();
            const uint32_t qb = sQ + x * LY::kTile;
  #pragma unroll
            for (int k = 0; k < D / 16; ++k) {
              const uint64_t a = desc_sw128(qb + (k >> 2) * kHalf + (k & 3) * 32, 16, 1024);
              const uint64_t b = desc_sw128(kb + (k >> 2) * kHalf + (k & 3) * 32, 16, 1024);
              tc_mma_f16(tmem + x * kKeysTc, a, b, kIdescQK, k > 0 ? 1u : 0u);
            }
            tc_commit(smem_addr(&bars.s_full[x]));
            return true;
          };
          auto pv = [&](int x, uint32_t g1, bool first) -> bool {
            const int sv = g1 % NV;
            if (!wait_or_abort(bars, smem_addr(&bars.v_full[sv]), (g1 / NV) & 1)) return false;
            if (!wait_or_abort(bars, smem_addr(&bars.p_full[x]), g1 & 1)) return false;
            tc_fence_after();
            const uint32_t vb = sV + sv * LY::kTile;
  #pragma unroll
            for (int k = 0; k < kKeysTc / 16; ++k) {
              const uint64_t b = desc_sw128(vb + k * 2048, kHalf, 1024);
              tc_mma_f16_ts(tmem + kColO + x * 128, tmem + x * kKeysTc + k * 8, b, kIdescPV, (!first || k > 0) ? 1u : 0u);
            }
            tc_commit(smem_addr(&bars.o_done[x]));
            if (x == 1) tc_commit(smem_addr(&bars.v_empty[sv]));   // both value products of tile g1 issued
            pending = true;
            pend_bar = smem_addr(&bars.o_done[x]);
            pend_par = g1 & 1;
            return true;
          };
          const uint32_t g_first = gg;
          for (int j = 0; j < n_kt; ++j, ++gg) {
            const int sk = gg % NK;
            if (!wait_or_abort(bars, smem_addr(&bars.k_full[sk]), (gg / NK) & 1)) { ok = false; break; }
            const uint32_t kb = sK + sk * LY::kTile;
            if (!qk(0, gg, kb)) { ok = false; break; }
            if (j >= 1 && !pv(1, gg - 1, gg - 1 == g_first)) { ok = false; break; }
            if (!qk(1, gg, kb)) { ok = false; break; }
            tc_commit(smem_addr(&bars.k_empty[sk]));
            if (j == n_kt - 1) tc_commit(smem_addr(&bars.q_empty));
            if (!pv(0, gg, j == 0)) { ok = false; break; }
          }
          if (ok && !pv(1, gg - 1, n_kt == 1)) ok = false;
        }
        if (!ok) fail(bars, p.status);
        if (pending && aborted(bars)) mbar_wait(pend_bar, pend_par);
      }
    } else if (ws.header->n_split > 0) {
      // ---------------------------------------------------------------- warps 10-11: merges
      if (!merge_split_units<D, true>(p, ws, bars, bars.job[1], 4, 64, tid - 320, n_items) && (tid & 31) == 0)
        fail(bars, p.status);
    }
  } else {
    regs_increase<kRegsHigh>();
    // ---------------------------------------------------------------- softmax + epilogue
    const int x = warp >> 2;                 // tile A (warps 0-3) or B (warps 4-7)
    const int r = tid & 127;                 // row of the tile = TMEM lane
    const int R = x * kTileRows + r;         // row of the unit
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    const uint32_t colS = x * kKeysTc, colO = kColO + x * 128;
    uint32_t gg = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const bool got_it = wait_or_abort(bars, smem_addr(&bars.iq_full[k & 1]), (k >> 1) & 1);
      if (!__all_sync(0xffffffffu, got_it)) { ok = false; break; }
      const int it = bars.ring[k & 1];
      mbar_arrive(smem_addr(&bars.iq_empty[k & 1]));
      if (it < 0) break;
      const Item item = ws.items[it];
      const Unit un = ws.units[item.unit];
      const int n_kt = (item.v_end - item.v_begin + EPT - 1) / EPT;
      const int seg = un.seg;
      const int h = seg % p.Hkv;
      const int32_t* lrow = p.page_logical ? p.page_logical + int64_t(seg) * p.max_pages : nullptr;
      const int rows_valid = un.ntok * G;
      const int pos = un.pos0 + R / G;
      const int L = __ldg(p.seq_len + un.b);
      const int cls = __ldg(p.head_class + seg);
      const bool local = cls == RK_CLASS_LOCAL;
      const int W = local ? __ldg(p.window + seg) : 0;
      const int S = (local && p.sink) ? __ldg(p.sink + seg) : 0;
      float m_ref = -INFINITY, l_sum = 0.f;
      // logical pages of the entries of tile j, requested one tile ahead
      auto load_lp = [&](int j, int (&lp)[EPT]) {
        const int v0 = item.v_begin + j * EPT;
#pragma unroll
        for (int pg = 0; pg < EPT; ++pg) {
          const int v = v0 + pg;
          lp[pg] = -1;
          if (j < n_kt && v < item.v_end) {
            const int e = unit_entry(un, v);
            lp[pg] = lrow ? __ldg(lrow + e) : e;
          }
        }
      };
      int lp_next[EPT];
      load_lp(0, lp_next);
      for (int j = 0; j < n_kt; ++j, ++gg) {
        int lp[EPT];
#pragma unroll
        for (int pg = 0; pg < EPT; ++pg) lp[pg] = lp_next[pg];
        load_lp(j + 1, lp_next);
        const bool got = wait_or_abort(bars, smem_addr(&bars.s_full[x]), gg & 1);
        if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
        tc_fence_after();
        // visibility of the tile's keys for this row: the whole tile (the common case) is
        // settled from its first and last page; otherwise one bit per slot of each page
        constexpr uint32_t kAll = P == 32 ? 0xffffffffu : 0xffffu;
        bool full;
        {
          bool all_listed = true;
          int lp_last = lp[0];
#pragma unroll
          for (int pg = 0; pg < EPT; ++pg) {
            all_listed &= lp[pg] >= 0;
            lp_last = lp[pg] >= 0 ? lp[pg] : lp_last;
          }
          const int j_min = lp[0] * P, j_max = lp_last * P + P - 1;
          full = all_listed && j_max <= pos && j_max < L && (!local || j_min > pos - W || j_max < S);
        }
        uint32_t pm[EPT];
        if (!full) {
#pragma unroll
          for (int pg = 0; pg < EPT; ++pg) {
            uint32_t m = 0u;
            if (lp[pg] >= 0) {
              const int base = lp[pg] * P;
              const int hi = min(pos, L - 1) - base;          // last visible slot (causal, length)
              m = hi < 0 ? 0u : (hi >= P - 1 ? kAll : (2u << hi) - 1u);
              if (local) {
                const int lo = pos - W + 1 - base;            // first slot inside the window
                const int sk = S - base;                      // slots before this are sink
                const uint32_t wm = lo <= 0 ? kAll : (lo >= P ? 0u : kAll & ~((1u << lo) - 1u));
                const uint32_t sm = sk <= 0 ? 0u : (sk >= P ? kAll : (1u << sk) - 1u);
                m &= wm | sm;
              }
            }
            pm[pg] = m;
          }
        }
        // the row's 128 scores, loaded from TMEM once; masked slots become -inf, which adds
        // nothing to the maximum and gives exp2 = 0
        const float sc = p.scale_log2;
        uint32_t v[kKeysTc];
#pragma unroll
        for (int q4 = 0; q4 < kKeysTc / 32; ++q4)
          tmem_ld32(tmem + lane_base + colS + q4 * 32, *reinterpret_cast<uint32_t(*)[32]>(&v[q4 * 32]));
        tmem_wait_ld();
        if (!full) {
#pragma unroll
          for (int c = 0; c < kKeysTc; ++c)
            if (!((pm[c / P] >> (c % P)) & 1u)) v[c] = __float_as_uint(-INFINITY);
        }
        float mx;
        {
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};   // four independent chains
#pragma unroll
          for (int i = 0; i < kKeysTc / 2; ++i)
            m4[i & 3] = fmax3(m4[i & 3], __uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
          mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * sc;
        }
        const float m_new = fmaxf(m_ref, mx);
        const bool rescale = m_new > m_ref + kRescaleThreshold;   // false while both are -inf
        // O_x already holds earlier tiles of this item (their value products completed before
        // this S was computed): rescale the rows whose maximum moved
        if (j > 0 && __any_sync(0xffffffffu, rescale)) {
          const float alpha = rescale ? fast_exp2(m_ref - m_new) : 1.f;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_base + colO + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(tmem + lane_base + colO + c * 32, o);
          }
          tmem_wait_st();
        }
        if (rescale) {
          l_sum = (m_ref == -INFINITY) ? 0.f : l_sum * fast_exp2(m_ref - m_new);
          m_ref = m_new;
        }
        const float nref = m_ref == -INFINITY ? 0.f : -m_ref;
        // P = 2^(S - m) as bf16 pairs: the 32 scores of chunk c become packed columns
        // 16c .. 16c+15 (their scores are already in registers)
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < kKeysTc / 32; ++c) {
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float e0 = fast_exp2(fmaf(__uint_as_float(v[c * 32 + 2 * i]), sc, nref));
            const float e1 = fast_exp2(fmaf(__uint_as_float(v[c * 32 + 2 * i + 1]), sc, nref));
            ps[i & 3] += e0 + e1;
            w[i] = pack_bf16(e0, e1);
          }
          tmem_st16(tmem + lane_base + colS + c * 16, w);
        }
        const float psum = (ps[0] + ps[1]) + (ps[2] + ps[3]);
        l_sum += psum;
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(smem_addr(&bars.p_full[x]));
      }
      if (!ok) break;
      // epilogue: O / l -> output (or split partial), 32 columns at a time
      if (n_kt > 0) {
        const bool got_o = wait_or_abort(bars, smem_addr(&bars.o_done[x]), (gg - 1) & 1);
        if (!__all_sync(0xffffffffu, got_o)) { ok = false; break; }
        tc_fence_after();
      }
      const bool split = un.n_splits > 1;
      const bool row_ok = R < rows_valid;
      const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
      const float lse = l_sum > 0.f ? (m_ref + fast_log2(l_sum)) * 0.69314718055994531f : -INFINITY;
      const int t = un.tok0 + R / G, hq = h * G + R % G;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        if (n_kt > 0) {
          tmem_ld32(tmem + lane_base + colO + c * 32, v);
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
          float* prow = ws.part_o + (int64_t(it) * ws.rows + R) * D + c * 32;
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(prow + i) =
                make_float4(__uint_as_float(v[i]) * inv, __uint_as_float(v[i + 1]) * inv,
                            __uint_as_float(v[i + 2]) * inv, __uint_as_float(v[i + 3]) * inv);
        }
      }
      tc_fence_before();
      if (row_ok) {
        if (!split) {
          if (p.lse) p.lse[int64_t(t) * p.Hq + hq] = lse;
        } else {
          ws.part_lse[int64_t(it) * ws.rows + R] = lse;
        }
      }
      if (split) {   // this warp's rows of the partial are stored: count them for the merge
        __threadfence();
        __syncwarp();
        if (lane == 0) atomicAdd(ws.unit_done + item.unit, 1);
      }
    }
    if (!ok && lane == 0) fail(bars, p.status);
    // every softmax warp gets here (all waits above are bounded); merge only if all are well
    if (named_bar_and(3, 256, ok) && ws.header->n_split > 0 &&
        !merge_split_units<D, false>(p, ws, bars, bars.job[0], 3, 256, tid, n_items) && lane == 0)
      fail(bars, p.status);
  }

  __syncthreads();
  if (warp == 9) {
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
  const cuuint32_t qbox[3] = {64, cuuint32_t(p.G), cuuint32_t(kTileRows / p.G)};
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
    // the warpgroups' register budgets add up to 384 x kRegsLaunch: a build launched with any
    // other count could leave the softmax warpgroups waiting for registers, so refuse it
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, prefill_tc_kernel<D, P>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != kRegsLaunch) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(prefill_tc_kernel<D, P>, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::kSmem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(grid), dim3(kTcThreads), LY::kSmem, stream, attr);
  return cudaLaunchKernelEx(&cfg, prefill_tc_kernel<D, P>, mq, mk, mv, p, ws);
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

int prefill_tc_rows() { return kUnitRows; }
int prefill_tc_keys() { return kKeysTc; }

cudaError_t launch_prefill_tc(const AttnParams& p, const AttnWorkspace& ws, int grid, cudaStream_t stream) {
  if (p.d == 128) return p.P == 16 ? launch_tc<128, 16>(p, ws, grid, stream) : launch_tc<128, 32>(p, ws, grid, stream);
  return p.P == 16 ? launch_tc<64, 16>(p, ws, grid, stream) : launch_tc<64, 32>(p, ws, grid, stream);
}

}  // namespace rk
