// SegPaged decode on the 5th-generation tensor cores (tcgen05 + TMEM), sm_103a.
//
// What it computes is stated in include/rk_api.h: one query per sequence at position
// seq_len - 1 attends to the keys its KV head lists in its own page table, with the
// window / sink edge applied as a predicate ("小红书 RedKnot" section 3, fourth component;
// "RedKnot" article, SegPagedAttention paragraph).  Decode reads every visible K/V row
// once and is bound by HBM bandwidth ("LLM 推理原理详解": decode is memory-bound).  All G
// query heads of a KV head share each K/V row, so the contraction runs on the tensor
// cores with the keys on the MMA's M side, which keeps the per-row arithmetic far below
// the memory time:
//   S^T[key][g]  = K[key][:] . q[g][:]           M = 128 keys, N = 16 (G heads, padded), K = d
//   O^T[c][g]   += V^T[c][key] . P^T[key][g]     M = 128 channels, N = 16, K = 128 keys
//
// Schedule: the 128-key tiles of all head segments form one sequence of T tiles and CTA c
// takes the share [cut(c), cut(c+1)) of it, cut(c) = c*T/gs (gs = the smaller of the grid,
// one CTA per SM, and T).  On the single-launch path, with early start the last shares are
// tapered (the CTAs dispatched last start late), and a cut that falls inside a segment of at
// most kShortTiles tiles moves to the nearer end of that segment, so short segments (the
// windows of local heads) are never split and need no merge; only long segments are shared
// by several CTAs.  Two exceptions: with no more tiles than CTAs every tile gets its own CTA
// (windows split too), and when no segment has more than kAlignTiles tiles and there are no
// more segments than CTAs, CTA c takes segment c whole.  Up to kDecFusedSegs head
// segments every CTA plans this itself (visible ranges in three interleaved rounds of
// loads, a block scan of the tile counts) and a segment shared by several CTAs is merged
// inside the kernel; beyond that, plan_decode_kernel (rk_plan.cu) plans and
// combine_decode_tc_kernel merges.  A share is walked as "portions" (the part of one
// segment inside the share).
//   warp 4   controller: walks the share, pushes each portion into a 2-entry ring, loads its
//            G query rows (TMA) into one of two Q buffers, and for every tile publishes into
//            a stage descriptor the physical page of each of its pages (from the page table),
//            the coefficient row of each page turned on load (k_rot), and the row that holds
//            the appended token (k_new / v_new).  Segment records and page ids are requested
//            one step ahead of their use.
//   warps 6-9 copy: gather each tile's K and V rows from the shared pools into a ring of
//            kStages stages with 16-byte cp.async copies, straight into the swizzled layout
//            the MMA reads (the appended row comes from k_new / v_new and is also stored into
//            its pool slot); with k_rot they turn the K rows of listed offline pages in shared
//            memory before releasing the stage.
//   warp 5   MMA issuer (one thread): issues whichever of S^T(j) (data landed, S buffer
//            free) or O^T += V^T P^T (P^T written) is ready, so neither waits on the other.
//   warps 0-3 softmax: thread t owns key t of the tile (TMEM lane t): masks it, finds the
//            tile maximum of every head (transposing shuffle reduction, one barrier),
//            keeps a per-head running maximum that moves only when it grows by more than
//            2^8 (then O^T is rescaled in TMEM), writes P^T = 2^(S - m) as bf16 into shared
//            memory, and at the end of a portion normalises O^T and stores it -- the output
//            itself, or, for a segment shared with other CTAs, a partial result for the
//            log-sum-exp merge.
// Every wait is bounded; a timeout sets RK_ERR_TIMEOUT and all roles leave.
#include "rk_internal.cuh"
#include "rk_sm100.cuh"

#include <algorithm>

namespace rk {

namespace {

using namespace sm100;

constexpr int kThreads = 320;           // warps 0-3 softmax, 4 controller, 5 MMA, 6-9 copy
constexpr int kCopyWarp0 = 6;
constexpr int kKeys = kDecTileKeys;     // keys per tile (MMA M of S^T)
constexpr int kN = 16;                  // MMA N: query heads of the group, padded
constexpr int kRing = 2;                // portion ring depth
constexpr float kRescale = 8.0f;        // log2 units
constexpr uint32_t kTmemCols = 64;      // S buffers at 0 and 16, O^T at 32
constexpr uint32_t kColO = 32;
constexpr int kHalfBytes = kKeys * 128; // one [128 keys][64 channels] bf16 box column
constexpr int kGrp = 32;                // list entries whose page ids the producer warp loads at once
constexpr uint64_t kWaitNs = 1000000000ull;
constexpr int kMaxTaperGrid = 256;  // tapered shares on grids up to this size

template <int D>
struct DecLayout {
  static constexpr int kStages = D == 128 ? 3 : 6;
  static constexpr int kStageBytes = (D / 64) * kHalfBytes;     // K (or V) of one tile
  static constexpr int kQBuf = (D / 64) * 2048;                 // [16][D] bf16, SW128 K-major
  static constexpr int kQ = 0;                                  // 2 Q buffers
  static constexpr int kP = kQ + 2 * kQBuf;                     // 2 x [16][128 keys] bf16
  static constexpr int kV = kP + 2 * 4096;                      // V stages, then K stages: for D = 64
  static constexpr int kK = kV + kStages * kStageBytes;         // V^T's second M half reads past a V stage
  static constexpr int kPlan = kK + kStages * kStageBytes;      // single-launch path: per-segment ranges
  static constexpr int kOrder = kPlan + kDecFusedSegs * 16;     // single-launch path: segment at each sequence
  static constexpr int kRank = kOrder + kDecFusedSegs * 2;      // position, and the position of each segment
  static constexpr int kBytes = kRank + kDecFusedSegs * 2;
  static constexpr int kSmem = kBytes + 1024;
};

// One segment's part of a CTA's share, as the producer hands it to the other roles.
struct Portion {
  int32_t seg, v_begin, v_end, slot;    // slot < 0: write the output directly
  int32_t n_kt, b, tok, pos;
  int32_t cls, W, S, L;
  int32_t n_splits, cta0, tile0;        // CTAs sharing the segment, the first of them, its first tile
  int32_t c0_later;                     // the segment is not the first portion of cta0's share
};

struct DecShared {
  uint64_t kv_full[6], kv_empty[6];
  uint64_t s_full[2], s_empty[2];
  uint64_t p_full[2], p_empty[2];
  uint64_t q_full[2], q_empty[2];
  uint64_t iq_full[kRing], iq_empty[kRing];
  Portion ring[kRing];
  uint64_t desc_full[6];    // controller -> copy warps: a stage's page ids are published
  int lp[6][8];             // logical page of each page slot of a stage (-1: none)
  int pid[6][8];            // physical page of each page slot of a stage (-1: none, zeros are copied)
  int cmd[6];               // per stage: 0 stop, 1 copy
  int app_row[6];           // per stage: the tile row that takes the new token (k_new / v_new), or -1
  int rot[6][8];            // per page slot of a stage: coefficient row of its K turn, or -1
  int any_rot[6];           // some page of the stage is turned
  int app_seg[6];           // its head segment
  float red[2][4][kN];      // per-warp tile maxima (double-buffered by tile parity)
  float redl[4][kN];        // per-warp denominators
  float lse2[kN];
  uint32_t tmem_slot;
  int abort;
  int T, gs, seg_first, last;   // single-launch path: the schedule, and "this CTA merges the splits"
  int tb, te, aligned, max_nt, long_first;
  int short_lim;                // segments of at most this many tiles are never split
  int taper;                    // tapered shares (0: equal shares); their raw cuts:
  int cuts[kMaxTaperGrid + 1];
  int s_warp[32];
  unsigned long long s_warp64[32];
};

__device__ __forceinline__ bool aborted(DecShared& sh) { return *reinterpret_cast<volatile int*>(&sh.abort) != 0; }
__device__ __forceinline__ void set_abort(DecShared& sh, int32_t* status) {
  report(status, RK_ERR_TIMEOUT);
  *reinterpret_cast<volatile int*>(&sh.abort) = 1;
}

// Bounded wait that also gives up as soon as another role has aborted.
__device__ __forceinline__ bool wait_or_abort(DecShared& sh, uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (aborted(sh)) return false;
    if (globaltimer() - t0 > kWaitNs) return false;
  }
}

__device__ __forceinline__ int seg_entry(const DecSeg& s, int v) { return v < s.e_sink ? v : s.e_w + (v - s.e_sink); }

// 16-byte global -> shared copy (L2 only); src_bytes 0 fills zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" :: "r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
// Arrive on the mbarrier once this thread's earlier cp.async copies have landed (counts as
// one of its expected arrivals).
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" :: "r"(bar) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" :: "r"(addr), "h"(v) : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" :: "r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// Reduce NG per-lane values over the 32 lanes of a warp, transposing as it goes: returns
// the reduction of column lane / (32 / NG) (every lane of that column group holds it).
template <int NG, bool MAX>
__device__ __forceinline__ float warp_reduce_cols(float (&v)[NG]) {
  int cnt = NG;
#pragma unroll
  for (int lvl = 0; lvl < 5; ++lvl) {
    const int off = 16 >> lvl;
    if (cnt > 1) {
      const int half = cnt >> 1;
      const bool upper = (threadIdx.x & off) != 0;
#pragma unroll
      for (int i = 0; i < NG / 2; ++i) {
        if (i < half) {
          const float keep = upper ? v[i + half] : v[i];
          const float send = upper ? v[i] : v[i + half];
          const float got = __shfl_xor_sync(0xffffffffu, send, off);
          v[i] = MAX ? fmaxf(keep, got) : keep + got;
        }
      }
      cnt = half;
    } else {
      const float got = __shfl_xor_sync(0xffffffffu, v[0], off);
      v[0] = MAX ? fmaxf(v[0], got) : v[0] + got;
    }
  }
  return v[0];
}

constexpr int kMergeFan = 12;   // partials one CTA merges at a time (single-launch path)
constexpr int kAlignTiles = 8;  // all segments this short and no more of them than CTAs: one segment per CTA
constexpr int kShortTiles = 8;  // single-launch path: segments this short are never split, unless
constexpr bool kSpread = true;  // there are no more tiles than CTAs: then every tile gets a CTA
constexpr int kLateShares = 8;  // short segments go last when they fill at most this many shares
// With early start the last gs / div shares shrink linearly, the last one by pct per cent of a
// full share: the strong setting when some segment spans more CTAs than one merge group.
constexpr int kTaperStrongDiv = 3, kTaperStrongPct = 60;
constexpr int kTaperMildDiv = 6, kTaperMildPct = 40;

// Partial slot of CTA c for a split segment (two per CTA: its first and its last portion):
// c's portion of the segment is its first one unless c = cta0 and c's share began in an
// earlier segment (c0_later).
__device__ __forceinline__ int split_slot(int c, int cta0, int c0_later) {
  return (c == cta0 && c0_later) ? 2 * c + 1 : 2 * c;
}

// Tapered shares.  With early start the CTAs are dispatched in index order as the SMs of
// the preceding call free up, and the last of them start several microseconds late (their
// SMs run that call's last CTAs, which also merge).  So the last L shares shrink linearly:
// share i < gs - L weighs 200 L, share gs - L + k - 1 (k = 1..L) weighs 200 L - 2 pct k,
// and share c begins at tile T * W(c) / W(gs), W(c) the weight of the shares before it.
// A segment spread over more CTAs than one merge group waits, for its final merge, for the
// latest of them, so such a call tapers more (kTaperStrongDiv / kTaperStrongPct).
__device__ __forceinline__ long long share_weight(int c, int gs, int L, int pct) {
  const long long m = max(0, c - (gs - L));
  return 200LL * L * c - pct * m * (m + 1);
}
// L for a call: none without early start or on a grid above kMaxTaperGrid, and none when the
// smallest share would hold less than one tile (consecutive cuts must stay distinct: every
// CTA between the first and the last of a split segment holds a piece of it).
__device__ __forceinline__ int taper_count(bool early, long long T, int gs, int div, int pct) {
  const int L = early && gs <= kMaxTaperGrid ? gs / div : 0;
  if (L == 0) return 0;
  return T * (2LL * L * (100 - pct)) >= share_weight(gs, gs, L, pct) ? L : 0;
}
__device__ __forceinline__ int share_raw(int c, long long T, int gs, int L, int pct) {
  if (c <= 0) return 0;
  if (c >= gs) return int(T);
  return L ? int(T * share_weight(c, gs, L, pct) / share_weight(gs, gs, L, pct)) : int((long long)c * T / gs);
}
// The CTA whose share holds tile t of a segment longer than kShortTiles: the last c whose
// raw first tile is at or before t.  cuts[c] = share_raw(c) when the shares are tapered, else
// NULL (closed form).
__device__ __forceinline__ int share_owner(long long t, long long T, int gs, const int* cuts) {
  if (!cuts) return int(((t + 1) * gs + T - 1) / T) - 1;
  int lo = 0, hi = gs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cuts[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// First tile of CTA c's share on the single-launch path: its raw first tile (c*T/gs, or the
// tapered cut), moved to the nearer end of the segment it falls in when that segment has at
// most kShortTiles tiles (ties go to its start).  Monotone in c, so the shares stay disjoint
// and cover [0, T).  A tile of a longer segment belongs to the same CTA as without the move:
// cuts inside it are not moved, and cuts moved within other segments stay on their side of
// it.  plan[s].w is the first tile of segment s in the sequence, plan[s].z its visible
// entries, order[i] the segment at sequence position i (or, with order NULL, segment i).
__device__ __forceinline__ int share_cut(int c, long long T, long long gs, const int* cuts, const int4* plan,
                                         const int16_t* order, int nseg, int ept, int short_lim) {
  if (c <= 0) return 0;
  if (c >= gs) return int(T);
  const int raw = cuts ? cuts[c] : int((long long)c * T / gs);
  int lo = 0, hi = nseg - 1;   // last sequence position whose segment starts at or before raw
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (plan[order ? order[mid] : mid].w <= raw) lo = mid; else hi = mid - 1;
  }
  const int s = order ? order[lo] : lo;
  const int t0 = plan[s].w, nt = (plan[s].z + ept - 1) / ept;
  if (raw <= t0 || raw >= t0 + nt || nt > short_lim) return raw;
  return raw - t0 <= t0 + nt - raw ? t0 : t0 + nt;
}

// Merge protocol of a split segment (single-launch path).  Each CTA holding a piece takes a
// ticket from the segment's (or group's) counter as its epilogue starts; the CTA with the
// last ticket merges.  Every other piece stores its partial and then raises its slot's flag
// with a release store (one thread, after a barrier of the storing threads); the merger
// waits for those flags with acquire loads, lowers them and returns the counter to zero, so
// all of it is zero again when the kernel ends.  The merger waits only for CTAs that took a
// ticket before it, which are running.
__device__ __forceinline__ int take_ticket(int32_t* cnt) { return atomicAdd(cnt, 1); }
__device__ __forceinline__ void raise_flag(int32_t* f) {
  asm volatile("st.release.gpu.s32 [%0], 1;" :: "l"(f) : "memory");
}
__device__ __forceinline__ void zero_word(int32_t* f) {
  asm volatile("st.relaxed.gpu.s32 [%0], 0;" :: "l"(f) : "memory");
}
__device__ __forceinline__ bool wait_flag(int32_t* f) {
  int v;
  asm volatile("ld.acquire.gpu.s32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
  if (v) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    __nanosleep(32);
    asm volatile("ld.acquire.gpu.s32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
    if (v) return true;
    if (globaltimer() - t0 > kWaitNs) return false;
  }
}

// Log-sum-exp merge of n normalised partials (lse in log2 units) of one segment, whose slots
// belong to CTAs c_first, c_first + stride, ...: into the bf16 output rows (and lse, natural
// log) or into one partial slot.  The 128 softmax threads each take (head, 4 channels)
// columns, two at a time, eight partials' loads in flight.
template <int D>
__device__ __forceinline__ void merge_splits(int n, int c_first, int stride, int cta0, int c0_later,
                                             const float* src_lse, const float* src_o, int G,
                                             __nv_bfloat16* out_row, float* lse_row, float* dst_lse, float* dst_o,
                                             int t) {
  constexpr int C4 = D / 4;
  const int NU = G * C4;
  for (int ub = 0; ub < NU; ub += 256) {
    const int u[2] = {ub + t, ub + 128 + t};
    float M[2] = {-INFINITY, -INFINITY}, den[2] = {0.f, 0.f};
    float4 acc[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
    for (int k0 = 0; k0 < n; k0 += 8) {
      float lv[2][8];
      float4 ov[2][8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int slot = k0 + k < n ? split_slot(c_first + (k0 + k) * stride, cta0, c0_later) : -1;
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          lv[x][k] = -INFINITY;
          ov[x][k] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (slot >= 0 && u[x] < NU) {
            const int g = u[x] / C4, c4 = u[x] - g * C4;
            lv[x][k] = __ldcg(src_lse + int64_t(slot) * G + g);
            ov[x][k] = __ldcg(reinterpret_cast<const float4*>(src_o + (int64_t(slot) * G + g) * D) + c4);
          }
        }
      }
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        float mc = M[x];
#pragma unroll
        for (int k = 0; k < 8; ++k) mc = fmaxf(mc, lv[x][k]);
        if (mc == -INFINITY) continue;
        const float f = fast_exp2(M[x] - mc);   // 0 while M is -inf
        den[x] *= f;
        acc[x].x *= f; acc[x].y *= f; acc[x].z *= f; acc[x].w *= f;
        M[x] = mc;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float w = fast_exp2(lv[x][k] - mc);
          den[x] += w;
          acc[x].x = fmaf(w, ov[x][k].x, acc[x].x); acc[x].y = fmaf(w, ov[x][k].y, acc[x].y);
          acc[x].z = fmaf(w, ov[x][k].z, acc[x].z); acc[x].w = fmaf(w, ov[x][k].w, acc[x].w);
        }
      }
    }
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      if (u[x] >= NU) continue;
      const int g = u[x] / C4, c4 = u[x] - g * C4;
      const float inv = den[x] > 0.f ? 1.f / den[x] : 0.f;
      const float l2 = den[x] > 0.f ? M[x] + fast_log2(den[x]) : -INFINITY;
      if (out_row) {
        uint2 o;
        o.x = pack_bf16(acc[x].x * inv, acc[x].y * inv);
        o.y = pack_bf16(acc[x].z * inv, acc[x].w * inv);
        *reinterpret_cast<uint2*>(out_row + g * D + c4 * 4) = o;
        if (lse_row && c4 == 0) lse_row[g] = l2 * 0.69314718055994531f;
      } else {
        *reinterpret_cast<float4*>(dst_o + g * D + c4 * 4) =
            make_float4(acc[x].x * inv, acc[x].y * inv, acc[x].z * inv, acc[x].w * inv);
        if (c4 == 0) dst_lse[g] = l2;
      }
    }
  }
}

template <int D, int NG, bool FUSED, bool ROT>
__global__ __launch_bounds__(kThreads, 1) void decode_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                                                                 AttnParams p, DecWorkspace ws) {
  using LY = DecLayout<D>;
  constexpr int NS = LY::kStages;
  constexpr int HALVES = D / 64;
  constexpr uint32_t kIdescQK = idesc_bf16(kKeys, kN, 0, 0);
  constexpr uint32_t kIdescPV = idesc_bf16(128, kN, 0, 1);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ DecShared sh;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sbase = smem_addr(smem);
  const uint32_t sQ = sbase + LY::kQ, sP = sbase + LY::kP, sV = sbase + LY::kV, sK = sbase + LY::kK;
  const int P = p.P, EPT = kKeys / P;

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_addr(&sh.kv_full[s]), 128);   // one arrival per copy thread, when its copies land
      mbar_init(smem_addr(&sh.kv_empty[s]), 1);
      mbar_init(smem_addr(&sh.desc_full[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_addr(&sh.s_full[s]), 1);
      mbar_init(smem_addr(&sh.s_empty[s]), 128);
      mbar_init(smem_addr(&sh.p_full[s]), 128);
      mbar_init(smem_addr(&sh.p_empty[s]), 1);
      mbar_init(smem_addr(&sh.q_full[s]), 1);
      mbar_init(smem_addr(&sh.q_empty[s]), 1);
    }
    for (int s = 0; s < kRing; ++s) {
      mbar_init(smem_addr(&sh.iq_full[s]), 1);
      mbar_init(smem_addr(&sh.iq_empty[s]), 129);
    }
    sh.abort = 0;
    sh.seg_first = p.B * p.Hkv;
    sh.max_nt = 0;
    mbar_fence_init();
  }
  if (warp == 4 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" :: "l"(&tmQ) : "memory");
  }
  if (warp == 5) {
    tmem_alloc(smem_addr(&sh.tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp < 4) {   // Q rows >= G and P^T rows >= G stay zero for the whole kernel
    for (int i = tid; i < (LY::kV - LY::kQ) / 16; i += 128) st_shared_v4(sQ + i * 16, make_uint4(0, 0, 0, 0));
    fence_proxy_async_smem();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_slot;
  // Stable metadata (single-launch path): plan and page ids are read while the preceding
  // kernel finishes; each role waits for it before touching q, the pools or any output.
  const bool early = FUSED && (p.flags & RK_ATTN_METADATA_STABLE) != 0;
  if (!early) grid_dependency_wait();   // the plan (and everything before it in the stream) is complete
  grid_launch_dependents();             // the next kernel may be scheduled as CTAs of this one finish

  const int G = p.G;
  const int nseg = p.B * p.Hkv;
  const int4* s_plan = reinterpret_cast<const int4*>(smem + LY::kPlan);

  if constexpr (FUSED) {
    // ---------------------------------------------------------------- plan (every CTA alike)
    // Thread i takes segments [i*per, i*per + per) (per <= 2), finds their visible ranges in
    // three interleaved rounds of loads, and block scans of their tile counts give each
    // segment's first tile; the share of this CTA follows as in the separate planner.
    int4* plan = reinterpret_cast<int4*>(smem + LY::kPlan);
    constexpr int kPer = (kDecFusedSegs + kThreads - 1) / kThreads;
    const int per = (nseg + kThreads - 1) / kThreads;
    const int s0 = tid * per;
    DecRange rr[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) if (i < per && s0 + i < nseg) rr[i].load1(p, s0 + i);
#pragma unroll
    for (int i = 0; i < kPer; ++i) if (i < per && s0 + i < nseg) rr[i].load2();
#pragma unroll
    for (int i = 0; i < kPer; ++i) if (i < per && s0 + i < nseg) rr[i].load3(p);
    // When the short segments (at most kShortTiles tiles: the windows of local heads) fill
    // only the last few shares, the sequence of tiles holds the longer segments first and the
    // short ones after them, each class in segment order: the CTAs dispatched last (whose SMs
    // the preceding call still holds, so they start late) then hold whole short segments,
    // and the pieces of long segments, which must all be done before their merge, go to CTAs
    // that start on time.  Otherwise (many windows: they would load the late CTAs with many
    // portions) the sequence is in segment order.  order[] / rank[] map sequence positions
    // and segments.  One scan counts, per thread's segments: short tiles (bits 0-12), long
    // segments (bits 13-22) and long tiles (bits 32-63).
    int nt[kPer], mx = 0;
    unsigned long long pk = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      nt[i] = 0;
      if (i < per && s0 + i < nseg) {
        rr[i].finish();
        nt[i] = (rr[i].n_vis + EPT - 1) / EPT;
        pk += nt[i] > kShortTiles ? (unsigned long long)nt[i] << 32 | (1ull << 13) : (unsigned long long)nt[i];
      }
      mx = max(mx, nt[i]);
    }
    if (mx > 0) atomicMax(&sh.max_nt, mx);   // read after the scan's barriers
    unsigned long long PK;
    const unsigned long long q0 = block_exclusive_scan64(pk, &PK, sh.s_warp64);
    const int TL = int(PK >> 32), TS = int(PK & 0x1fff), n_long = int((PK >> 13) & 0x3ff);
    const int T = TL + TS;
    const int l0 = int(q0 >> 32), s_tiles0 = int(q0 & 0x1fff), l_segs0 = int((q0 >> 13) & 0x3ff);
    const bool long_first = (long long)TS * min(int(gridDim.x), max(T, 1)) <= (long long)kLateShares * T;
    int16_t* order = reinterpret_cast<int16_t*>(smem + LY::kOrder);
    int16_t* rank = reinterpret_cast<int16_t*>(smem + LY::kRank);
    // Few, short segments (at most kAlignTiles tiles each, no more segments than CTAs): CTA c
    // takes segment c whole, so nothing is split.  Otherwise the equal shares.
    // No more tiles than CTAs: every tile its own CTA, windows split too (their pieces all
    // load at once, and a merge of a few partials costs less than a second round of copies).
    const bool spread = kSpread && T <= int(gridDim.x);
    const bool aligned = !spread && sh.max_nt <= kAlignTiles && nseg <= int(gridDim.x);
    const int short_lim = spread ? 0 : kShortTiles;
    const int gs = min(int(gridDim.x), T);
    const int c = blockIdx.x;
    // the longest segment spans about max_nt * gs / T CTAs
    const bool strong = (long long)sh.max_nt * gs > (long long)kMergeFan * T;
    const int tdiv = strong ? kTaperStrongDiv : kTaperMildDiv, tpct = strong ? kTaperStrongPct : kTaperMildPct;
    const int taper = aligned ? 0 : taper_count(early, T, gs, tdiv, tpct);
    if (taper)
      for (int i = tid; i <= gs; i += kThreads) sh.cuts[i] = share_raw(i, T, gs, taper, tpct);
    {
      // running first tile and sequence position of this thread's next long / short segment
      // (in segment order: of its next segment)
      int lt = l0, st = TL + s_tiles0, lr = l_segs0, sr = s0 - l_segs0, it = l0 + s_tiles0;
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int seg = s0 + i;
        if (i < per && seg < nseg) {
          const bool lg = nt[i] > kShortTiles;
          const int t1 = !long_first ? it : lg ? lt : st;
          const int r = !long_first ? seg : lg ? lr : n_long + sr;
          it += nt[i];
          plan[seg] = make_int4(rr[i].e_sink, rr[i].e_w, rr[i].n_vis, t1);
          order[r] = int16_t(seg);
          rank[seg] = int16_t(r);
          if (aligned && seg == c) {
            sh.tb = nt[i] > 0 ? t1 : T;
            sh.te = nt[i] > 0 ? t1 + nt[i] : T;
            sh.seg_first = seg;
          }
          if (lg) { lt += nt[i]; ++lr; } else { st += nt[i]; ++sr; }
        }
      }
    }
    if (tid == 0) {
      sh.T = T;
      sh.gs = gs;
      sh.aligned = aligned;
      sh.short_lim = short_lim;
      sh.long_first = long_first;
      sh.taper = taper;
      if (aligned && c >= nseg) sh.tb = sh.te = T;
    }
    __syncthreads();
    if (!aligned) {
      if (tid == 0) {
        const int* cuts = taper ? sh.cuts : nullptr;
        sh.tb = share_cut(c, T, gs, cuts, plan, long_first ? order : nullptr, nseg, EPT, short_lim);
        sh.te = share_cut(c + 1, T, gs, cuts, plan, long_first ? order : nullptr, nseg, EPT, short_lim);
      }
      __syncthreads();
      const int tb = sh.tb;
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int seg = s0 + i;
        if (i < per && seg < nseg && nt[i] > 0 && plan[seg].w <= tb && tb < plan[seg].w + nt[i]) sh.seg_first = seg;
      }
    }
    __syncthreads();
  }

  if (warp == 4) {
    // ------------------------------------------------------------------ producer
    DecCta my;
    if constexpr (FUSED) {
      my.seg0 = sh.seg_first;
      my.tile_begin = sh.tb;
      my.tile_end = sh.te;
    } else {
      my = ws.ctas[blockIdx.x];
    }
    int seg = my.seg0, t = my.tile_begin;
    const int t_end = my.tile_end;
    // the segment after s in the tile sequence (single launch: long segments first)
    const bool reordered = FUSED && sh.long_first;
    const int16_t* order = reordered ? reinterpret_cast<const int16_t*>(smem + LY::kOrder) : nullptr;
    const int16_t* rank = reinterpret_cast<const int16_t*>(smem + LY::kRank);
    auto next_seg = [&](int s) -> int {
      if (reordered) {
        if (s >= nseg) return nseg;
        const int r = rank[s] + 1;
        return r < nseg ? int(order[r]) : nseg;
      } else {
        return s + 1;
      }
    };
    // raw page id / logical page of entry v_begin + grp*32 + lane of segment s (present: listed)
    auto fetch = [&](int s, const DecSeg& sd, int v_begin, int v_end, int grp, int& raw_page, int& raw_lp,
                     int& raw_rot, bool& present) {
      const int v = v_begin + grp * kGrp + lane;
      present = s < nseg && v < v_end;
      raw_page = -1;
      raw_lp = -1;
      raw_rot = -1;
      if (present) {
        const int en = seg_entry(sd, v);
        raw_page = __ldg(p.page_table + int64_t(s) * p.max_pages + en);
        raw_lp = p.page_logical ? __ldg(p.page_logical + int64_t(s) * p.max_pages + en) : en;
        if constexpr (ROT) raw_rot = __ldg(p.k_rot + int64_t(s) * p.max_pages + en);
      }
    };
    auto load_seg = [&](int s) {
      DecSeg d;
      if (s < nseg) {
        if constexpr (FUSED) {
          const int4 r = s_plan[s];
          d.e_sink = r.x;
          d.e_w = r.y;
          d.n_vis = r.z;
          d.tile0 = r.w;
          d.n_tiles = (r.z + EPT - 1) / EPT;
          d.b = s / p.Hkv;
          d.tok = d.b;
          d.L = __ldg(p.seq_len + d.b);
          d.pos = d.L - 1;
          d.cls = __ldg(p.head_class + s);
          const bool local = d.cls == RK_CLASS_LOCAL;
          d.W = local ? __ldg(p.window + s) : 0;
          d.S = local && p.sink ? __ldg(p.sink + s) : 0;
          // only segments longer than kShortTiles are shared; the CTAs holding their tiles are
          // the ones the raw cuts give (cuts inside them are not moved)
          const long long T = sh.T;
          const int gs = sh.gs;
          const int* cuts = sh.taper ? sh.cuts : nullptr;
          const bool cut = d.n_tiles > sh.short_lim && !sh.aligned;
          const int c0 = cut ? share_owner(d.tile0, T, gs, cuts) : s;
          const int c1 = cut ? share_owner((long long)d.tile0 + d.n_tiles - 1, T, gs, cuts) : s;
          d.cta0 = c0;
          d.n_splits = c1 - c0 + 1;
          d.slot0 = (cut && c1 > c0) ? int(share_cut(c0, T, gs, cuts, s_plan, order, nseg, EPT, sh.short_lim) < d.tile0) : 0;   // c0_later
        } else {
          d = ws.segs[s];
        }
      } else {
        d.n_tiles = 0;
        d.tile0 = 0x7fffffff;
        d.n_vis = 0;
        d.e_sink = 0;
        d.e_w = 0;
      }
      return d;
    };
    uint32_t gg = 0, qn = 0;
    int last_q = -1;
    uint32_t last_q_parity = 0;
    bool ok = true;
    DecSeg cur = load_seg(t < t_end ? seg : nseg);
    while (t < t_end && cur.n_tiles == 0 && seg < nseg) {
      seg = next_seg(seg);
      cur = load_seg(seg);
    }
    int raw_page, raw_lp, raw_rot;
    bool present;
    fetch(seg, cur, (t < t_end && seg < nseg) ? (t - cur.tile0) * EPT : 0, cur.n_vis, 0, raw_page, raw_lp, raw_rot,
          present);
    // with stable metadata the page ids are published before the preceding kernel completes
    // (the copy warps wait for it before copying); q is read after that wait, just before the
    // first step that may block on the pipeline
    bool waited = !early;
    for (int k = 0; ok; ++k) {
      const int slot = k % kRing;
      if (k >= kRing) {
        bool got = true;
        if (lane == 0) got = wait_or_abort(sh, smem_addr(&sh.iq_empty[slot]), ((k / kRing) - 1) & 1);
        if (!__shfl_sync(0xffffffffu, got, 0)) { ok = false; break; }
      }
      const bool live = t < t_end && seg < nseg;
      Portion po;
      int lt1 = 0;
      if (live) {
        const int lt0 = t - cur.tile0;
        lt1 = min(cur.n_tiles, t_end - cur.tile0);
        po.seg = seg;
        po.v_begin = lt0 * EPT;
        po.v_end = min(cur.n_vis, lt1 * EPT);
        po.n_kt = lt1 - lt0;
        if constexpr (FUSED)   // two slots per CTA: its first portion and its last one
          po.slot = cur.n_splits > 1 ? 2 * int(blockIdx.x) + (t == my.tile_begin ? 0 : 1) : -1;
        else
          po.slot = cur.n_splits > 1 ? cur.slot0 + (int(blockIdx.x) - cur.cta0) : -1;
        po.n_splits = cur.n_splits;
        po.cta0 = cur.cta0;
        po.tile0 = cur.tile0;
        po.c0_later = FUSED ? cur.slot0 : 0;
        po.b = cur.b;
        po.tok = cur.tok;
        po.pos = cur.pos;
        po.cls = cur.cls;
        po.W = cur.W;
        po.S = cur.S;
        po.L = cur.L;
      } else {
        po.seg = -1;
        po.n_kt = 0;
      }
      if (lane == 0) {
        sh.ring[slot] = po;
        mbar_arrive(smem_addr(&sh.iq_full[slot]));
      }
      if (!live) break;
      // the next segment's record, used when this portion's last group is issued
      const bool more = cur.tile0 + lt1 < t_end;
      int nseg_idx = next_seg(seg);
      DecSeg nxt = load_seg(more ? nseg_idx : nseg);
      bool q_done = false;
      // Q rows of the group -> buffer qn & 1, free once the MMAs of portion qn - 2 are done
      auto load_q = [&]() -> bool {
        if (q_done) return true;
        if (!waited) {
          grid_dependency_wait();
          waited = true;
        }
        bool got = true;
        if (lane == 0) {
          const int b = qn & 1;
          if (qn >= 2) got = wait_or_abort(sh, smem_addr(&sh.q_empty[b]), ((qn >> 1) - 1) & 1);
          if (got) {
            const uint32_t bar = smem_addr(&sh.q_full[b]);
            mbar_arrive_expect_tx(bar, HALVES * G * 128);
#pragma unroll
            for (int hf = 0; hf < HALVES; ++hf)
              tma_load_3d(sQ + b * LY::kQBuf + hf * 2048, &tmQ, hf * 64, (po.seg % p.Hkv) * G, po.tok, bar);
            last_q = b;
            last_q_parity = (qn >> 1) & 1;
          }
        }
        q_done = true;
        ++qn;
        return __shfl_sync(0xffffffffu, got, 0);
      };
      const int lt_first = po.v_begin / EPT;            // tile of the segment the portion starts at
      const int tpg = kGrp / EPT;                       // tiles per group
      const int n_grp = (po.n_kt + tpg - 1) / tpg;
      for (int grp = 0; ok && grp < n_grp; ++grp) {
        int raw_page_n, raw_lp_n, raw_rot_n;
        bool present_n;
        if (grp + 1 < n_grp) {
          fetch(seg, cur, po.v_begin, po.v_end, grp + 1, raw_page_n, raw_lp_n, raw_rot_n, present_n);
        } else if (more) {
          while (nxt.n_tiles == 0 && nseg_idx < nseg) {   // segments with nothing visible
            nseg_idx = next_seg(nseg_idx);
            nxt = load_seg(nseg_idx);
          }
          fetch(nseg_idx, nxt, 0, nxt.n_vis, 0, raw_page_n, raw_lp_n, raw_rot_n, present_n);
        } else {
          raw_page_n = raw_lp_n = raw_rot_n = -1;
          present_n = false;
        }
        // this group's page ids go to the copy warps, one stage (tile) at a time
        const bool page_ok = present && raw_page >= 0 && raw_page < p.n_pool_pages;
        if (present && !page_ok) report(p.status, RK_ERR_DEVICE_BOUNDS);
        const int pidv = page_ok ? raw_page : -1;
        const int lpv = page_ok ? raw_lp : -1;
        int rotv = -1;
        if constexpr (ROT) {
          const bool rot_ok = raw_rot >= -1 && raw_rot < p.n_rot;
          if (page_ok && !rot_ok) report(p.status, RK_ERR_DEVICE_BOUNDS);
          rotv = page_ok && rot_ok ? raw_rot : -1;
        }
        const int tiles = min(tpg, po.n_kt - grp * tpg);
        for (int jt = 0; jt < tiles; ++jt, ++gg) {
          const int st = gg % NS;
          int lps[8], pids[8], rots[8];
#pragma unroll
          for (int pg = 0; pg < 8; ++pg) {
            lps[pg] = __shfl_sync(0xffffffffu, lpv, (jt * EPT + pg) & 31);
            pids[pg] = __shfl_sync(0xffffffffu, pidv, (jt * EPT + pg) & 31);
            rots[pg] = ROT ? __shfl_sync(0xffffffffu, rotv, (jt * EPT + pg) & 31) : -1;
          }
          // the segment's last tile holds the query position, where the new token goes
          int app_r = -1;
          if (p.k_new && lt_first + grp * tpg + jt == cur.n_tiles - 1) {
            const int pg = (cur.n_vis - 1) % EPT;
            int lpa = -1, pia = -1;
#pragma unroll
            for (int x = 0; x < 8; ++x)
              if (x == pg) { lpa = lps[x]; pia = pids[x]; }
            if (lpa == po.pos / P && pia >= 0) app_r = pg * P + po.pos % P;
            else if (lane == 0) report(p.status, RK_ERR_DEVICE_BOUNDS);
          }
          if (gg >= NS && !load_q()) { ok = false; break; }   // the wait below may block: q first
          bool got = true;
          if (lane == 0) {
            if (gg >= NS) got = wait_or_abort(sh, smem_addr(&sh.kv_empty[st]), ((gg / NS) - 1) & 1);
            if (got) {
              int any = 0;
#pragma unroll
              for (int pg = 0; pg < 8; ++pg) {
                sh.lp[st][pg] = pg < EPT ? lps[pg] : -1;
                sh.pid[st][pg] = pg < EPT ? pids[pg] : -1;
                if constexpr (ROT) {
                  sh.rot[st][pg] = pg < EPT ? rots[pg] : -1;
                  any |= (pg < EPT && rots[pg] >= 0) ? 1 : 0;
                }
              }
              if constexpr (ROT) sh.any_rot[st] = any;
              sh.cmd[st] = 1;
              sh.app_row[st] = app_r;
              sh.app_seg[st] = po.seg;
              mbar_arrive(smem_addr(&sh.desc_full[st]));
            }
          }
          if (!__shfl_sync(0xffffffffu, got, 0)) { ok = false; break; }
        }
        raw_page = raw_page_n;
        raw_lp = raw_lp_n;
        raw_rot = raw_rot_n;
        present = present_n;
      }
      if (ok && !load_q()) ok = false;
      t = cur.tile0 + lt1;
      seg = nseg_idx;
      cur = nxt;
    }
    if (ok && lane == 0) {   // no more tiles: the copy warps stop
      const int st = gg % NS;
      if (gg < NS || wait_or_abort(sh, smem_addr(&sh.kv_empty[st]), ((gg / NS) - 1) & 1)) {
        sh.cmd[st] = 0;
        mbar_arrive(smem_addr(&sh.desc_full[st]));
      } else {
        ok = false;
      }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok && lane == 0) set_abort(sh, p.status);
    // a Q copy still in flight after an abort lands before the CTA exits (bounded)
    if (lane == 0 && aborted(sh) && last_q >= 0) mbar_wait(smem_addr(&sh.q_full[last_q]), last_q_parity);
  } else if (warp >= kCopyWarp0) {
    // ------------------------------------------------------------------ copy warps
    // Tile rows go straight from the pools into the 128-byte-swizzled layout the MMA reads
    // (row r of a 64-channel block at r * 128 bytes, its 16-byte chunk c at chunk c ^ (r % 8)),
    // with 16-byte cp.async copies: a warp instruction moves whole rows of one page (512
    // contiguous bytes), and a copy thread's arrival on kv_full fires once its copies have landed.
    constexpr int CH = D / 8;                         // 16-byte chunks per row
    constexpr int RPI = 32 / CH;                      // rows per warp instruction
    const int cw = warp - kCopyWarp0;
    const int c16 = lane % CH, half = c16 >> 3, c = c16 & 7;
    const int rsub = lane / CH;
    const char* kb = reinterpret_cast<const char*>(p.k_pool);
    const char* vb = reinterpret_cast<const char*>(p.v_pool);
    const int pshift = P == 16 ? 4 : 5;
    // Repositioning on load: K rows of pages with a coefficient row are turned in shared memory
    // once this thread's copies of the stage have landed (each thread turns the chunks it
    // copied; the partner chunk of a half-split pair is the lane CH/2 away), then the stage
    // is released with a plain arrival.  The turn is rotate_pair, as in the RoPE kernel.
    constexpr int HCH = CH / 2;                       // chunks per half of a row
    const bool a_lane = c16 < HCH;
    int cur_rot = -1;
    float4 cf[8];
    auto turn_stage = [&](int st) {
      const int app = sh.app_row[st];
#pragma unroll
      for (int i = 0; i < 32 / RPI; ++i) {
        const int r = cw * 32 + i * RPI + rsub;
        const int rot = sh.rot[st][r >> pshift];
        const uint32_t addr = sK + st * LY::kStageBytes + half * kHalfBytes + r * 128 + ((c ^ (r & 7)) << 4);
        uint4 x;
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(x.x), "=r"(x.y), "=r"(x.z), "=r"(x.w) : "r"(addr));
        const bool go = rot >= 0 && r != app;
        if (go && rot != cur_rot) {   // coefficient rows change only between segments
          cur_rot = rot;
          const int i0 = p.rot_style == RK_ROPE_HALF_SPLIT ? 8 * (c16 % HCH) : 4 * c16;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            if (p.rot_style == RK_ROPE_HALF_SPLIT || k < 4) cf[k] = __ldg(p.rot_coef + int64_t(rot) * (D / 2) + i0 + k);
        }
        uint4 y = x;
        if (p.rot_style == RK_ROPE_HALF_SPLIT) {
          uint4 o;                                    // the partner chunk (same row, other half)
          o.x = __shfl_xor_sync(0xffffffffu, x.x, HCH);
          o.y = __shfl_xor_sync(0xffffffffu, x.y, HCH);
          o.z = __shfl_xor_sync(0xffffffffu, x.z, HCH);
          o.w = __shfl_xor_sync(0xffffffffu, x.w, HCH);
          if (go) {
            const uint4 xa = a_lane ? x : o, xb = a_lane ? o : x;
            float r8[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint32_t ua = (k >> 1) == 0 ? xa.x : (k >> 1) == 1 ? xa.y : (k >> 1) == 2 ? xa.z : xa.w;
              const uint32_t ub = (k >> 1) == 0 ? xb.x : (k >> 1) == 1 ? xb.y : (k >> 1) == 2 ? xb.z : xb.w;
              float ya, yb;
              rotate_pair((k & 1) ? bf16hi(ua) : bf16lo(ua), (k & 1) ? bf16hi(ub) : bf16lo(ub), cf[k], ya, yb);
              r8[k] = a_lane ? ya : yb;
            }
            y.x = pack_bf16(r8[0], r8[1]); y.y = pack_bf16(r8[2], r8[3]);
            y.z = pack_bf16(r8[4], r8[5]); y.w = pack_bf16(r8[6], r8[7]);
          }
        } else if (go) {                              // pairs (2i, 2i+1) inside the chunk
          float r8[8];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t u = k == 0 ? x.x : k == 1 ? x.y : k == 2 ? x.z : x.w;
            rotate_pair(bf16lo(u), bf16hi(u), cf[k], r8[2 * k], r8[2 * k + 1]);
          }
          y.x = pack_bf16(r8[0], r8[1]); y.y = pack_bf16(r8[2], r8[3]);
          y.z = pack_bf16(r8[4], r8[5]); y.w = pack_bf16(r8[6], r8[7]);
        }
        if (go) st_shared_v4(addr, y);
      }
      fence_proxy_async_smem();   // the turned rows (generic proxy) before the MMA reads them
      mbar_arrive(smem_addr(&sh.kv_full[st]));
    };
    int pending = -1;                                 // stage whose turn waits for its copies
    // the pools (and k_new / v_new) are read and written from here on; with stable pools the
    // copies start while the preceding kernel is still finishing
    if (early && !(p.flags & RK_ATTN_POOLS_STABLE)) grid_dependency_wait();
    for (uint32_t gg = 0;; ++gg) {
      const int st = gg % NS;
      if (!wait_or_abort(sh, smem_addr(&sh.desc_full[st]), (gg / NS) & 1)) break;
      const int cmd = sh.cmd[st];
      if (cmd == 0) break;
      // the new token (row app_r, if this stage holds it) is copied from k_new / v_new
      const int app_r = sh.app_row[st];
      const int64_t noff = int64_t(sh.app_seg[st]) * (D * 2) + c16 * 16;
      const char* kn = reinterpret_cast<const char*>(p.k_new) + noff;
      const char* vn = reinterpret_cast<const char*>(p.v_new) + noff;
#pragma unroll
      for (int i = 0; i < 32 / RPI; ++i) {
        const int r = cw * 32 + i * RPI + rsub;       // key of the tile
        const int pid = sh.pid[st][r >> pshift];
        const uint32_t doff = st * LY::kStageBytes + half * kHalfBytes + r * 128 + ((c ^ (r & 7)) << 4);
        const int64_t soff = pid >= 0 ? ((int64_t(pid) << pshift) + (r & (P - 1))) * (D * 2) + c16 * 16 : 0;
        const bool app = r == app_r;
        const uint32_t nb = (pid >= 0 || app) ? 16u : 0u;
        cp_async16(sK + doff, app ? kn : kb + soff, nb);
        cp_async16(sV + doff, app ? vn : vb + soff, nb);
      }
      if (app_r >= 0 && app_r / 32 == cw && (app_r % 32) % RPI == rsub) {
        // and stored into its pool slot for the later steps (the lanes that copied that row)
        const int pid = sh.pid[st][app_r >> pshift];
        const int64_t soff = ((int64_t(pid) << pshift) + (app_r & (P - 1))) * (D * 2) + c16 * 16;
        *reinterpret_cast<uint4*>(const_cast<char*>(kb) + soff) = __ldg(reinterpret_cast<const uint4*>(kn));
        *reinterpret_cast<uint4*>(const_cast<char*>(vb) + soff) = __ldg(reinterpret_cast<const uint4*>(vn));
      }
      if constexpr (ROT) {
        asm volatile("cp.async.commit_group;" ::: "memory");
        if (pending >= 0) {   // the previous stage's copies have landed once at most this one is open
          asm volatile("cp.async.wait_group 1;" ::: "memory");
          __syncwarp();
          turn_stage(pending);
          pending = -1;
        }
        if (sh.any_rot[st]) pending = st;
        else cp_async_arrive(smem_addr(&sh.kv_full[st]));
      } else {
        cp_async_arrive(smem_addr(&sh.kv_full[st]));
      }
    }
    cp_async_wait_all();   // nothing may land in shared memory after the CTA leaves
    if (pending >= 0 && !aborted(sh)) {
      __syncwarp();
      turn_stage(pending);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t gg = 0, qn = 0;
      bool ok = true, pending = false;
      uint32_t pend_bar = 0, pend_parity = 0;
      for (int k = 0; ok; ++k) {
        const int slot = k % kRing;
        if (!wait_or_abort(sh, smem_addr(&sh.iq_full[slot]), (k / kRing) & 1)) { ok = false; break; }
        const Portion po = sh.ring[slot];
        mbar_arrive(smem_addr(&sh.iq_empty[slot]));
        if (po.seg < 0) break;
        const int n_kt = po.n_kt;
        const int qb = qn & 1;
        if (!wait_or_abort(sh, smem_addr(&sh.q_full[qb]), (qn >> 1) & 1)) { ok = false; break; }
        const uint32_t sQb = sQ + qb * LY::kQBuf;
        tc_fence_after();
        // issue S^T(j) and the value product of earlier tiles in whatever order they become ready
        int qk = 0, pv = 0;
        uint64_t t_idle = 0;
        uint32_t spins = 0;
        while (pv < n_kt) {
          bool did = false;
          if (qk < n_kt) {
            const uint32_t g1 = gg + qk;
            const int st = g1 % NS, sb = g1 & 1;
            if (mbar_test(smem_addr(&sh.kv_full[st]), (g1 / NS) & 1) &&
                (g1 < 2 || mbar_test(smem_addr(&sh.s_empty[sb]), ((g1 >> 1) - 1) & 1))) {
              tc_fence_after();
              fence_proxy_async_smem();   // the copy warps' writes (generic proxy) before the MMA reads them
              const uint32_t kb = sK + st * LY::kStageBytes;
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint64_t a = desc_sw128(kb + (kk >> 2) * kHalfBytes + (kk & 3) * 32, 16, 1024);
                const uint64_t b = desc_sw128(sQb + (kk >> 2) * 2048 + (kk & 3) * 32, 16, 1024);
                tc_mma_f16(tmem + sb * kN, a, b, kIdescQK, kk > 0 ? 1u : 0u);
              }
              tc_commit(smem_addr(&sh.s_full[sb]));
              if (qk == n_kt - 1) tc_commit(smem_addr(&sh.q_empty[qb]));   // last read of this Q buffer
              ++qk;
              did = true;
            }
          }
          if (pv < qk) {
            const uint32_t g1 = gg + pv;
            const int st = g1 % NS, pb = g1 & 1;
            if (mbar_test(smem_addr(&sh.p_full[pb]), (g1 >> 1) & 1)) {
              tc_fence_after();
              const uint32_t vb = sV + st * LY::kStageBytes, pbase = sP + pb * 4096;
#pragma unroll
              for (int kk = 0; kk < kKeys / 16; ++kk) {
                const uint64_t a = desc_sw128(vb + kk * 2048, kHalfBytes, 1024);
                const uint64_t b = desc_sw128(pbase + (kk >> 2) * 2048 + (kk & 3) * 32, 16, 1024);
                tc_mma_f16(tmem + kColO, a, b, kIdescPV, (pv == 0 && kk == 0) ? 0u : 1u);
              }
              tc_commit(smem_addr(&sh.kv_empty[st]));
              tc_commit(smem_addr(&sh.p_empty[pb]));
              pending = true;
              pend_bar = smem_addr(&sh.p_empty[pb]);
              pend_parity = (g1 >> 1) & 1;
              ++pv;
              did = true;
            }
          }
          if (did) {
            t_idle = 0;
            spins = 0;
          } else if ((++spins & 255) == 0) {   // the timer and the abort flag are checked now and then
            if (aborted(sh)) { ok = false; break; }
            const uint64_t now = globaltimer();
            if (t_idle == 0) t_idle = now;
            else if (now - t_idle > kWaitNs) { ok = false; break; }
          }
        }
        gg += n_kt;
        ++qn;
      }
      if (!ok) set_abort(sh, p.status);
      if (pending && aborted(sh)) mbar_wait(pend_bar, pend_parity);
    }
  } else {
    // ------------------------------------------------------------------ softmax + epilogue (warps 0-3)
    const int t = tid;                               // key of the tile = TMEM lane
    const uint32_t lane_base = uint32_t(warp * 32) << 16;
    const float scale = p.scale_log2;
    constexpr int LPC = 32 / NG;                     // lanes per column after the transposing reduction
    const int my_col = lane / LPC;
    uint32_t gg = 0;
    bool ok = true;
    if (early) grid_dependency_wait();
    if ((p.flags & RK_ATTN_DIAG_EXPIRE_WAIT) && blockIdx.x == 0) {
      // diagnostic: a wait on a header word that nothing sets runs out; all roles then leave
      const bool got = t == 0 ? wait_flag(&ws.header->pad[0]) : true;
      ok = named_bar_and(1, 128, got);
    }
    if constexpr (FUSED) {
      // segments with nothing visible (every CTA planned them): out = 0, lse = -inf, written
      // by CTA seg % grid
      for (int seg = blockIdx.x; seg < nseg; seg += gridDim.x) {
        if (s_plan[seg].z != 0) continue;
        const int b = seg / p.Hkv, h = seg - b * p.Hkv;
        uint4* o = reinterpret_cast<uint4*>(p.out + (int64_t(b) * p.Hq + h * G) * D);
        for (int k = t; k < G * D / 8; k += 128) o[k] = make_uint4(0, 0, 0, 0);
        if (p.lse && t < G) p.lse[int64_t(b) * p.Hq + h * G + t] = -INFINITY;
      }
    }
    for (int k = 0; ok; ++k) {
      const int slot = k % kRing;
      const bool got_item = wait_or_abort(sh, smem_addr(&sh.iq_full[slot]), (k / kRing) & 1);
      if (!named_bar_and(1, 128, got_item)) { ok = false; break; }
      const Portion po = sh.ring[slot];
      mbar_arrive(smem_addr(&sh.iq_empty[slot]));
      if (po.seg < 0) break;
      const int h = po.seg % p.Hkv;
      const int n_kt = po.n_kt;
      const bool local = po.cls == RK_CLASS_LOCAL;

      float m[NG], l[NG];
#pragma unroll
      for (int g = 0; g < NG; ++g) { m[g] = -INFINITY; l[g] = 0.f; }
      // waits whose failure is only acted on at the next barrier (so all 128 threads leave together)
      bool good = true;
      for (int j = 0; j < n_kt; ++j, ++gg) {
        const int sb = gg & 1, st = gg % NS;
        // visibility of key t (the producer published the tile's logical pages before its copies)
        bool got = wait_or_abort(sh, smem_addr(&sh.kv_full[st]), (gg / NS) & 1);
        const int lp = sh.lp[st][t / P];
        const int jpos = lp * P + (t % P);
        const bool vis = lp >= 0 && jpos < po.L && jpos <= po.pos && (!local || jpos > po.pos - po.W || jpos < po.S);

        got &= wait_or_abort(sh, smem_addr(&sh.s_full[sb]), (gg >> 1) & 1);
        tc_fence_after();
        uint32_t sv[16];
        tmem_ld16(tmem + lane_base + sb * kN, sv);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(smem_addr(&sh.s_empty[sb]));
        float x[NG], r[NG];
        bool over = false;   // a key of this thread exceeds its head's running maximum by 2^8
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          x[g] = (vis && g < G) ? __uint_as_float(sv[g]) * scale : -INFINITY;
          r[g] = x[g];
          over |= x[g] > m[g] + kRescale;
        }
        // The running maxima move only when a key exceeds them by more than 2^8, so the tile's
        // maxima are needed only when some key does (always on a head's first visible key):
        // one barrier reduction over the 128 threads settles it.  A failed wait takes the
        // same branch, whose barrier then stops all of them.
        bool need = false;
        float mt[NG];
        if (named_bar_or(1, 128, over || !(got && good))) {
          const float wmax = warp_reduce_cols<NG, true>(r);
          if (lane % LPC == 0) sh.red[gg & 1][warp][my_col] = wmax;
          if (!named_bar_and(1, 128, got && good)) { ok = false; break; }
#pragma unroll
          for (int g = 0; g < NG; ++g) {
            mt[g] = fmaxf(fmaxf(sh.red[gg & 1][0][g], sh.red[gg & 1][1][g]),
                          fmaxf(sh.red[gg & 1][2][g], sh.red[gg & 1][3][g]));
            need |= mt[g] > m[g] + kRescale;
          }
        }
        if (need) {   // uniform across the 128 threads
          float alpha[NG];
#pragma unroll
          for (int g = 0; g < NG; ++g) {
            const float mn = mt[g] > m[g] + kRescale ? mt[g] : m[g];
            alpha[g] = m[g] == -INFINITY ? 0.f : fast_exp2(m[g] - mn);
            m[g] = mn;
            l[g] *= alpha[g];
          }
          if (j > 0) {   // O^T holds earlier tiles of this portion: wait for the last PV, rescale
            good &= wait_or_abort(sh, smem_addr(&sh.p_empty[(gg - 1) & 1]), ((gg - 1) >> 1) & 1);
            tc_fence_after();
            uint32_t ov[16];
            tmem_ld16(tmem + lane_base + kColO, ov);
            tmem_wait_ld();
#pragma unroll
            for (int g = 0; g < NG; ++g) ov[g] = __float_as_uint(__uint_as_float(ov[g]) * alpha[g]);
            tmem_st16(tmem + lane_base + kColO, ov);
            tmem_wait_st();
          }
        }
        // P^T buffer (gg & 1) is free once the PV of tile gg - 2 has completed
        if (gg >= 2) good &= wait_or_abort(sh, smem_addr(&sh.p_empty[gg & 1]), ((gg - 2) >> 1) & 1);
        const uint32_t pb = sP + (gg & 1) * 4096 + (t >> 6) * 2048 + ((t & 7) << 1);
        const int chunk = (t & 63) >> 3;
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          const float pv = fast_exp2(x[g] - (m[g] == -INFINITY ? 0.f : m[g]));
          l[g] += pv;
          const __nv_bfloat16 hb = __float2bfloat16_rn(pv);
          st_shared_u16(pb + g * 128 + ((chunk ^ (g & 7)) << 4), *reinterpret_cast<const uint16_t*>(&hb));
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(smem_addr(&sh.p_full[gg & 1]));
      }
      if (!ok) break;

      // ------------------------------------------------------------ epilogue
      const bool split = po.slot >= 0;
      // split segment: take the merge ticket now; its round trip overlaps the epilogue
      int ticket = 0;
      int32_t* cnt = nullptr;
      int need = 1, n_grp = 1, cq = 0, gslot = 0;
      bool two = false;
      if constexpr (FUSED) {
        if (split) {
          const int n = po.n_splits, j = int(blockIdx.x) - po.cta0;
          two = n > kMergeFan;
          n_grp = (n + kMergeFan - 1) / kMergeFan;
          const int q = j / kMergeFan;
          cq = po.cta0 + q * kMergeFan;
          gslot = split_slot(cq, po.cta0, po.c0_later);
          cnt = two ? ws.counters + kDecMaxGrid + gslot : ws.counters + po.cta0;
          need = two ? min(kMergeFan, n - q * kMergeFan) : n;
          if (t == 0) ticket = take_ticket(cnt);
        }
      }
      const bool got_o = wait_or_abort(sh, smem_addr(&sh.p_empty[(gg - 1) & 1]), ((gg - 1) >> 1) & 1);
      tc_fence_after();
      uint32_t ov[16];
      tmem_ld16(tmem + lane_base + kColO, ov);
      tmem_wait_ld();
      tc_fence_before();
      {
        float r[NG];
#pragma unroll
        for (int g = 0; g < NG; ++g) r[g] = l[g];
        const float wsum = warp_reduce_cols<NG, false>(r);
        if (lane % LPC == 0) sh.redl[warp][my_col] = wsum;
      }
      if (!named_bar_and(1, 128, got_o && good)) { ok = false; break; }
      float lt[NG];
#pragma unroll
      for (int g = 0; g < NG; ++g) lt[g] = sh.redl[0][g] + sh.redl[1][g] + sh.redl[2][g] + sh.redl[3][g];
      if (t < NG) {   // per-head lse in log2 units
        float mm = -INFINITY, ll = 0.f;
#pragma unroll
        for (int g = 0; g < NG; ++g) if (g == t) { mm = m[g]; ll = lt[g]; }
        sh.lse2[t] = ll > 0.f ? mm + fast_log2(ll) : -INFINITY;
      }
      named_bar_sync(1, 128);
      if (t < D) {
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          if (g < G) {
            const float val = lt[g] > 0.f ? __uint_as_float(ov[g]) / lt[g] : 0.f;
            if (!split) p.out[(int64_t(po.tok) * p.Hq + h * G + g) * D + t] = __float2bfloat16_rn(val);
            else ws.part_o[(int64_t(po.slot) * G + g) * D + t] = val;
          }
        }
      }
      if (t < G) {
        if (!split) {
          if (p.lse) p.lse[int64_t(po.tok) * p.Hq + h * G + t] = sh.lse2[t] * 0.69314718055994531f;
        } else {
          ws.part_lse[int64_t(po.slot) * G + t] = sh.lse2[t];
        }
      }
      if constexpr (FUSED) {
        if (split) {
          // Log-sum-exp merge of the segment's pieces by the CTA with the last ticket; beyond
          // kMergeFan pieces in two levels (groups of kMergeFan consecutive CTAs, then the
          // group results).
          int32_t* flags = ws.counters + 3 * kDecMaxGrid;    // per partial slot
          int32_t* gflags = ws.counters + 5 * kDecMaxGrid;   // per group slot
          named_bar_sync(1, 128);                            // every partial store of the CTA is done
          if (t == 0) sh.last = ticket == need - 1;
          named_bar_sync(1, 128);
          if (!sh.last) {
            if (t == 0) raise_flag(flags + po.slot);
          } else {
            int ticket2 = 0;
            if (t == 0) {
              zero_word(cnt);
              if (two) ticket2 = take_ticket(ws.counters + po.cta0);
            }
            if (t < need) {   // the group's (or segment's) other pieces
              const int s = split_slot(cq + t, po.cta0, po.c0_later);
              if (s != po.slot) {
                if (!wait_flag(flags + s)) report(p.status, RK_ERR_TIMEOUT);
                zero_word(flags + s);
              }
            }
            named_bar_sync(1, 128);
            __nv_bfloat16* out_row = p.out + (int64_t(po.tok) * p.Hq + h * G) * D;
            float* lse_row = p.lse ? p.lse + int64_t(po.tok) * p.Hq + h * G : nullptr;
            if (!two) {
              merge_splits<D>(need, cq, 1, po.cta0, po.c0_later, ws.part_lse, ws.part_o, G, out_row, lse_row,
                              nullptr, nullptr, t);
            } else {
              merge_splits<D>(need, cq, 1, po.cta0, po.c0_later, ws.part_lse, ws.part_o, G, nullptr, nullptr,
                              ws.grp_lse + int64_t(gslot) * G, ws.grp_o + int64_t(gslot) * G * D, t);
              named_bar_sync(1, 128);                        // the group result is stored
              if (t == 0) sh.last = ticket2 == n_grp - 1;
              named_bar_sync(1, 128);
              if (!sh.last) {
                if (t == 0) raise_flag(gflags + gslot);
              } else {
                if (t == 0) zero_word(ws.counters + po.cta0);
                if (t < n_grp) {
                  const int s = split_slot(po.cta0 + t * kMergeFan, po.cta0, po.c0_later);
                  if (s != gslot) {
                    if (!wait_flag(gflags + s)) report(p.status, RK_ERR_TIMEOUT);
                    zero_word(gflags + s);
                  }
                }
                named_bar_sync(1, 128);
                merge_splits<D>(n_grp, po.cta0, kMergeFan, po.cta0, po.c0_later, ws.grp_lse, ws.grp_o, G,
                                out_row, lse_row, nullptr, nullptr, t);
              }
            }
          }
        }
      }
      named_bar_sync(1, 128);   // sh.redl / sh.lse2 / sh.last are rewritten by the next portion
    }
    if (!ok && lane == 0) set_abort(sh, p.status);
  }

  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Merge the partial results of the split segments, one (segment, head) unit per block at
// a time: warp w takes partials w, w+8, ... (64 per round, all loads of a round in flight)
// and keeps a running log-sum-exp merge; lane l owns channels [4l, 4l+4).  The warps'
// states are merged at the end.
template <int D>
__global__ __launch_bounds__(256) void combine_decode_tc_kernel(AttnParams p, DecWorkspace ws) {
  grid_dependency_wait();   // the decode kernel is complete
  constexpr int C4 = D / 4;
  constexpr int PER = 8;    // partials per warp and round
  __shared__ float s_m[8], s_den[8];
  __shared__ float4 s_acc[8][C4];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.G;
  const int units = ws.header->n_split * G;
  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    const int seg = ws.split_segs[u / G], g = u % G;
    const DecSeg sd = ws.segs[seg];
    const int n = sd.n_splits, s0 = sd.slot0;
    float M = -INFINITY, den = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int base = 0; base < n; base += 8 * PER) {
      float lv[PER];
      float4 ov[PER];
#pragma unroll
      for (int k = 0; k < PER; ++k) {
        const int s = base + warp + 8 * k;
        lv[k] = -INFINITY;
        ov[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (s < n) {
          lv[k] = ws.part_lse[int64_t(s0 + s) * G + g];
          if (lane < C4) ov[k] = *reinterpret_cast<const float4*>(ws.part_o + (int64_t(s0 + s) * G + g) * D + lane * 4);
        }
      }
      float mc = M;
#pragma unroll
      for (int k = 0; k < PER; ++k) mc = fmaxf(mc, lv[k]);
      if (mc == -INFINITY) continue;
      const float f = M == -INFINITY ? 0.f : fast_exp2(M - mc);
      den *= f;
      acc.x *= f; acc.y *= f; acc.z *= f; acc.w *= f;
      M = mc;
#pragma unroll
      for (int k = 0; k < PER; ++k) {
        const float w = lv[k] == -INFINITY ? 0.f : fast_exp2(lv[k] - M);
        den += w;
        acc.x = fmaf(w, ov[k].x, acc.x); acc.y = fmaf(w, ov[k].y, acc.y);
        acc.z = fmaf(w, ov[k].z, acc.z); acc.w = fmaf(w, ov[k].w, acc.w);
      }
    }
    if (lane == 0) { s_m[warp] = M; s_den[warp] = den; }
    if (lane < C4) s_acc[warp][lane] = acc;
    __syncthreads();
    if (warp == 0 && lane < C4) {
      float Mt = s_m[0];
#pragma unroll
      for (int w = 1; w < 8; ++w) Mt = fmaxf(Mt, s_m[w]);
      float d = 0.f;
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        const float f = s_m[w] == -INFINITY ? 0.f : fast_exp2(s_m[w] - Mt);
        d += f * s_den[w];
        a.x = fmaf(f, s_acc[w][lane].x, a.x); a.y = fmaf(f, s_acc[w][lane].y, a.y);
        a.z = fmaf(f, s_acc[w][lane].z, a.z); a.w = fmaf(f, s_acc[w][lane].w, a.w);
      }
      const float inv = d > 0.f ? 1.f / d : 0.f;
      const int hq = (seg % p.Hkv) * G + g;
      uint2 o;
      o.x = pack_bf16(a.x * inv, a.y * inv);
      o.y = pack_bf16(a.z * inv, a.w * inv);
      *reinterpret_cast<uint2*>(p.out + (int64_t(sd.tok) * p.Hq + hq) * D + lane * 4) = o;
      if (p.lse && lane == 0)
        p.lse[int64_t(sd.tok) * p.Hq + hq] = d > 0.f ? (Mt + fast_log2(d)) * 0.69314718055994531f : -INFINITY;
    }
    __syncthreads();
  }
}

template <int D, int NG>
cudaError_t launch_t(const AttnParams& p, const DecWorkspace& ws, cudaStream_t stream) {
  const bool fused = p.B * p.Hkv <= kDecFusedSegs;
  using LY = DecLayout<D>;
  CUtensorMap mq;
  const cuuint64_t qdims[3] = {cuuint64_t(D), cuuint64_t(p.Hq), cuuint64_t(p.total_q)};
  const cuuint64_t qstr[2] = {cuuint64_t(D) * 2, cuuint64_t(p.Hq) * D * 2};
  const cuuint32_t qbox[3] = {64, cuuint32_t(p.G), 1};
  if (!encode_tmap_bf16(&mq, p.q, 3, qdims, qstr, qbox))
    return cudaErrorInvalidValue;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    cudaError_t e = cudaSuccess;
    for (auto* k : {decode_tc_kernel<D, NG, true, false>, decode_tc_kernel<D, NG, false, false>,
                    decode_tc_kernel<D, NG, true, true>, decode_tc_kernel<D, NG, false, true>})
      if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::kSmem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(ws.grid), dim3(kThreads), LY::kSmem, stream, attr);
  // the turn on load is compiled only into the kernels that use it
  const bool rot = p.k_rot != nullptr;
  if (fused)
    return rot ? cudaLaunchKernelEx(&cfg, decode_tc_kernel<D, NG, true, true>, mq, p, ws)
               : cudaLaunchKernelEx(&cfg, decode_tc_kernel<D, NG, true, false>, mq, p, ws);
  cudaError_t e = launch_plan_decode(p, ws, stream);
  if (e != cudaSuccess) return e;
  e = rot ? cudaLaunchKernelEx(&cfg, decode_tc_kernel<D, NG, false, true>, mq, p, ws)
          : cudaLaunchKernelEx(&cfg, decode_tc_kernel<D, NG, false, false>, mq, p, ws);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr2[1];
  cudaLaunchConfig_t cfg2 = pdl_config(dim3(4 * ws.grid), dim3(256), 0, stream, attr2);
  return cudaLaunchKernelEx(&cfg2, combine_decode_tc_kernel<D>, p, ws);
}

template <int D>
cudaError_t launch_d(const AttnParams& p, const DecWorkspace& ws, cudaStream_t stream) {
  switch (p.G) {
    case 1: case 2: case 4: return launch_t<D, 4>(p, ws, stream);
    case 8: return launch_t<D, 8>(p, ws, stream);
    case 16: return launch_t<D, 16>(p, ws, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_decode_tc(const AttnParams& p, const DecWorkspace& ws, cudaStream_t stream) {
  return p.d == 128 ? launch_d<128>(p, ws, stream) : launch_d<64>(p, ws, stream);
}

}  // namespace rk
