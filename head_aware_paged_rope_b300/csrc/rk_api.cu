// C-ABI entry points of librk: argument validation, workspace layout, launches.
// The computations themselves are described in include/rk_api.h and in the kernel files.
#include "rk_internal.cuh"

#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <string>

namespace rk {

int prefill_tc_rows();
int prefill_tc_keys();
cudaError_t launch_prefill_tc(const AttnParams& p, const AttnWorkspace& ws, int grid, cudaStream_t stream);

int device_sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
  if (dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  if (dev < 64) cache[dev] = n;
  return n;
}

namespace {

bool supported_dp(int d, int P) { return (d == 64 || d == 128) && (P == 16 || P == 32); }

// Prefill workspace sizes, shared by the workspace-size function and the entry point.
struct AttnLayout {
  int rows;         // rows per unit (query tile rows)
  int tok_per_unit;
  int max_units;
  int max_items;
  size_t off_units, off_items, off_lse, off_o, off_prefix, off_done, off_split, total;
};

rk_status check_attn(const rk_attn_args* a, bool decode) {
  if (!a) return RK_ERR_INVALID_ARG;
  if (a->B < 0 || a->Hq <= 0 || a->Hkv <= 0 || a->max_pages < 0 || a->total_q < 0 || a->max_q < 0 ||
      a->n_pool_pages < 0)
    return RK_ERR_INVALID_ARG;
  if (a->Hq % a->Hkv != 0) return RK_ERR_INVALID_ARG;
  if (!supported_dp(a->d, a->P)) return RK_ERR_UNSUPPORTED;
  const int G = a->Hq / a->Hkv;
  if (G > 16 || (G & (G - 1)) != 0) return RK_ERR_UNSUPPORTED;
  if (decode) {
    if (a->total_q != a->B || (a->B > 0 && a->max_q != 1)) return RK_ERR_INVALID_ARG;
  } else {
    if (a->max_q > a->total_q) return RK_ERR_INVALID_ARG;
    if (a->B > 0 && !a->cu_seqlens_q) return RK_ERR_INVALID_ARG;
  }
  if (a->B == 0 || a->total_q == 0) return RK_OK;
  if (!a->q || !a->seq_len || !a->k_pool || !a->v_pool || !a->n_pages || !a->head_class ||
      !a->window || !a->out)
    return RK_ERR_INVALID_ARG;
  if (a->max_pages > 0 && !a->page_table) return RK_ERR_INVALID_ARG;
  if (a->n_pool_pages * int64_t(a->P) >= (int64_t(1) << 31) || int64_t(a->total_q) * a->Hq >= (int64_t(1) << 31))
    return RK_ERR_UNSUPPORTED;   // row coordinates of the tensor maps are int32
  if (!std::isfinite(a->scale)) return RK_ERR_INVALID_ARG;
  if (a->flags & ~(RK_ATTN_METADATA_STABLE | RK_ATTN_POOLS_STABLE | RK_ATTN_DIAG_EXPIRE_WAIT)) return RK_ERR_INVALID_ARG;
  if ((a->k_new != nullptr) != (a->v_new != nullptr) || (!decode && a->k_new)) return RK_ERR_INVALID_ARG;
  if (a->k_rot) {
    if (!decode) return RK_ERR_UNSUPPORTED;   // prefill reads repositioned pages (rk_rope_reposition)
    if (!a->rot_coef || a->n_rot < 0 || (reinterpret_cast<uintptr_t>(a->rot_coef) & 15u) != 0) return RK_ERR_INVALID_ARG;
    if (a->rot_style != RK_ROPE_HALF_SPLIT && a->rot_style != RK_ROPE_INTERLEAVED) return RK_ERR_UNSUPPORTED;
  }
  return RK_OK;
}

// q, the pools and out are read and written with 16-byte vectors and TMA.
bool aligned16(const rk_attn_args* a) {
  const auto ok = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; };
  return ok(a->q) && ok(a->k_pool) && ok(a->v_pool) && ok(a->out) && ok(a->k_new) && ok(a->v_new);
}

AttnLayout attn_layout(const rk_attn_args* a) {
  AttnLayout l{};
  const int G = a->Hq / a->Hkv;
  l.rows = prefill_tc_rows();
  l.tok_per_unit = l.rows / G;
  const int64_t tiles = (int64_t(a->total_q) + l.tok_per_unit - 1) / l.tok_per_unit + a->B;
  l.max_units = int(std::min<int64_t>(tiles * a->Hkv, int64_t(1) << 30));
  l.max_items = l.max_units + kTargetItems;
  size_t off = align256(sizeof(PlanHeader));
  l.off_units = off;
  off += align256(sizeof(Unit) * size_t(l.max_units));
  l.off_items = off;
  off += align256(sizeof(Item) * size_t(l.max_items));
  l.off_lse = off;
  off += align256(sizeof(float) * size_t(l.max_items) * l.rows);
  l.off_o = off;
  off += sizeof(float) * size_t(l.max_items) * l.rows * a->d;   // tile prefix follows directly
  l.off_prefix = off;
  off += align256(sizeof(int32_t) * size_t(a->B + 1));
  l.off_done = off;
  off += align256(sizeof(int32_t) * size_t(l.max_units));
  l.off_split = off;
  off += align256(sizeof(int32_t) * size_t(l.max_units));
  l.total = off;
  return l;
}

AttnParams make_params(const rk_attn_args* a, const AttnLayout& l) {
  AttnParams p;
  p.q = static_cast<const __nv_bfloat16*>(a->q);
  p.cu_seqlens_q = a->cu_seqlens_q;
  p.seq_len = a->seq_len;
  p.k_pool = static_cast<const __nv_bfloat16*>(a->k_pool);
  p.v_pool = static_cast<const __nv_bfloat16*>(a->v_pool);
  p.n_pool_pages = a->n_pool_pages;
  p.page_table = a->page_table;
  p.page_logical = a->page_logical;
  p.n_pages = a->n_pages;
  p.head_class = a->head_class;
  p.window = a->window;
  p.sink = a->sink;
  p.B = a->B; p.Hq = a->Hq; p.Hkv = a->Hkv; p.d = a->d; p.P = a->P;
  p.max_pages = a->max_pages; p.total_q = a->total_q; p.max_q = a->max_q;
  p.G = a->Hq / a->Hkv;
  p.tok_per_unit = l.tok_per_unit;
  const float scale = a->scale > 0.f ? a->scale : 1.0f / std::sqrt(float(a->d));
  p.scale_log2 = scale * 1.4426950408889634f;
  p.out = static_cast<__nv_bfloat16*>(a->out);
  p.lse = a->lse;
  p.status = a->status;
  p.flags = a->flags;
  p.k_new = static_cast<const __nv_bfloat16*>(a->k_new);
  p.v_new = static_cast<const __nv_bfloat16*>(a->v_new);
  p.k_rot = a->k_rot;
  p.rot_coef = static_cast<const float4*>(a->rot_coef);
  p.n_rot = a->n_rot;
  p.rot_style = a->rot_style;
  return p;
}

AttnWorkspace make_ws(void* base, const AttnLayout& l) {
  uint8_t* b = static_cast<uint8_t*>(base);
  AttnWorkspace ws;
  ws.header = reinterpret_cast<PlanHeader*>(b);
  ws.units = reinterpret_cast<Unit*>(b + l.off_units);
  ws.items = reinterpret_cast<Item*>(b + l.off_items);
  ws.part_lse = reinterpret_cast<float*>(b + l.off_lse);
  ws.part_o = reinterpret_cast<float*>(b + l.off_o);
  ws.unit_done = reinterpret_cast<int32_t*>(b + l.off_done);
  ws.split_list = reinterpret_cast<int32_t*>(b + l.off_split);
  ws.max_units = l.max_units;
  ws.max_items = l.max_items;
  ws.rows = l.rows;
  return ws;
}

// Workspace of the tcgen05 decode path.
// The split counters sit at the same offset for every decode shape, so that one workspace
// serves any sequence of decode calls.
struct DecLayoutHost {
  int nseg, grid, max_slots;
  size_t off_counters, off_segs, off_ctas, off_split, off_lse, off_o, off_glse, off_go, total;
};

DecLayoutHost dec_layout(const rk_attn_args* a) {
  DecLayoutHost l{};
  const int G = a->Hq / a->Hkv;
  l.nseg = a->B * a->Hkv;
  l.grid = std::min(device_sm_count(), kDecMaxGrid);
  // separate planner: every CTA boundary splits at most one more segment;
  // single launch: two slots per CTA (its first and its last portion)
  l.max_slots = std::max(l.nseg + l.grid, 2 * l.grid);
  static_assert(sizeof(DecHeader) == 256, "the split counters start at byte 256");
  size_t off = align256(sizeof(DecHeader));
  l.off_counters = off;
  off += align256(sizeof(int32_t) * size_t(7 * kDecMaxGrid));   // ends at kDecCounterBytes
  l.off_segs = off;
  off += align256(sizeof(DecSeg) * size_t(l.nseg));
  l.off_ctas = off;
  off += align256(sizeof(DecCta) * size_t(l.grid));
  l.off_split = off;
  off += align256(sizeof(int32_t) * size_t(l.nseg));
  l.off_lse = off;
  off += align256(sizeof(float) * size_t(l.max_slots) * G);
  l.off_o = off;
  off += align256(sizeof(float) * size_t(l.max_slots) * G * a->d);
  l.off_glse = off;
  off += align256(sizeof(float) * size_t(2 * l.grid) * G);
  l.off_go = off;
  off += align256(sizeof(float) * size_t(2 * l.grid) * G * a->d);
  l.total = off;
  return l;
}

DecWorkspace make_dec_ws(void* base, const DecLayoutHost& l) {
  uint8_t* b = static_cast<uint8_t*>(base);
  DecWorkspace ws;
  ws.header = reinterpret_cast<DecHeader*>(b);
  ws.counters = reinterpret_cast<int32_t*>(b + l.off_counters);
  ws.segs = reinterpret_cast<DecSeg*>(b + l.off_segs);
  ws.ctas = reinterpret_cast<DecCta*>(b + l.off_ctas);
  ws.split_segs = reinterpret_cast<int32_t*>(b + l.off_split);
  ws.part_lse = reinterpret_cast<float*>(b + l.off_lse);
  ws.part_o = reinterpret_cast<float*>(b + l.off_o);
  ws.grp_lse = reinterpret_cast<float*>(b + l.off_glse);
  ws.grp_o = reinterpret_cast<float*>(b + l.off_go);
  ws.max_slots = l.max_slots;
  ws.grid = l.grid;
  return ws;
}

size_t decode_ws_bytes(const rk_attn_args* a) { return dec_layout(a).total; }

rk_status check_ws(void* ws, size_t bytes, size_t need) {
  if (need == 0) return RK_OK;
  if (!ws || bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return RK_ERR_WORKSPACE;
  return RK_OK;
}

rk_status run_attention(const rk_attn_args* a, void* workspace, size_t bytes, cudaStream_t stream, bool decode) {
  rk_status st = check_attn(a, decode);
  if (st != RK_OK) return st;
  if (a->B == 0 || a->total_q == 0) return RK_OK;
  const int sms = device_sm_count();
  if (decode) {
    if (int64_t(a->B) * a->Hkv > kDecMaxSegs) return RK_ERR_UNSUPPORTED;
    const DecLayoutHost dl = dec_layout(a);
    st = check_ws(workspace, bytes, dl.total);
    if (st != RK_OK) return st;
    if (!aligned16(a)) return RK_ERR_INVALID_ARG;
    AttnLayout l{};
    l.rows = a->Hq / a->Hkv;
    l.tok_per_unit = 1;
    const AttnParams p = make_params(a, l);
    const DecWorkspace ws = make_dec_ws(workspace, dl);
    const cudaError_t e = launch_decode_tc(p, ws, stream);
    return e == cudaSuccess ? RK_OK : RK_ERR_CUDA;
  }
  const AttnLayout l = attn_layout(a);
  st = check_ws(workspace, bytes, l.total);
  if (st != RK_OK) return st;
  if (!aligned16(a)) return RK_ERR_INVALID_ARG;
  const AttnParams p = make_params(a, l);
  const AttnWorkspace ws = make_ws(workspace, l);
  const int grid = std::max(1, std::min(l.max_items, sms));
  const int ept = prefill_tc_keys() / a->P;
  cudaError_t e = launch_plan(p, ws, l.tok_per_unit, ept, std::min(kTargetItems, grid * kItemsPerCta), kMinChunkTiles, stream);
  if (e == cudaSuccess) e = launch_prefill_tc(p, ws, grid, stream);
  return e == cudaSuccess ? RK_OK : RK_ERR_CUDA;
}

}  // namespace
}  // namespace rk

extern "C" {

size_t rk_rope_workspace_size(int32_t n_runs, int32_t d) {
  if (n_runs < 0 || d <= 0) return 0;
  return rk::align256(sizeof(float4) * size_t(n_runs) * size_t(d / 2));
}

rk_status rk_rope_reposition(const rk_rope_args* a, void* workspace, size_t workspace_bytes, rk_stream_t stream) {
  if (!a) return RK_ERR_INVALID_ARG;
  if (a->n_runs < 0 || a->max_tok < 0 || a->n_src_pages < 0 || a->n_dst_pages < 0 || a->n_src_entries < 0 ||
      a->n_dst_entries < 0)
    return RK_ERR_INVALID_ARG;
  if (!rk::supported_dp(a->d, a->P)) return RK_ERR_UNSUPPORTED;
  if (a->style != RK_ROPE_HALF_SPLIT && a->style != RK_ROPE_INTERLEAVED) return RK_ERR_UNSUPPORTED;
  if (!(a->theta > 1.0) || !std::isfinite(a->theta)) return RK_ERR_INVALID_ARG;
  if (a->n_runs == 0 || a->max_tok == 0) return RK_OK;
  if (!a->k_src || !a->k_dst || !a->src_tables || !a->dst_tables || !a->runs) return RK_ERR_INVALID_ARG;
  if (a->max_tok > 65535 * 128) return RK_ERR_UNSUPPORTED;
  const size_t need = rk_rope_workspace_size(a->n_runs, a->d);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return RK_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(a->k_src) & 15u) != 0 || (reinterpret_cast<uintptr_t>(a->k_dst) & 15u) != 0)
    return RK_ERR_INVALID_ARG;   // rows move by 16-byte bulk copies and vector stores
  const cudaError_t e = rk::launch_rope(*a, workspace, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? RK_OK : RK_ERR_CUDA;
}

rk_status rk_rope_coefficients(const int32_t* deltas, int32_t n, int32_t d, double theta, void* coef,
                               rk_stream_t stream) {
  if (n < 0) return RK_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return RK_ERR_UNSUPPORTED;
  if (!(theta > 1.0) || !std::isfinite(theta)) return RK_ERR_INVALID_ARG;
  if (n == 0) return RK_OK;
  if (!deltas || !coef || (reinterpret_cast<uintptr_t>(coef) & 15u) != 0) return RK_ERR_INVALID_ARG;
  if (n > 65535) return RK_ERR_UNSUPPORTED;
  return rk::launch_rope_coefficients(deltas, n, d, theta, coef, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? RK_OK : RK_ERR_CUDA;
}

size_t rk_segpaged_prefill_workspace_size(const rk_attn_args* a) {
  if (rk::check_attn(a, false) != RK_OK) return 0;
  if (a->B == 0 || a->total_q == 0) return 0;
  return rk::attn_layout(a).total;
}

size_t rk_segpaged_decode_workspace_size(const rk_attn_args* a) {
  if (rk::check_attn(a, true) != RK_OK) return 0;
  if (a->B == 0 || a->total_q == 0) return 0;
  return rk::decode_ws_bytes(a);
}

rk_status rk_segpaged_prefill(const rk_attn_args* a, void* ws, size_t bytes, rk_stream_t stream) {
  return rk::run_attention(a, ws, bytes, reinterpret_cast<cudaStream_t>(stream), false);
}

rk_status rk_segpaged_decode(const rk_attn_args* a, void* ws, size_t bytes, rk_stream_t stream) {
  return rk::run_attention(a, ws, bytes, reinterpret_cast<cudaStream_t>(stream), true);
}

rk_status rk_append_kv(const rk_append_args* a, rk_stream_t stream) {
  if (!a) return RK_ERR_INVALID_ARG;
  if (a->B < 0 || a->Hkv < 0 || a->max_pages < 0 || a->n_pool_pages < 0) return RK_ERR_INVALID_ARG;
  if (!rk::supported_dp(a->d, a->P)) return RK_ERR_UNSUPPORTED;
  if (a->B == 0 || a->Hkv == 0) return RK_OK;
  if (!a->k_new || !a->v_new || !a->pos || !a->k_pool || !a->v_pool || !a->page_table || !a->n_pages)
    return RK_ERR_INVALID_ARG;
  const auto al16 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; };
  if (!al16(a->k_new) || !al16(a->v_new) || !al16(a->k_pool) || !al16(a->v_pool)) return RK_ERR_INVALID_ARG;
  if (int64_t(a->B) * a->Hkv >= (int64_t(1) << 31) / 32) return RK_ERR_UNSUPPORTED;
  return rk::launch_append_kv(*a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? RK_OK : RK_ERR_CUDA;
}

rk_status rk_ring_advance(const rk_ring_args* a, rk_stream_t stream) {
  if (!a) return RK_ERR_INVALID_ARG;
  if (a->B < 0 || a->Hkv < 0 || a->max_pages < 0) return RK_ERR_INVALID_ARG;
  if (a->P != 16 && a->P != 32) return RK_ERR_UNSUPPORTED;
  if (a->B == 0 || a->Hkv == 0) return RK_OK;
  if (!a->pos || !a->page_table || !a->page_logical || !a->n_pages || !a->ring || !a->window)
    return RK_ERR_INVALID_ARG;
  if (!a->src_page_table != !a->src_page_logical) return RK_ERR_INVALID_ARG;   // both or neither
  if (a->src_page_table && (a->src_page_table == a->page_table || a->src_page_logical == a->page_logical ||
                            a->src_page_table == a->page_logical || a->src_page_logical == a->page_table))
    return RK_ERR_INVALID_ARG;
  if (int64_t(a->B) * a->Hkv >= (int64_t(1) << 31) / 32) return RK_ERR_UNSUPPORTED;
  return rk::launch_ring_advance(*a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? RK_OK : RK_ERR_CUDA;
}

namespace {
rk_status check_ffn(const rk_sparse_ffn_args* a) {
  if (!a) return RK_ERR_INVALID_ARG;
  if (a->T < 0 || a->d_model <= 0 || a->d_ff <= 0 || a->keep < 0 || a->keep > a->T) return RK_ERR_INVALID_ARG;
  if (a->d_model % 256 != 0 || a->d_ff % 128 != 0 || a->T > 65536) return RK_ERR_UNSUPPORTED;
  if (a->T == 0) return RK_OK;
  if (!a->x || !a->importance || !a->out || (a->keep > 0 && (!a->w_gate || !a->w_up || !a->w_down || !a->kept)))
    return RK_ERR_INVALID_ARG;
  const auto al16 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; };
  if (!al16(a->x) || !al16(a->out) || !al16(a->w_gate) || !al16(a->w_up) || !al16(a->w_down)) return RK_ERR_INVALID_ARG;
  return RK_OK;
}
}  // namespace

size_t rk_sparse_ffn_workspace_size(const rk_sparse_ffn_args* a) {
  if (check_ffn(a) != RK_OK || a->keep == 0) return 0;
  return rk::sparse_ffn_ws_bytes(a->keep, a->d_model, a->d_ff);
}

rk_status rk_sparse_ffn(const rk_sparse_ffn_args* a, void* ws, size_t bytes, rk_stream_t stream) {
  const rk_status st = check_ffn(a);
  if (st != RK_OK || a->T == 0) return st;
  if (a->keep > 0) {
    const size_t need = rk::sparse_ffn_ws_bytes(a->keep, a->d_model, a->d_ff);
    if (!ws || bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return RK_ERR_WORKSPACE;
  }
  return rk::launch_sparse_ffn(*a, ws, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? RK_OK : RK_ERR_CUDA;
}

const char* rk_status_string(rk_status s) {
  switch (s) {
    case RK_OK: return "ok";
    case RK_ERR_INVALID_ARG: return "invalid argument";
    case RK_ERR_UNSUPPORTED: return "unsupported configuration";
    case RK_ERR_CUDA: return "CUDA error";
    case RK_ERR_DEVICE_BOUNDS: return "device-side bounds check failed";
    case RK_ERR_TIMEOUT: return "device-side wait timed out";
    case RK_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case RK_ERR_DEVICE_ORDER: return "device-side check failed: page_logical list not ascending";
  }
  return "unknown status";
}

int32_t rk_version(void) { return 100; }

}  // extern "C"
