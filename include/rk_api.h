/*
 * rk_api.h -- C ABI of librk: RoPE repositioning of cached K and SegPagedAttention
 * (per-head paged attention without an attention mask) on NVIDIA B300 (sm_103a).
 *
 * What the calls compute, and where the RedKnot pages state it:
 *
 *  - rk_rope_reposition: "RedKnot" article (is96.com), paragraphs on RoPE and on the
 *    correction RedKnot applies to reused KV: K of a reusable segment was cached with
 *    the rotation of its offline position; the call turns it back by that rotation and
 *    forward by the rotation of its online position.  "小红书 RedKnot" product page,
 *    section 3, second component (offline KV reuse + RoPE repositioning).
 *  - rk_segpaged_prefill / rk_segpaged_decode: "小红书 RedKnot", section 3, fourth
 *    component (SegPagedAttention: an own page table per head, segmented KV storage, a
 *    different visible window per head class, no attn_mask); "RedKnot" article,
 *    SegPagedAttention paragraph (each head segment's table records which pages the
 *    head reads); head classes from section 3, first component (global, local,
 *    retrieval, dense); page pool and block tables from "PagedAttention &
 *    RadixAttention", section "The Solution: Fixed-size blocks".
 *
 * Conventions common to every call
 *  - bf16 tensors are passed as `void*` to 2-byte elements (IEEE bfloat16 bit patterns).
 *  - Every pointer argument is a DEVICE pointer owned by the caller, except the
 *    argument struct itself, which is read on the host during the call only.
 *  - The library never allocates device memory and never synchronises.  Work is
 *    enqueued on `stream` (a cudaStream_t; NULL = the legacy default stream).  Scratch
 *    memory is the caller's `workspace`, sized by the matching *_workspace_size call.
 *    RoPE and prefill workspaces need no initialisation and are undefined afterwards;
 *    a decode workspace must be zero-filled before its first decode call (see
 *    rk_segpaged_decode).
 *  - Host-side validation happens before anything is enqueued; on an error nothing is
 *    enqueued.  Checks that need device data (page ids inside the pool, slots inside a
 *    table) run in the kernels: a failing access is skipped and RK_ERR_DEVICE_BOUNDS
 *    is written to `*status` (when `status` is non-NULL; the first error code wins, the
 *    caller zeroes the word and reads it after synchronising).
 *  - Page pools are [n_pages][P][d] bf16, d contiguous; page id p refers to the same
 *    page index in the K pool and in the V pool.  P in {16, 32}; d in {64, 128}.
 *  - A head segment is one (sequence b, KV head h) pair with index b*Hkv + h.
 */
#ifndef RK_API_H
#define RK_API_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define RK_API __attribute__((visibility("default")))
#else
#define RK_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* rk_stream_t; /* same type as cudaStream_t */

typedef enum rk_status {
  RK_OK = 0,
  RK_ERR_INVALID_ARG = 1,    /* host-side validation failed; nothing enqueued */
  RK_ERR_UNSUPPORTED = 2,    /* valid but not implemented (e.g. d or P outside the sets above) */
  RK_ERR_CUDA = 3,           /* a CUDA runtime call or kernel launch failed */
  RK_ERR_DEVICE_BOUNDS = 4,  /* device-side check: page id / slot / table index out of range */
  RK_ERR_TIMEOUT = 5,        /* device-side bounded wait gave up */
  RK_ERR_WORKSPACE = 6,      /* workspace NULL, misaligned (256 B) or smaller than required */
  RK_ERR_DEVICE_ORDER = 7    /* device-side check: a page_logical list is not ascending */
} rk_status;

/* Head classes ("小红书 RedKnot", section 3, first component). */
enum { RK_CLASS_GLOBAL = 0, RK_CLASS_LOCAL = 1, RK_CLASS_RETRIEVAL = 2, RK_CLASS_DENSE = 3 };

/* Channel pairing of the rotation: (i, i + d/2) or (2i, 2i + 1). */
enum { RK_ROPE_HALF_SPLIT = 0, RK_ROPE_INTERLEAVED = 1 };

/* ------------------------------------------------------------------------------------
 * RoPE repositioning
 *
 * One run moves n_tok consecutive tokens of one head segment.  Token t (0 <= t < n_tok)
 *   - is read from the offline store: logical slot s = pos_off0 + t of the run's source
 *     table, i.e. row (src_tables[src_tab_off + s / P], s % P) of k_src;
 *   - is written to the online pool: logical slot u = pos_on0 + t of the run's
 *     destination table, i.e. row (dst_tables[dst_tab_off + u / P], u % P) of k_dst;
 *   - is rotated, for every channel pair i < d/2, back by pos_off * w_i and forward by
 *     pos_on * w_i, with w_i = theta^(-2i/d), pos_off = pos_off0 + t, pos_on = pos_on0 + t.
 * Since both positions advance together the two rotations compose into one turn by
 * (pos_on0 - pos_off0) * w_i, which is what the kernel applies; its cos/sin are taken
 * in double precision and the product is formed in fp32 with a split (hi + lo)
 * coefficient, so the bf16 result is within 1 bf16 ulp of the exact rotation.
 * Output is rounded to bf16 (round to nearest even).
 * ------------------------------------------------------------------------------------ */
typedef struct rk_rope_run {
  int32_t src_tab_off; /* first entry of this run's table inside src_tables */
  int32_t src_tab_len; /* entries of that table (bounds: (pos_off0+n_tok-1)/P < len) */
  int32_t dst_tab_off; /* first entry of this run's table inside dst_tables */
  int32_t dst_tab_len;
  int32_t pos_off0;    /* offline position of token 0, >= 0 */
  int32_t pos_on0;     /* online position of token 0, >= 0 */
  int32_t n_tok;       /* >= 0 */
  int32_t reserved;    /* unused, set to 0 */
} rk_rope_run;

typedef struct rk_rope_args {
  const void* k_src;          /* bf16 [n_src_pages][P][d], offline store (read only) */
  int64_t n_src_pages;
  void* k_dst;                /* bf16 [n_dst_pages][P][d], online pool (rows written) */
  int64_t n_dst_pages;
  const int32_t* src_tables;  /* int32 [n_src_entries] physical page ids */
  int64_t n_src_entries;
  const int32_t* dst_tables;  /* int32 [n_dst_entries] physical page ids */
  int64_t n_dst_entries;
  const rk_rope_run* runs;    /* [n_runs] run descriptors (device memory) */
  int32_t n_runs;
  int32_t max_tok;            /* host-known upper bound of runs[i].n_tok (sizes the grid) */
  int32_t P;                  /* tokens per page: 16 or 32 */
  int32_t d;                  /* head dim: 64 or 128 */
  double theta;               /* RoPE base, > 1 */
  int32_t style;              /* RK_ROPE_HALF_SPLIT or RK_ROPE_INTERLEAVED */
  int32_t* status;            /* optional device int32 error word, may be NULL */
} rk_rope_args;

/* Bytes of workspace rk_rope_reposition needs (per-run rotation coefficients). */
RK_API size_t rk_rope_workspace_size(int32_t n_runs, int32_t d);

/* Enqueue the repositioning of every run.  Rows of different runs must not overlap in
 * k_dst, and k_dst may alias k_src only when every token reads and writes the very same
 * row (in-place update).  Errors: RK_ERR_INVALID_ARG (NULL pointers with n_runs > 0,
 * negative sizes, theta <= 1 or not finite, k_src or k_dst not 16-byte aligned),
 * RK_ERR_UNSUPPORTED (P, d, style, or max_tok above 8388480), RK_ERR_WORKSPACE,
 * RK_ERR_CUDA.  On the device, a run with n_tok > max_tok or a negative position or table
 * offset is skipped whole; a table slot beyond its run's table or the table array, or a
 * page id outside its pool, skips the rows of that page; both set RK_ERR_DEVICE_BOUNDS.
 * A wait that exceeds its limit sets RK_ERR_TIMEOUT. */
RK_API rk_status rk_rope_reposition(const rk_rope_args* args, void* workspace, size_t workspace_bytes,
                             rk_stream_t stream);

/* Rotation coefficients for repositioning on load (rk_attn_args.k_rot): row r of `coef`
 * (device, fp32 [n][d/2][4], 16-byte aligned, caller-owned) describes the turn by deltas[r]
 * (online minus offline position, device int32 [n]): for pair i, cos and sin of
 * deltas[r] * theta^(-2i/d) in double precision, each split into a head with 16 significant
 * bits and an fp32 tail -- exactly the values rk_rope_reposition computes for a run with
 * that delta, so that rotating on load gives the same bf16 K.  Errors: RK_ERR_INVALID_ARG
 * (n < 0, NULL or misaligned pointers with n > 0, theta <= 1 or not finite),
 * RK_ERR_UNSUPPORTED (d, n > 65535), RK_ERR_CUDA. */
RK_API rk_status rk_rope_coefficients(const int32_t* deltas, int32_t n, int32_t d, double theta, void* coef,
                                      rk_stream_t stream);

/* ------------------------------------------------------------------------------------
 * SegPagedAttention
 *
 * For query token t of sequence b (position p = seq_len[b] - nq_b + i for its i-th
 * query, nq_b = cu_seqlens_q[b+1] - cu_seqlens_q[b]) and query head hq, read KV head
 * h = hq / (Hq / Hkv) of head segment s = b*Hkv + h.  Its visible keys are
 *     V = { j : logical page j / P is listed in page_logical[s][0 .. n_pages[s]),
 *               j < seq_len[b], j <= p,
 *               and, when head_class[s] == RK_CLASS_LOCAL, j > p - window[s] or j < sink[s] }
 * (global, retrieval and dense heads differ only in which pages they list).  Key j is
 * row (page_table[s][e], j % P) of k_pool / v_pool for the entry e listing page j / P.
 *     out[t][hq][:] = sum_{j in V} softmax_j(scale * q[t][hq] . k_j) v_j      (bf16)
 *     lse[t][hq]    = log sum_{j in V} exp(scale * q[t][hq] . k_j)             (fp32)
 * An empty visible set gives out = 0 and lse = -inf.  Accumulation is fp32; the
 * probabilities enter the value product as bf16.
 * ------------------------------------------------------------------------------------ */
typedef struct rk_attn_args {
  const void* q;               /* bf16 [total_q][Hq][d] */
  const int32_t* cu_seqlens_q; /* int32 [B+1], prefix sums of queries per sequence; decode: NULL (one query each) */
  const int32_t* seq_len;      /* int32 [B], context length including the queries */
  const void* k_pool;          /* bf16 [n_pool_pages][P][d] */
  const void* v_pool;          /* bf16 [n_pool_pages][P][d] */
  int64_t n_pool_pages;
  const int32_t* page_table;   /* int32 [B*Hkv][max_pages] physical page of each listed entry */
  const int32_t* page_logical; /* int32 [B*Hkv][max_pages] strictly ascending logical page of each
                                  entry, or NULL: entry e is logical page e.  The kernels find the
                                  visible entries by searching these lists, so a list that is not
                                  ascending gives an undefined visible set (reads stay inside the
                                  pools); a list whose last entry is below its first is reported
                                  as RK_ERR_DEVICE_ORDER, other violations go undetected */
  const int32_t* n_pages;      /* int32 [B*Hkv] listed entries, 0 <= n <= max_pages */
  const int32_t* head_class;   /* int32 [B*Hkv] RK_CLASS_* */
  const int32_t* window;       /* int32 [B*Hkv] local window W >= 1 (read for local heads) */
  const int32_t* sink;         /* int32 [B*Hkv] sink length S >= 0, or NULL for all zero */
  int32_t B, Hq, Hkv, d, P, max_pages;
  int32_t total_q;             /* host-known: cu_seqlens_q[B] (decode: B) */
  int32_t max_q;               /* host-known: max nq_b (decode: 1) */
  float scale;                 /* softmax scale; <= 0 selects 1/sqrt(d) */
  void* out;                   /* bf16 [total_q][Hq][d] */
  float* lse;                  /* fp32 [total_q][Hq] or NULL */
  int32_t* status;             /* optional device int32 error word, may be NULL */
  int32_t flags;               /* RK_ATTN_* bits below, 0 for none */
  const void* k_new;           /* decode only, or NULL: bf16 [B][Hkv][d], the K of the token at
                                  position seq_len[b] - 1, stored into its page slot before the
                                  keys are read (as rk_append_kv would, within the same kernel) */
  const void* v_new;           /* decode only, or NULL: bf16 [B][Hkv][d], its V; both or neither */
  const int32_t* k_rot;        /* or NULL: int32 [B*Hkv][max_pages], per listed entry the row of
                                  rot_coef whose turn is applied to that page's K rows as they are
                                  read (repositioning on load), or -1 for none */
  const void* rot_coef;        /* with k_rot: fp32 [n_rot][d/2][4] from rk_rope_coefficients, 16-byte aligned */
  int32_t n_rot;               /* with k_rot: rows of rot_coef; an entry outside [-1, n_rot) is skipped
                                  (K used unturned) and reported as RK_ERR_DEVICE_BOUNDS */
  int32_t rot_style;           /* with k_rot: RK_ROPE_HALF_SPLIT or RK_ROPE_INTERLEAVED */
} rk_attn_args;

/* Repositioning on load ("RedKnot" article, RoPE and SegPagedAttention paragraphs): with
 * k_rot, a page of a reusable segment can be listed as it was cached offline -- its K still
 * turned by the offline positions -- and the kernels turn each of its K rows by the entry's
 * coefficient row before use.  With coefficients from rk_rope_coefficients for delta = online
 * minus offline position, the K the kernels use is bit for bit the bf16 K that
 * rk_rope_reposition would have written, so the attention output is the same as repositioning
 * first; no repositioned copy is written.  All tokens of such a page must share the delta
 * (segments that start on a page boundary of both the offline and the online positions).
 * Decode only: rk_segpaged_prefill returns RK_ERR_UNSUPPORTED for a non-NULL k_rot -- a
 * prefill reads every K tile once per query tile and is bound by the tensor cores, so it
 * reads pages repositioned once by rk_rope_reposition instead; decode reads each K row once
 * and is bound by memory, so the turn costs no time there. */

/* The table and length arrays (cu_seqlens_q, seq_len, page_table, page_logical, n_pages,
 * head_class, window, sink, k_rot) were written by work that completed before the kernel
 * preceding this call on `stream` began, or by an rk_ring_advance earlier on the stream --
 * e.g. copied or advanced once at the start of a decode step, before the layers run.  The
 * decode kernel then plans its work from them while that kernel is still finishing, and
 * waits for it only before reading q and the pools and before writing.  Without the flag nothing is read before the preceding work has
 * completed.  Ignored by prefill. */
#define RK_ATTN_METADATA_STABLE 1

/* Decode, with RK_ATTN_METADATA_STABLE: the K and V pools, k_new and v_new were written by
 * work that completed before the kernel preceding this call began (earlier decode steps,
 * or other layers' pools written by the preceding kernels), and no kernel that may still
 * be running when this call starts reads the slot this call's k_new / v_new are stored
 * into.  The decode kernel then starts reading the pools while the preceding kernel is
 * still finishing; it still waits for that kernel before reading q and before writing its
 * outputs.  In a decode step where each call stores its own new token (k_new / v_new), the
 * calls of the layers after rk_ring_advance satisfy this. */
#define RK_ATTN_POOLS_STABLE 2

/* Diagnostic: a bounded wait is made to run out, and the call ends with RK_ERR_TIMEOUT in
 * the status word, the way a wait that never completes would end it, without any fault;
 * every role of the kernel leaves.  For testing that error path only.
 *  - Decode: the first CTA also waits for a word of the workspace header that nothing sets
 *    (1 s).  Zero the workspace again before its next use.
 *  - Prefill: the merge of query tiles cut into several pieces waits for one piece more
 *    than there are; it gives up 1 s after the last piece was taken (the outputs of those
 *    tiles are then undefined).  Calls without a split tile wait for nothing.  The next
 *    call needs no reset: the planner re-initialises the workspace. */
#define RK_ATTN_DIAG_EXPIRE_WAIT (1 << 30)

/* Bytes of workspace rk_segpaged_prefill / rk_segpaged_decode need for these sizes
 * (work list plus split-KV partial results).  Returns 0 for invalid sizes. */
RK_API size_t rk_segpaged_prefill_workspace_size(const rk_attn_args* args);
RK_API size_t rk_segpaged_decode_workspace_size(const rk_attn_args* args);

/* Prefill: any number of queries per sequence (a suffix at the end of the context).  A query
 * tile whose key list is cut into several pieces is merged (log-sum-exp) inside the same
 * kernel, by CTAs that have run out of pieces; a merge that waits longer than 1 s for its
 * pieces sets RK_ERR_TIMEOUT in the status word.
 * Errors: RK_ERR_INVALID_ARG (NULL pointers, k_new or v_new set, q / k_pool / v_pool / out not 16-byte aligned,
 * B/Hq/Hkv/max_pages/total_q < 0, Hq % Hkv,
 * max_q > total_q), RK_ERR_UNSUPPORTED (d, P, Hq/Hkv > 16), RK_ERR_WORKSPACE, RK_ERR_CUDA. */
RK_API rk_status rk_segpaged_prefill(const rk_attn_args* args, void* workspace, size_t workspace_bytes,
                              rk_stream_t stream);

/* Decode: one query per sequence at position seq_len[b] - 1 (q is [B][Hq][d]); split-KV
 * over each head's visible pages, partial results merged by log-sum-exp.  With k_new and
 * v_new the call first stores the new token's K and V at position seq_len[b] - 1 of every
 * head segment -- the slot of the page its list gives for that logical page, which must
 * be listed (else RK_ERR_DEVICE_BOUNDS and no store) -- so that a decode step needs no
 * separate append.  Same errors as prefill (k_new / v_new: both or neither, 16-byte
 * aligned), and RK_ERR_UNSUPPORTED when B * Hkv exceeds 16384.
 *
 * Workspace: its first 28928 bytes hold per-call split counters and flags.  They must be zero before
 * the first decode call that uses the workspace (e.g. cudaMemsetAsync of the whole
 * buffer once, after allocating it); every call returns them to zero before it completes,
 * so the workspace can be reused by any later decode call, of any shape, on the same
 * stream without clearing.  Do not use it for other calls in between.  After a call that
 * reported RK_ERR_TIMEOUT, zero it again. */
RK_API rk_status rk_segpaged_decode(const rk_attn_args* args, void* workspace, size_t workspace_bytes,
                             rk_stream_t stream);

/* Decode without a caller workspace, for callers that cannot allocate device memory:
 * plugins whose host owns all device memory and hands them no allocator, and code on a
 * latency-critical path that must not call cudaMalloc (which can synchronise the device).
 * The pages describe no such call; it is a deployment convenience of this library.
 *
 * Same arguments, computation and errors as rk_segpaged_decode; the scratch memory is a
 * fixed device array of RK_DECODE_NOALLOC_SCRATCH_BYTES inside the library (reserved on
 * every GPU that loads the library, until the process exits).  Calls whose
 * rk_segpaged_decode_workspace_size exceeds it return RK_ERR_UNSUPPORTED and enqueue
 * nothing; use rk_segpaged_decode with a workspace for those.  The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress, once per device,
 * with that device current) and enqueues the zeroing of the array's split counters on
 * `stream`, ahead of its decode; so make that first call before any stream capture.  No call
 * allocates memory.  Every call on a device shares the one array: calls that may overlap
 * on the GPU (different streams, or different host threads) race and must be serialised
 * by the caller; calls on one stream are ordered.  Every call leaves the split counters at
 * zero (after RK_ERR_TIMEOUT on the device, the array cannot be reused: the process should
 * start over). */
#define RK_DECODE_NOALLOC_SCRATCH_BYTES (16u << 20)
RK_API rk_status rk_segpaged_decode_noalloc(const rk_attn_args* args, rk_stream_t stream);

/* ------------------------------------------------------------------------------------
 * Decode-time storage: appending a step's K/V, and the page ring of local heads
 *
 * "小红书 RedKnot", section 3, first and fourth components: local heads keep only a window
 * of KV (segmented per-head storage), which is what lets more sessions share a GPU.  Pages
 * follow "PagedAttention & RadixAttention", section "The Solution: Fixed-size blocks":
 * a token at position j lives in slot j % P of the page listed for logical page j / P.
 *
 * A decode step, per layer: rk_append_kv writes the new token's K and V (or the decode call
 * does, with k_new / v_new), then rk_segpaged_decode attends to them.  Once per step, before
 * the layers, the tables of window-only local heads are advanced with rk_ring_advance.  No
 * kernel enqueued after rk_ring_advance starts before it has completed, so the decode calls
 * that follow it may pass RK_ATTN_METADATA_STABLE.
 * ------------------------------------------------------------------------------------ */
typedef struct rk_append_args {
  const void* k_new;           /* bf16 [B][Hkv][d], the new token's K per head segment */
  const void* v_new;           /* bf16 [B][Hkv][d] */
  const int32_t* pos;          /* int32 [B] position of the new token, >= 0 */
  void* k_pool;                /* bf16 [n_pool_pages][P][d] */
  void* v_pool;                /* bf16 [n_pool_pages][P][d] */
  int64_t n_pool_pages;
  const int32_t* page_table;   /* int32 [B*Hkv][max_pages], as for attention */
  const int32_t* page_logical; /* int32 [B*Hkv][max_pages] ascending, or NULL (entry e is page e) */
  const int32_t* n_pages;      /* int32 [B*Hkv] */
  int32_t B, Hkv, d, P, max_pages;
  int32_t* status;             /* optional device int32 error word, may be NULL */
} rk_append_args;

/* For every head segment s = b*Hkv + h, copy k_new[b][h] and v_new[b][h] bit for bit into
 * slot pos[b] % P of the page the list gives for logical page pos[b] / P.  The list and its
 * tables are only read.  Errors: RK_ERR_INVALID_ARG (NULL pointers with B*Hkv > 0, negative
 * sizes, a pointer of k_new / v_new / k_pool / v_pool not 16-byte aligned), RK_ERR_UNSUPPORTED
 * (d, P), RK_ERR_CUDA; on the device, a position whose page is not listed, a negative position,
 * n_pages outside [0, max_pages] or a page id outside the pool skips that head segment and sets
 * RK_ERR_DEVICE_BOUNDS. */
RK_API rk_status rk_append_kv(const rk_append_args* args, rk_stream_t stream);

typedef struct rk_ring_args {
  const int32_t* pos;          /* int32 [B] position of the token about to be appended */
  int32_t* page_table;         /* int32 [B*Hkv][max_pages], updated in place */
  int32_t* page_logical;       /* int32 [B*Hkv][max_pages] ascending, updated in place (required) */
  const int32_t* n_pages;      /* int32 [B*Hkv] (unchanged by the call) */
  const int32_t* ring;         /* int32 [B*Hkv] ring size R > 0 of a window-only local head, 0 for
                                  any other head segment (left alone) */
  const int32_t* window;       /* int32 [B*Hkv] window W of the ring heads */
  const int32_t* sink;         /* int32 [B*Hkv] sink S, or NULL for all zero */
  int32_t B, Hkv, P, max_pages;
  int32_t* status;             /* optional device int32 error word, may be NULL */
  const int32_t* src_page_table;   /* or NULL (in place): int32 [B*Hkv][max_pages], the tables to
                                      advance from; the advanced lists go to page_table */
  const int32_t* src_page_logical; /* with src_page_table: int32 [B*Hkv][max_pages]; both or neither */
} rk_ring_args;

/* Advance the page ring of every head segment with ring[s] = R > 0.  Its list is the sink
 * pages (logical pages below ceil(S/P)) followed by R window pages.  When pos[b] / P is
 * above its last logical page, the first window entry -- the oldest page, which must end at
 * or before position pos[b] - W, i.e. lie wholly outside the new token's window -- gives its
 * physical page to logical page pos[b] / P: the window entries move down by one and the new
 * page takes the last entry.  R = ceil(W/P) + 1 window pages ending at the page before
 * pos[b] / P always satisfy this.  Several layers can be advanced in one call by laying
 * their tables out as extra sequences.  Errors: RK_ERR_INVALID_ARG (NULL pointers with
 * B*Hkv > 0, negative sizes), RK_ERR_UNSUPPORTED (P), RK_ERR_CUDA; on the device, a ring
 * that is not full or whose oldest page is still inside the window, or n_pages outside
 * [1, max_pages], leaves that head segment unchanged and sets RK_ERR_DEVICE_BOUNDS.
 *
 * Out of place (src_page_table / src_page_logical given): entries [0, n_pages) of every ring
 * head's row are read from the source tables and written, advanced (or unchanged), to
 * page_table / page_logical; rows of other head segments are neither read nor written, so
 * both copies must hold them.  Source and destination must not overlap.  The call then lets
 * the kernels after it start before it completes (programmatic dependent launch) and waits
 * for the kernels before it only before it writes.  This serves double-buffered decode
 * steps: before step s, advance step s's tables into the other buffer for step s + 1, then
 * run step s's decode calls on step s's buffer.  The decode calls of step s + 1 may then
 * pass RK_ATTN_METADATA_STABLE: each decode CTA holds a whole SM and waits for the kernel
 * before it before it exits, so a kernel enqueued before the previous decode call's
 * predecessor has completed whenever a decode call begins. */
RK_API rk_status rk_ring_advance(const rk_ring_args* args, rk_stream_t stream);

/* ------------------------------------------------------------------------------------
 * Token-level sparse FFN
 *
 * "小红书 RedKnot", section 3, third component (elastic / sparse FFN): the tokens are ranked
 * by their attention importance and only the `keep` most important go through the
 * feed-forward network; the others skip it (their FFN output is zero, so a residual add
 * leaves them as they were).  The FFN is the gated form of the Qwen / Llama models the
 * pages evaluate:  FFN(x) = W_down (silu(W_gate x) * (W_up x)),  silu(g) = g / (1 + e^-g).
 *
 *   kept = the `keep` tokens with the largest importance (equal scores: the lower token
 *          index first; NaN ranks below every number), in ascending token order
 *   out[t][:] = FFN(x[t])  for t in kept,   0 otherwise                            (bf16)
 * Accumulation is fp32; the gated activation is rounded to bf16 before W_down.
 * ------------------------------------------------------------------------------------ */
typedef struct rk_sparse_ffn_args {
  const void* x;             /* bf16 [T][d_model] */
  const float* importance;   /* fp32 [T] */
  int32_t T, d_model, d_ff;
  int32_t keep;              /* tokens that go through the FFN, 0 <= keep <= T */
  const void* w_gate;        /* bf16 [d_ff][d_model] */
  const void* w_up;          /* bf16 [d_ff][d_model] */
  const void* w_down;        /* bf16 [d_model][d_ff] */
  void* out;                 /* bf16 [T][d_model], written whole */
  int32_t* kept;             /* int32 [keep], written */
  int32_t* status;           /* optional device int32 error word, may be NULL */
} rk_sparse_ffn_args;

/* Workspace bytes: the gathered rows and the activation ([keep][d_model] + [keep][d_ff] bf16),
 * then fp32 sums of output tiles (128 x 256, at most one per SM of the current device) for
 * the down projection, which splits an incomplete last wave of output tiles along K, and
 * their tickets.  The pieces of a split tile are added with atomic additions, so the bf16
 * rounding of those rows may differ by one unit between calls.  Query the size on the
 * device the call will run on. */
RK_API size_t rk_sparse_ffn_workspace_size(const rk_sparse_ffn_args* args);

/* Errors: RK_ERR_INVALID_ARG (NULL pointers, sizes out of range, pointers not 16-byte
 * aligned), RK_ERR_UNSUPPORTED (d_model not a multiple of 256, d_ff not a multiple of 128,
 * T above 65536), RK_ERR_WORKSPACE, RK_ERR_CUDA; a wait that exceeds its limit sets
 * RK_ERR_TIMEOUT in *status. */
RK_API rk_status rk_sparse_ffn(const rk_sparse_ffn_args* args, void* workspace, size_t workspace_bytes,
                               rk_stream_t stream);

/* Static text for a status code. */
RK_API const char* rk_status_string(rk_status status);

/* Library version as major*10000 + minor*100 + patch. */
RK_API int32_t rk_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RK_API_H */
