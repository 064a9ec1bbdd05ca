/*
 * pg.h -- C ABI of the GB300 paged two-family QKV prep + paged attention library.
 *
 * Sources of the operations (three pages of one inference-engine project):
 *   [P1] "feat(kernels): Rust wrapper for the hd256 windowed paged prefill", Description
 *        and Verification: plan-driven paged prefill attention, explicit sm_scale,
 *        inclusive-distance window_left, checked geometry, checked i32 narrowing, plan
 *        bounds compared with the pool before every launch, and the reject list.
 *   [P2] "gemma4: serving prep needs pool-write forms", Description and Proposed Plan:
 *        the fused norm + rotary + paged-scatter prep for head_dim 256 (Q, K, V) and
 *        head_dim 512 (V is the weightless norm of the same raw K), the checked-geometry
 *        helper, and the slot contract slot = start_pos + token.
 *   [P3] "feat(gemma4): paged KV serving across both attention families", Description
 *        and review findings: one pool per family (hd256 local, 8 KV heads, sliding
 *        window; hd512 global, 1 KV head, full attention), decode through the prefill
 *        entry at one token, and the rule that work is bound to one stream.
 *
 * Conventions for every entry point:
 *   - Device pointers are plain CUDA device addresses owned by the caller; host
 *     pointers (plan inputs) are read during the call only.
 *   - bf16 tensors are IEEE bfloat16 bit patterns (pg_bf16_t); float tensors are fp32.
 *   - Calls are asynchronous on `stream`. The returned status covers the host-side
 *     checks and the launch only. On any nonzero status nothing was launched and no
 *     caller memory was written.
 *   - Element strides and offsets are in elements, not bytes.
 */
#ifndef PG_H_
#define PG_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t pg_bf16_t;               /* IEEE bfloat16 bit pattern          */
typedef struct CUstream_st* pg_stream_t;  /* same type as cudaStream_t          */
typedef struct pg_plan* pg_plan_t;        /* opaque; see pg_plan_paged_prefill  */

/* ---------------------------------------------------------------- status codes */
enum {
  PG_OK = 0,
  PG_ERR_ARG = -1,            /* null pointer, negative count, non-monotone indptr, zero-length request */
  PG_ERR_PAGE_OOB = -2,       /* a page id outside [0, num_pages) of the pool ([P1] Verification) */
  PG_ERR_LAST_PAGE_LEN = -3,  /* last_page_len outside [1, page_size] ([P1] Verification)        */
  PG_ERR_I32_OVERFLOW = -4,   /* a length / indptr / offset past int32, or a stride product past int64 */
  PG_ERR_ZERO_KV_HEADS = -5,  /* num_kv_heads == 0, caught before any division ([P1] Description) */
  PG_ERR_HEADS = -6,          /* num_qo_heads <= 0, num_kv_heads < 0 or num_qo_heads % num_kv_heads != 0 */
  PG_ERR_NONFINITE = -7,      /* sm_scale or eps not finite, or eps <= 0, or theta <= 0        */
  PG_ERR_ROPE_RANGE = -8,     /* a query position at or past rope_rows ([P2] Proposed Plan)   */
  PG_ERR_COVERAGE = -9,       /* pages do not cover exactly [0, start_pos + qo_len) (ring: the window plus the step) */
  PG_ERR_LAYER = -10,         /* layer outside [0, num_layers)                                 */
  PG_ERR_LAYOUT = -11,        /* pool strides / capacity / head geometry inconsistent          */
  PG_ERR_PLAN_MISMATCH = -12, /* plan heads, head_dim, page_size or cta_tile_q disagree        */
  PG_ERR_WINDOW = -13,        /* window_left < -1, or outside [0, plan window] on a ring plan  */
  PG_ERR_WORKSPACE = -14,     /* workspace null or smaller than pg_workspace_bytes             */
  PG_ERR_STREAM = -15,        /* call stream differs from the plan's stream ([P3] review)      */
  PG_ERR_CUDA = -16,          /* a CUDA runtime call failed                                    */
  PG_ERR_DEVICE_BOUNDS = -17, /* a kernel saw out-of-range metadata and skipped the access     */
  PG_ERR_ALIGN = -18,         /* a device pointer or token stride breaks its stated alignment  */
  PG_ERR_DEVICE_TIMEOUT = -19 /* a kernel's bounded wait ran out; its outputs are not valid    */
};

/* ---------------------------------------------------------------- pool descriptor */
/*
 * One family's paged K/V pool. Layout (fixed, checked): bf16 elements
 *   pool[layer][page][kv][kv_head][slot][d],  kv = 0 for K, 1 for V,
 * so one head row of one slot is head_dim contiguous elements. The strides must
 * equal the dense ones re-derived from the geometry with overflow-checked products:
 *   stride_slot = head_dim, stride_head = page_size*head_dim,
 *   stride_kv = num_kv_heads*stride_head, stride_page = 2*stride_kv,
 *   stride_layer = num_pages*stride_page,
 * and capacity (elements in the caller's buffer) must equal num_layers*stride_layer
 * (a whole number of pages per layer). base must be 16-byte aligned.
 */
typedef struct {
  pg_bf16_t* base;
  int32_t num_layers, num_pages, page_size, num_kv_heads, head_dim;
  int64_t stride_layer, stride_page, stride_kv, stride_head, stride_slot;
  int64_t capacity;
} pg_pool_t;

/* ---------------------------------------------------------------- plan */
/*
 * pg_plan_paged_prefill -- build (*plan == NULL) or update in place (*plan != NULL)
 * the ragged batch plan that prep and attention consume ([P1] Description:
 * PrefillPagedPlan; [P3] Description: both families' plans are built over the same
 * token span).
 *
 * Inputs (host memory, read during the call):
 *   qo_indptr[num_req+1]       int64, qo_indptr[0] == 0, strictly increasing (every
 *                              request has >= 1 query token); tokens of request r are
 *                              rows qo_indptr[r] .. qo_indptr[r+1]-1 of q/k/v/out.
 *   kv_page_indptr[num_req+1]  int64, kv_page_indptr[0] == 0, strictly increasing.
 *   page_ids[kv_page_indptr[num_req]]  int32 physical page ids, >= 0.
 *   last_page_len[num_req]     int32 in [1, page_size].
 *   start_pos[num_req]         int64 >= 0: position of the request's first new token.
 * Coverage: (pages_r - 1) * page_size + last_page_len_r must equal
 * start_pos_r + qo_len_r, i.e. the pages hold exactly KV positions [0, kv_len_r).
 * The token at row qo_indptr[r] + t has position start_pos_r + t and writes KV slot
 * start_pos_r + t ([P2] Proposed Plan, slot contract).
 *
 * The head relation is settled before anything divides: num_kv_heads == 0 fails with
 * PG_ERR_ZERO_KV_HEADS. Every length narrowed to int32 is checked (PG_ERR_I32_OVERFLOW).
 * The plan records the largest page id and largest last_page_len from its host inputs;
 * prep and attention compare them with the pool before every launch.
 *
 * Device metadata is uploaded on `stream`; the plan is bound to that stream and later
 * calls on another stream fail with PG_ERR_STREAM. An update checks every input on the
 * host before anything changes: on any error the plan is left exactly as it was. The
 * metadata then goes through a pinned host staging buffer of the plan (the call does not
 * wait for the stream) into the plan's device storage, in place when it is large enough
 * (ordered after every call already queued on the stream, which read the old metadata;
 * a CUDA graph that captured the plan's calls reads the new), else into fresh storage that
 * replaces the old. num_req == 0 is a valid empty plan (calls launch nothing).
 */
int pg_plan_paged_prefill(pg_plan_t* plan, int32_t num_req, const int64_t* qo_indptr,
                          const int64_t* kv_page_indptr, const int32_t* page_ids,
                          const int32_t* last_page_len, const int64_t* start_pos,
                          int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                          int32_t page_size, pg_stream_t stream);

/*
 * pg_plan_paged_prefill_ring -- the same plan for window-crossing requests, with ring
 * slot addressing ([P2] Proposed Plan: slots equal positions only below the sliding
 * window, and callers that cross it need a separate slot mapping). Request r holds
 * pages_r = kv_page_indptr[r+1] - kv_page_indptr[r] pages as a ring: position p lives
 * in page page_ids[kv_page_indptr[r] + (p / page_size) mod pages_r], slot
 * p mod page_size. Prep writes the step's K/V there; attention reads keys
 * [max(0, p - window_left), p] of each query position p from the same slots.
 *
 * Inputs as for pg_plan_paged_prefill, without last_page_len (the ring has no last page):
 *   window_left  >= 0: the largest window attention may run with on this plan.
 * Coverage: pages_r * page_size >= window_left + qo_len_r, or no position has wrapped yet
 * (start_pos_r + qo_len_r <= pages_r * page_size), for every request, so no key that a
 * query of the step can see is overwritten by the step's own writes (PG_ERR_COVERAGE
 * otherwise); window_left < 0 fails with PG_ERR_WINDOW. A ring may so grow page by page
 * while the request is shorter than it. A request may
 * start at any position (start_pos is not bounded by its pages), and all positions
 * below start_pos_r must have been written through the same ring by earlier steps.
 * Attention on a ring plan requires 0 <= window_left <= the plan's window
 * (PG_ERR_WINDOW otherwise). Everything else (stream binding, in-place update, checks)
 * is as for pg_plan_paged_prefill.
 */
int pg_plan_paged_prefill_ring(pg_plan_t* plan, int32_t num_req, const int64_t* qo_indptr,
                               const int64_t* kv_page_indptr, const int32_t* page_ids,
                               const int64_t* start_pos, int32_t num_qo_heads,
                               int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                               int32_t window_left, pg_stream_t stream);

/*
 * pg_plan_paged_segment -- a plan over key segments, for cascade attention: requests that
 * share a key prefix attend to it once as one segment and to their own keys as another,
 * and pg_merge_attn_states combines the two results. (A variant the pages leave open:
 * attention over a request's keys is the softmax of [P1] Description; splitting the keys
 * into disjoint segments and merging by the softmax normalisers is exact.)
 *
 * Inputs as for pg_plan_paged_prefill, plus
 *   kv_start[num_req]  int64 >= 0: request r's pages hold key positions
 *                      [kv_start_r, kv_start_r + n_r), n_r = (pages_r - 1) * page_size
 *                      + last_page_len_r, position kv_start_r + i in slot i (page
 *                      i / page_size, offset i mod page_size) of its pages.
 * Coverage: kv_start_r + n_r <= start_pos_r + qo_len_r (a segment holds no key past the
 * step's last query; PG_ERR_COVERAGE otherwise). Queries see the keys of the segment
 * that the causal and window rules allow: keys before kv_start_r are not part of this
 * plan, and a query row that sees no key gets out = 0 and lse = -inf. Prep on a segment
 * plan is accepted only when every request's step tokens are its segment's tail
 * (kv_start_r <= start_pos_r and kv_start_r + n_r == start_pos_r + qo_len_r; prep calls
 * fail with PG_ERR_COVERAGE otherwise); the pool pages may repeat across requests (a
 * shared prefix lists the same pages for every request) as long as no prep writes them.
 * Everything else (stream binding, in-place update, checks) is as for
 * pg_plan_paged_prefill; kv_start == 0 for every request gives that plan.
 */
int pg_plan_paged_segment(pg_plan_t* plan, int32_t num_req, const int64_t* qo_indptr,
                          const int64_t* kv_page_indptr, const int32_t* page_ids,
                          const int32_t* last_page_len, const int64_t* kv_start,
                          const int64_t* start_pos, int32_t num_qo_heads, int32_t num_kv_heads,
                          int32_t head_dim, int32_t page_size, pg_stream_t stream);

/* Free a plan (host and device storage; device frees are ordered on its stream). NULL is a no-op. */
void pg_plan_destroy(pg_plan_t plan);

typedef struct {
  int32_t num_req, num_tokens, num_qo_heads, num_kv_heads, head_dim, page_size;
  int32_t max_page_id, max_last_page_len, max_qo_len, max_kv_len, max_pos_end;
  int32_t cta_tile_q;       /* query tokens per attention CTA the plan was tiled with */
  int32_t decode;           /* 1 when every request has exactly one query token       */
  int32_t kv_chunk;         /* keys per split-KV chunk (decode form)                  */
  int32_t max_chunks;       /* chunks per request the workspace is sized for           */
  int32_t num_work;         /* prefill work items (request, query tile)                */
  const int32_t* d_page_ids;/* device copy of page_ids (for diagnostics)              */
  pg_stream_t stream;
  int64_t metadata_bytes;   /* bytes of device metadata each build or update uploads  */
} pg_plan_info_t;

/* Copy the plan's recorded geometry and bounds into *info. */
int pg_plan_info(const pg_plan_t plan, pg_plan_info_t* info);

/* ---------------------------------------------------------------- rotary tables */
/*
 * Fill rope_cos / rope_sin (device, fp32, [rows, head_dim/2] each, row-major) with
 * cos and sin of pos * theta^(-2i/head_dim), evaluated in fp64 and rounded to fp32.
 * Element i of a row rotates the pair (i, i + head_dim/2) (half-split pairing).
 * Any stream. Errors: PG_ERR_ARG (null, rows < 1, odd head_dim), PG_ERR_NONFINITE.
 */
int pg_rope_table(float* rope_cos, float* rope_sin, int32_t rows, int32_t head_dim,
                  double theta, pg_stream_t stream);

/* ---------------------------------------------------------------- prep */
/*
 * pg_prep_paged_hd256 -- fused prep for the head_dim-256 family ([P2] Proposed Plan,
 * first item). For every token row t (position p = start_pos_r + t) and head h:
 *   q_out[t][h]           = rope_p( q_raw[t][h] * inv_rms(q_raw[t][h]) * w_q )
 *   K slot (layer, p)[g]  = rope_p( k_raw[t][g] * inv_rms(k_raw[t][g]) * w_k )
 *   V slot (layer, p)[g]  =         v_raw[t][g] * inv_rms(v_raw[t][g])        (never rotated)
 * with inv_rms(x) = 1/sqrt(mean(x^2) + eps), rope_p the half-split rotation by the
 * rope table row p, all in fp32 with one bf16 round-to-nearest-even at the store.
 * The K/V slot of position p is page page_ids[kv_page_indptr[r] + p / page_size],
 * slot p % page_size of `layer` in `pool`.
 *
 *   q_raw  [T][Hq][256]  bf16, token stride q_tok_stride (>= Hq*256, multiple of 8)
 *   k_raw, v_raw [T][Hkv][256] bf16, token strides k_tok_stride / v_tok_stride
 *   w_q, w_k [256] bf16; rope_cos/rope_sin [rope_rows][128] fp32 (see pg_rope_table)
 *   q_out  [T][Hq][256] bf16 contiguous (written)
 * Only the K/V rows of the plan's positions in `layer` are written; every other pool
 * byte is left untouched. Checks (before launch): plan/pool geometry and strides,
 * layer, plan page bounds vs pool, rope range (max position < rope_rows), eps finite
 * and > 0, 16-byte alignment, stream. Kernel-side second layer: a position or page
 * id out of range sets the device status word (pg_device_status) and the row is
 * skipped; the kernel never traps.
 */
int pg_prep_paged_hd256(const pg_plan_t plan, const pg_pool_t* pool, int32_t layer,
                        const pg_bf16_t* q_raw, int64_t q_tok_stride,
                        const pg_bf16_t* k_raw, int64_t k_tok_stride,
                        const pg_bf16_t* v_raw, int64_t v_tok_stride,
                        const pg_bf16_t* w_q, const pg_bf16_t* w_k, float eps,
                        const float* rope_cos, const float* rope_sin, int32_t rope_rows,
                        pg_bf16_t* q_out, pg_stream_t stream);

/*
 * pg_prep_paged_hd512 -- fused prep for the head_dim-512 family ([P2] Description and
 * Proposed Plan, second item). Q and K as in the hd256 form (head_dim 512, rope table
 * [rope_rows][256]); the V row is the weightless norm of the SAME raw K row, sharing
 * K's inverse RMS and never rotated: V = k_raw * inv_rms(k_raw). There is no v input.
 * Same checks, ownership and error behaviour as pg_prep_paged_hd256.
 */
int pg_prep_paged_hd512(const pg_plan_t plan, const pg_pool_t* pool, int32_t layer,
                        const pg_bf16_t* q_raw, int64_t q_tok_stride,
                        const pg_bf16_t* k_raw, int64_t k_tok_stride,
                        const pg_bf16_t* w_q, const pg_bf16_t* w_k, float eps,
                        const float* rope_cos, const float* rope_sin, int32_t rope_rows,
                        pg_bf16_t* q_out, pg_stream_t stream);

/* ---------------------------------------------------------------- attention */
/*
 * Bytes of device workspace pg_attn_* needs for this plan (0 when none). The decode
 * form (every qo_len == 1) splits each request's keys into chunks and needs room for
 * per-chunk partial outputs; prefill needs none.
 */
size_t pg_workspace_bytes(const pg_plan_t plan);

/*
 * pg_attn_paged_prefill -- paged prefill attention for the head_dim-256 family
 * ([P1] Description; [P3] Description: decode is this entry at one token).
 * For query row (t, h) of request r at position p = start_pos_r + t:
 *   out[t][h] = sum_j softmax_j( sm_scale * <q[t][h], K_j> ) V_j
 * over keys j in [0, kv_len_r) with j <= p and (window_left < 0 or p - j <= window_left)
 * (inclusive distance: window_left + 1 keys), K_j / V_j read from pool `layer` through
 * the page table, KV head h / (Hq / Hkv). fp32 softmax, bf16 output (RNE).
 *   q   [T][Hq][256] bf16 contiguous, 32-byte aligned (the prep's q_out)
 *   out [T][Hq][256] bf16 contiguous, 32-byte aligned (written)
 *   workspace: device scratch of ws_bytes >= pg_workspace_bytes(plan) (may be NULL when 0)
 * Checks (before launch): plan head_dim 256 and tile derivation, pool geometry, layer,
 * plan page bounds vs pool, window_left >= -1, sm_scale finite, workspace, alignment,
 * stream. sm_scale is model policy and is never derived from head_dim.
 */
int pg_attn_paged_prefill(const pg_plan_t plan, const pg_pool_t* pool, int32_t layer,
                          const pg_bf16_t* q, pg_bf16_t* out, int32_t window_left,
                          float sm_scale, void* workspace, size_t ws_bytes,
                          pg_stream_t stream);

/* Same as pg_attn_paged_prefill for the head_dim-512 family (1 KV head in the pages'
 * geometry; any Hq % Hkv == 0 with Hq / Hkv <= 16 is accepted). Full causal attention
 * is window_left = -1. */
int pg_attn_paged_prefill_hd512(const pg_plan_t plan, const pg_pool_t* pool, int32_t layer,
                                const pg_bf16_t* q, pg_bf16_t* out, int32_t window_left,
                                float sm_scale, void* workspace, size_t ws_bytes,
                                pg_stream_t stream);

/*
 * pg_attn_paged_prefill_lse / pg_attn_paged_prefill_hd512_lse -- the same attention,
 * also writing each row's softmax normaliser
 *   lse[t][h] = log( sum_j exp( sm_scale * <q[t][h], K_j> ) )   (natural log)
 * over the keys the row sees, or -inf when it sees none (its out row is then 0).
 *   lse [T][Hq] float32, 4-byte aligned, written (must not be NULL when T > 0:
 *       PG_ERR_ARG)
 * The kernels sum the bf16-rounded softmax weights they multiply V by, so lse agrees with
 * out's normalisation. Every other argument, check and error as for the entries above.
 */
int pg_attn_paged_prefill_lse(const pg_plan_t plan, const pg_pool_t* pool, int32_t layer,
                              const pg_bf16_t* q, pg_bf16_t* out, float* lse,
                              int32_t window_left, float sm_scale, void* workspace,
                              size_t ws_bytes, pg_stream_t stream);
int pg_attn_paged_prefill_hd512_lse(const pg_plan_t plan, const pg_pool_t* pool, int32_t layer,
                                    const pg_bf16_t* q, pg_bf16_t* out, float* lse,
                                    int32_t window_left, float sm_scale, void* workspace,
                                    size_t ws_bytes, pg_stream_t stream);

/*
 * pg_merge_attn_states -- combine two attention states over disjoint key sets, row by row:
 * with w_x = exp(lse_x - M), M = max(lse_a, lse_b),
 *   out = (w_a out_a + w_b out_b) / (w_a + w_b),   lse = M + log(w_a + w_b);
 * a side with lse = -inf contributes nothing (both -inf: out = 0, lse = -inf).
 *   out_a, out_b, out  [rows][head_dim] bf16, 16-byte aligned (out may alias either input)
 *   lse_a, lse_b       [rows] float32; lse [rows] float32 or NULL (not written)
 * head_dim > 0 and a multiple of 8; rows >= 0 (0 launches nothing), rows <= INT32_MAX.
 * Errors: PG_ERR_ARG (null input, bad sizes), PG_ERR_ALIGN, PG_ERR_I32_OVERFLOW,
 * PG_ERR_CUDA. Asynchronous on `stream`; no plan is involved.
 */
int pg_merge_attn_states(const pg_bf16_t* out_a, const float* lse_a, const pg_bf16_t* out_b,
                         const float* lse_b, pg_bf16_t* out, float* lse, int64_t rows,
                         int32_t head_dim, pg_stream_t stream);

/* ---------------------------------------------------------------- decode without allocation */
/*
 * Bytes of library-owned device scratch behind pg_attn_paged_decode_noalloc. The buffer is a
 * static device array of this size in the library image: every GPU that loads the library
 * holds it from first use until the process exits.
 */
#define PG_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

/*
 * pg_attn_paged_decode_noalloc -- the decode form of paged attention (a plan whose requests
 * each have exactly one query token, head_dim 256 or 512) with its split-KV partials kept in
 * the library's static scratch instead of a caller workspace. The pages have no counterpart
 * for this entry: it exists for callers that cannot allocate device memory at call time
 * (for example code running under an allocator that forbids cudaMalloc once serving has
 * started, or a host runtime that owns all device memory and hands out only the tensors it
 * manages). It computes exactly what pg_attn_paged_prefill / pg_attn_paged_prefill_hd512
 * compute for the same decode plan and arguments, with the same checks and status codes.
 *
 * The call allocates nothing. On the first call on a device it looks up the device address
 * of the static scratch (cudaGetSymbolAddress, with that device current); make that first
 * call before any stream capture. Every call on a device shares the one scratch buffer and
 * overwrites it: calls whose kernels overlap on the GPU (different streams, or several
 * plans in flight at once) race on it, so serialise them. Nothing in the scratch needs to
 * start at zero: each partial result the merge step reads is written by the same call.
 *
 * Errors: as pg_attn_paged_prefill, plus PG_ERR_PLAN_MISMATCH for a plan that is not a
 * decode plan, PG_ERR_WORKSPACE when pg_workspace_bytes(plan) exceeds
 * PG_NOALLOC_SCRATCH_BYTES, and PG_ERR_STREAM when the current device is not the plan's.
 */
int pg_attn_paged_decode_noalloc(const pg_plan_t plan, const pg_pool_t* pool, int32_t layer,
                                 const pg_bf16_t* q, pg_bf16_t* out, int32_t window_left,
                                 float sm_scale, pg_stream_t stream);

/* ---------------------------------------------------------------- diagnostics */
/* Synchronise `stream`, then read and clear the current device's status word.
 * Returns PG_OK, PG_ERR_DEVICE_BOUNDS (a kernel skipped an out-of-range access),
 * PG_ERR_DEVICE_TIMEOUT (a kernel gave up a bounded wait), or PG_ERR_CUDA. */
int pg_device_status(pg_stream_t stream);

/* Kernels this library has launched since it was loaded (all devices). */
int64_t pg_launch_count(void);

/*
 * Test hook for the kernels' bounded waits (failure detection without a GPU fault). With
 * withhold = 1, every later prefill attention launch on the tensor-core path has the leading
 * CTA of each pair skip the first key-tile arrival it owes (no copy is issued for that tile),
 * and every bounded wait of those launches gives up after wait_limit_ns (in [1e6, 2e9]): the
 * call's kernels then return with PG_ERR_DEVICE_TIMEOUT in the status word
 * (pg_device_status) and their outputs are not valid; the context stays usable. withhold = 0
 * restores normal launches and the two-second limit (wait_limit_ns is ignored). Process-wide;
 * not for use while other threads launch. Errors: PG_ERR_ARG.
 */
int pg_test_bounded_wait(int32_t withhold, int64_t wait_limit_ns);

/* Static text for a status code. */
const char* pg_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif /* PG_H_ */
