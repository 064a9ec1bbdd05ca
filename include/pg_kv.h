/*
 * pg_kv.h -- host-side page accounting for two-family paged KV serving.
 *
 * Source: "feat(gemma4): paged KV serving across both attention families", Description: one
 * pool per attention family (hd256 local layers with a sliding window, hd512 global layers),
 * a per-request state in each, admission that is atomic across both pools with the page
 * count as the exact frontier account, nothing changing state before a step is admissible,
 * page ids meaningful only against the pool that issued them, and the path failing closed
 * at the sliding window (cache slots equal positions only below it). Verification: a forced
 * partial failure leaves both pools at their pre-request occupancy. Review finding "Commit KV
 * frontiers only after a successful step": admission only reserves; the frontier moves when
 * the caller commits the step after its plan, copies and launches succeeded, and a step that
 * failed anywhere after admission is aborted, returning its pages with the frontier unchanged,
 * so a retry of the same step writes the same positions.
 *
 * Step life cycle per request: pg_kv_admit_step (pages reserved, step pending) ->
 * pg_kv_batch_plan_inputs (plan inputs covering the pending step) -> prep / attention ->
 * pg_kv_commit_step on success, or pg_kv_abort_step on any failure. A request holds at most
 * one pending step.
 *
 * This is host code only (no CUDA calls, no device memory). A server owns two page
 * allocators, one per family; each request holds a state in both: its page list and its
 * frontier (the number of KV positions committed, the same in both families). The page lists
 * feed pg_plan_paged_prefill's kv_page_indptr / page_ids / last_page_len / start_pos; a ring
 * server (pg_kv_server_create_ring) keeps the local family on a ring of pages past the window
 * instead of failing closed, for pg_plan_paged_prefill_ring.
 *
 * Errors: int status, PG_KV_OK = 0, negative = error. On any error no state changes: both
 * pools keep their occupancy and every request keeps its pages and frontier.
 * Not thread-safe: one server is driven by one thread (the serving loop's step boundary).
 */
#ifndef PG_KV_H_
#define PG_KV_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pg_kv_server* pg_kv_server_t;  /* opaque; owns both pools' allocators */

enum {
  PG_KV_OK = 0,
  PG_KV_ERR_ARG = -101,       /* null pointer, non-positive size, unknown family            */
  PG_KV_ERR_NO_PAGES = -102,  /* a family's pool cannot cover the step (admission refused)   */
  PG_KV_ERR_WINDOW = -103,    /* the step would carry the local family past its window      */
  PG_KV_ERR_ROPE = -104,      /* the step's last position is at or past the rotary tables   */
  PG_KV_ERR_FOREIGN = -105,   /* the request id was not issued by this server, or is closed  */
  PG_KV_ERR_FRONTIER = -106,  /* a request's families disagree on the frontier, or a family
                                 holds other than the pages its frontier accounts for        */
  PG_KV_ERR_CAPACITY = -107,  /* a caller buffer is too small                                */
  PG_KV_ERR_PENDING = -108    /* admit with a step already pending, or commit / abort / plan
                                 inputs with no step pending                                 */
};

enum { PG_KV_LOCAL = 0, PG_KV_GLOBAL = 1 };  /* the two families: hd256 local, hd512 global */

/* Create a server with `pages_local` / `pages_global` pages of `page_size` slots in the two
 * pools. window_left (>= 0, the local family's inclusive window) and fail_closed_at_window: when
 * nonzero, a step whose KV length would exceed window_left + 1 positions is refused
 * (PG_KV_ERR_WINDOW), because beyond the window cache slots would have to stop equalling
 * positions. rope_rows: positions must stay below it. Pages are issued lowest id first. */
int pg_kv_server_create(pg_kv_server_t* out, int32_t pages_local, int32_t pages_global,
                        int32_t page_size, int32_t window_left, int32_t fail_closed_at_window,
                        int32_t rope_rows);
/* A server whose local family keeps a ring of pages instead of failing closed at the window
 * ("gemma4: serving prep needs pool-write forms", Proposed Plan: callers that cross the
 * window need a separate slot mapping; the mapping is pg_plan_paged_prefill_ring's). Each
 * request's local family holds at most ring = ceil((window_left + ring_max_step) / page_size)
 * pages: ceil(frontier / page_size) while that is smaller, then the same ring pages, reused.
 * Steps are at most ring_max_step (>= 1) tokens (PG_KV_ERR_WINDOW otherwise, nothing
 * changed); the global family grows with the frontier as in pg_kv_server_create. The local
 * family's batch plan inputs feed pg_plan_paged_prefill_ring with window_left (its
 * last_page_len output is not read there). Other arguments and errors as pg_kv_server_create. */
int pg_kv_server_create_ring(pg_kv_server_t* out, int32_t pages_local, int32_t pages_global,
                             int32_t page_size, int32_t window_left, int32_t ring_max_step,
                             int32_t rope_rows);
void pg_kv_server_destroy(pg_kv_server_t srv);

/* Open a request (frontier 0, no pages) and return its id (> 0, never reused by this server). */
int pg_kv_request_open(pg_kv_server_t srv, int64_t* request_id);

/* Close a request: its pages return to both pools. PG_KV_ERR_FOREIGN for an unknown id. */
int pg_kv_request_close(pg_kv_server_t srv, int64_t request_id);

/* Admit one step of `n_tokens` (>= 1) new positions for a request, in both families at once.
 * The page count per family is the exact frontier account: ceil((frontier + n_tokens) /
 * page_size) (capped at the ring for the local family of a ring server) minus the pages the
 * family already holds. Before anything changes, the request
 * must belong to this server, have no step pending (PG_KV_ERR_PENDING), both families must
 * sit at the same frontier and hold exactly the pages it accounts for, and the window and
 * rotary bounds must hold. Then both families' pages are reserved; if either pool refuses, the
 * other reservation is dropped and PG_KV_ERR_NO_PAGES returned, with both pools at their
 * pre-request occupancy. When both reservations stand, the request holds them and the step is
 * pending: the frontier does not move until pg_kv_commit_step. */
int pg_kv_admit_step(pg_kv_server_t srv, int64_t request_id, int32_t n_tokens);

/* Commit the request's pending step once its plan, copies and launches have all succeeded:
 * the frontier advances by the step's tokens in both families. PG_KV_ERR_PENDING when no
 * step is pending; nothing changes on any error. */
int pg_kv_commit_step(pg_kv_server_t srv, int64_t request_id);

/* Abort the request's pending step (plan building, a copy, a launch or the step's tail failed
 * after admission): the pages the step reserved return to both pools and the frontier stays,
 * so the request is exactly as before pg_kv_admit_step and the step can be admitted again.
 * Positions the failed step may already have written past the frontier are rewritten by the
 * retry before any query reads them. PG_KV_ERR_PENDING when no step is pending. */
int pg_kv_abort_step(pg_kv_server_t srv, int64_t request_id);

/* Tokens of the request's pending step (0: none). */
int pg_kv_request_pending(pg_kv_server_t srv, int64_t request_id, int32_t* pending);

/* A request's frontier (positions committed) and, per family, its page count (a pending
 * step's pages included). */
int pg_kv_request_info(pg_kv_server_t srv, int64_t request_id, int32_t* frontier,
                       int32_t* pages_local, int32_t* pages_global);

/* Copy a request's page ids in one family (in position order) into out[0, cap);
 * *n receives the count. PG_KV_ERR_CAPACITY if cap is too small (nothing written). */
int pg_kv_request_pages(pg_kv_server_t srv, int64_t request_id, int32_t family, int32_t* out,
                        int32_t cap, int32_t* n);

/* Free pages in a family's pool. */
int pg_kv_free_pages(pg_kv_server_t srv, int32_t family, int32_t* n);

/* Test hook (the forced partial failure of the pages' verification): the next `count`
 * reservations in `family` are refused as if that pool were full. */
int pg_kv_inject_refusal(pg_kv_server_t srv, int32_t family, int32_t count);

/* Plan inputs of a batch for one family, covering each request's pending step of
 * step_tokens[i] tokens (which must equal the pending count: PG_KV_ERR_ARG otherwise;
 * PG_KV_ERR_PENDING when a request has no step pending): kv_page_indptr [n + 1], page_ids
 * (cap entries, in position order, or ring order for a ring server's local family),
 * last_page_len [n] (slots used in the page of the step's last position), start_pos [n]
 * (= the committed frontier), in the layout pg_plan_paged_prefill reads. *n_page_ids
 * receives the page-id count. */
int pg_kv_batch_plan_inputs(pg_kv_server_t srv, int32_t family, int32_t n,
                            const int64_t* request_ids, const int32_t* step_tokens,
                            int64_t* kv_page_indptr, int32_t* page_ids, int32_t cap,
                            int32_t* last_page_len, int64_t* start_pos, int32_t* n_page_ids);

#ifdef __cplusplus
}
#endif

#endif  /* PG_KV_H_ */
