// Host-side page accounting for two-family paged KV serving ("feat(gemma4): paged KV serving
// across both attention families", Description, Verification and the review finding "Commit KV
// frontiers only after a successful step"): one page allocator per family, a per-request state
// in both, admission atomic across both pools with the page count as the exact frontier
// account, every check before any state changes, the local family failing closed at its
// sliding window, and a step's frontier advanced only when the caller commits the step after
// its launches succeeded (an aborted step returns its pages and leaves the frontier).
// Declared in include/pg_kv.h.
#include "../../include/pg_kv.h"

#include <cstdint>
#include <new>
#include <set>
#include <unordered_map>
#include <vector>

namespace {

struct KvRequest {
  int32_t frontier[2] = {0, 0};     // positions committed, per family (kept equal)
  std::vector<int32_t> pages[2];    // page ids in position order, per family (pending included)
  int32_t pending = 0;              // tokens of the admitted, not yet committed step (0: none)
  int32_t pending_new[2] = {0, 0};  // pages that step took, per family (the tail of pages[f])
};

int32_t pages_for(int64_t len, int32_t ps) { return (int32_t)((len + ps - 1) / ps); }

}  // namespace

struct pg_kv_server {
  int32_t page_size = 0, window_left = 0, fail_closed = 0, rope_rows = 0;
  // ring mode (0: off): the local family holds at most ring_pages pages per request, reused as
  // a ring once the frontier passes them; steps are at most ring_max_step tokens
  int32_t ring_pages = 0, ring_max_step = 0;
  std::set<int32_t> free_pages[2];  // lowest id first
  int32_t refusals[2] = {0, 0};     // injected refusals still to come
  int64_t next_id = 1;
  std::unordered_map<int64_t, KvRequest> requests;

  // Take `need` pages from a family's pool, or none (false) when the pool cannot cover them
  // or a refusal was injected.
  bool reserve(int family, int32_t need, std::vector<int32_t>* got) {
    got->clear();
    if (need <= 0) return true;
    if (refusals[family] > 0) {
      --refusals[family];
      return false;
    }
    if ((int64_t)free_pages[family].size() < need) return false;
    auto it = free_pages[family].begin();
    for (int32_t i = 0; i < need; ++i) got->push_back(*it++);
    free_pages[family].erase(free_pages[family].begin(), it);
    return true;
  }
  void give_back(int family, const std::vector<int32_t>& pages) {
    free_pages[family].insert(pages.begin(), pages.end());
  }
  // Pages a family holds at a frontier: ceil(frontier / page_size), capped at the ring for
  // the local family in ring mode.
  int32_t held_for(int family, int64_t frontier) const {
    const int32_t n = pages_for(frontier, page_size);
    return (family == PG_KV_LOCAL && ring_pages > 0 && n > ring_pages) ? ring_pages : n;
  }
  // The frontier account: both families at one frontier, each holding exactly the pages of
  // the frontier plus its pending step.
  bool consistent(const KvRequest& r) const {
    if (r.frontier[0] != r.frontier[1] || r.pending < 0) return false;
    for (int f = 0; f < 2; ++f) {
      if ((int64_t)r.pages[f].size() != held_for(f, (int64_t)r.frontier[f] + r.pending)) return false;
      if (r.pending_new[f] < 0 || r.pending_new[f] > (int32_t)r.pages[f].size()) return false;
    }
    return true;
  }
};

extern "C" {

int pg_kv_server_create(pg_kv_server_t* out, int32_t pages_local, int32_t pages_global,
                        int32_t page_size, int32_t window_left, int32_t fail_closed_at_window,
                        int32_t rope_rows) {
  if (!out || pages_local < 0 || pages_global < 0 || page_size <= 0 || window_left < 0 ||
      rope_rows <= 0)
    return PG_KV_ERR_ARG;
  pg_kv_server* s = new (std::nothrow) pg_kv_server;
  if (!s) return PG_KV_ERR_ARG;
  s->page_size = page_size;
  s->window_left = window_left;
  s->fail_closed = fail_closed_at_window != 0;
  s->rope_rows = rope_rows;
  for (int32_t p = 0; p < pages_local; ++p) s->free_pages[PG_KV_LOCAL].insert(p);
  for (int32_t p = 0; p < pages_global; ++p) s->free_pages[PG_KV_GLOBAL].insert(p);
  *out = s;
  return PG_KV_OK;
}

int pg_kv_server_create_ring(pg_kv_server_t* out, int32_t pages_local, int32_t pages_global,
                             int32_t page_size, int32_t window_left, int32_t ring_max_step,
                             int32_t rope_rows) {
  if (ring_max_step < 1 || page_size <= 0 || window_left < 0) return PG_KV_ERR_ARG;
  const int64_t ring = ((int64_t)window_left + ring_max_step + page_size - 1) / page_size;
  if (ring > INT32_MAX) return PG_KV_ERR_ARG;
  const int rc = pg_kv_server_create(out, pages_local, pages_global, page_size, window_left, 0,
                                     rope_rows);
  if (rc != PG_KV_OK) return rc;
  (*out)->ring_pages = (int32_t)ring;
  (*out)->ring_max_step = ring_max_step;
  return PG_KV_OK;
}

void pg_kv_server_destroy(pg_kv_server_t srv) { delete srv; }

int pg_kv_request_open(pg_kv_server_t srv, int64_t* request_id) {
  if (!srv || !request_id) return PG_KV_ERR_ARG;
  const int64_t id = srv->next_id++;
  srv->requests.emplace(id, KvRequest());
  *request_id = id;
  return PG_KV_OK;
}

int pg_kv_request_close(pg_kv_server_t srv, int64_t request_id) {
  if (!srv) return PG_KV_ERR_ARG;
  auto it = srv->requests.find(request_id);
  if (it == srv->requests.end()) return PG_KV_ERR_FOREIGN;
  for (int f = 0; f < 2; ++f) srv->give_back(f, it->second.pages[f]);
  srv->requests.erase(it);
  return PG_KV_OK;
}

int pg_kv_admit_step(pg_kv_server_t srv, int64_t request_id, int32_t n_tokens) {
  if (!srv || n_tokens < 1) return PG_KV_ERR_ARG;
  auto it = srv->requests.find(request_id);
  if (it == srv->requests.end()) return PG_KV_ERR_FOREIGN;
  KvRequest& r = it->second;
  // every check before anything changes
  if (r.pending != 0) return PG_KV_ERR_PENDING;
  if (!srv->consistent(r)) return PG_KV_ERR_FRONTIER;
  const int64_t len = (int64_t)r.frontier[0] + n_tokens;
  if (len > INT32_MAX) return PG_KV_ERR_ARG;
  if (srv->fail_closed && len > (int64_t)srv->window_left + 1) return PG_KV_ERR_WINDOW;
  // a ring holds the window plus at most ring_max_step new positions
  if (srv->ring_pages > 0 && n_tokens > srv->ring_max_step) return PG_KV_ERR_WINDOW;
  if (len > srv->rope_rows) return PG_KV_ERR_ROPE;
  int32_t need[2];
  for (int f = 0; f < 2; ++f) need[f] = srv->held_for(f, len) - (int32_t)r.pages[f].size();
  // reserve both before recording either; a refused side drops the other
  std::vector<int32_t> got[2];
  if (!srv->reserve(PG_KV_LOCAL, need[PG_KV_LOCAL], &got[PG_KV_LOCAL])) return PG_KV_ERR_NO_PAGES;
  if (!srv->reserve(PG_KV_GLOBAL, need[PG_KV_GLOBAL], &got[PG_KV_GLOBAL])) {
    srv->give_back(PG_KV_LOCAL, got[PG_KV_LOCAL]);
    return PG_KV_ERR_NO_PAGES;
  }
  // the step is pending: its pages are held, the frontier stays until pg_kv_commit_step
  for (int f = 0; f < 2; ++f) {
    r.pages[f].insert(r.pages[f].end(), got[f].begin(), got[f].end());
    r.pending_new[f] = (int32_t)got[f].size();
  }
  r.pending = n_tokens;
  return PG_KV_OK;
}

int pg_kv_commit_step(pg_kv_server_t srv, int64_t request_id) {
  if (!srv) return PG_KV_ERR_ARG;
  auto it = srv->requests.find(request_id);
  if (it == srv->requests.end()) return PG_KV_ERR_FOREIGN;
  KvRequest& r = it->second;
  if (r.pending == 0) return PG_KV_ERR_PENDING;
  if (!srv->consistent(r)) return PG_KV_ERR_FRONTIER;
  for (int f = 0; f < 2; ++f) {
    r.frontier[f] += r.pending;
    r.pending_new[f] = 0;
  }
  r.pending = 0;
  return PG_KV_OK;
}

int pg_kv_abort_step(pg_kv_server_t srv, int64_t request_id) {
  if (!srv) return PG_KV_ERR_ARG;
  auto it = srv->requests.find(request_id);
  if (it == srv->requests.end()) return PG_KV_ERR_FOREIGN;
  KvRequest& r = it->second;
  if (r.pending == 0) return PG_KV_ERR_PENDING;
  if (!srv->consistent(r)) return PG_KV_ERR_FRONTIER;
  // the step's own pages go back to their pools; the pages before it and the frontier stay
  for (int f = 0; f < 2; ++f) {
    const size_t keep = r.pages[f].size() - (size_t)r.pending_new[f];
    std::vector<int32_t> back(r.pages[f].begin() + (std::ptrdiff_t)keep, r.pages[f].end());
    r.pages[f].resize(keep);
    srv->give_back(f, back);
    r.pending_new[f] = 0;
  }
  r.pending = 0;
  return PG_KV_OK;
}

int pg_kv_request_info(pg_kv_server_t srv, int64_t request_id, int32_t* frontier,
                       int32_t* pages_local, int32_t* pages_global) {
  if (!srv) return PG_KV_ERR_ARG;
  auto it = srv->requests.find(request_id);
  if (it == srv->requests.end()) return PG_KV_ERR_FOREIGN;
  if (frontier) *frontier = it->second.frontier[0];
  if (pages_local) *pages_local = (int32_t)it->second.pages[PG_KV_LOCAL].size();
  if (pages_global) *pages_global = (int32_t)it->second.pages[PG_KV_GLOBAL].size();
  return PG_KV_OK;
}

int pg_kv_request_pending(pg_kv_server_t srv, int64_t request_id, int32_t* pending) {
  if (!srv || !pending) return PG_KV_ERR_ARG;
  auto it = srv->requests.find(request_id);
  if (it == srv->requests.end()) return PG_KV_ERR_FOREIGN;
  *pending = it->second.pending;
  return PG_KV_OK;
}

int pg_kv_request_pages(pg_kv_server_t srv, int64_t request_id, int32_t family, int32_t* out,
                        int32_t cap, int32_t* n) {
  if (!srv || !n || (family != PG_KV_LOCAL && family != PG_KV_GLOBAL) || cap < 0)
    return PG_KV_ERR_ARG;
  auto it = srv->requests.find(request_id);
  if (it == srv->requests.end()) return PG_KV_ERR_FOREIGN;
  const std::vector<int32_t>& p = it->second.pages[family];
  if ((int64_t)p.size() > cap) return PG_KV_ERR_CAPACITY;
  if (!p.empty() && !out) return PG_KV_ERR_ARG;
  for (size_t i = 0; i < p.size(); ++i) out[i] = p[i];
  *n = (int32_t)p.size();
  return PG_KV_OK;
}

int pg_kv_free_pages(pg_kv_server_t srv, int32_t family, int32_t* n) {
  if (!srv || !n || (family != PG_KV_LOCAL && family != PG_KV_GLOBAL)) return PG_KV_ERR_ARG;
  *n = (int32_t)srv->free_pages[family].size();
  return PG_KV_OK;
}

int pg_kv_inject_refusal(pg_kv_server_t srv, int32_t family, int32_t count) {
  if (!srv || (family != PG_KV_LOCAL && family != PG_KV_GLOBAL) || count < 0) return PG_KV_ERR_ARG;
  srv->refusals[family] = count;
  return PG_KV_OK;
}

int pg_kv_batch_plan_inputs(pg_kv_server_t srv, int32_t family, int32_t n,
                            const int64_t* request_ids, const int32_t* step_tokens,
                            int64_t* kv_page_indptr, int32_t* page_ids, int32_t cap,
                            int32_t* last_page_len, int64_t* start_pos, int32_t* n_page_ids) {
  if (!srv || (family != PG_KV_LOCAL && family != PG_KV_GLOBAL) || n < 0 || cap < 0 ||
      !n_page_ids || !kv_page_indptr)
    return PG_KV_ERR_ARG;
  if (n > 0 && (!request_ids || !step_tokens || !last_page_len || !start_pos))
    return PG_KV_ERR_ARG;
  // validate everything first, then write
  int64_t total = 0;
  for (int32_t i = 0; i < n; ++i) {
    auto it = srv->requests.find(request_ids[i]);
    if (it == srv->requests.end()) return PG_KV_ERR_FOREIGN;
    const KvRequest& r = it->second;
    if (!srv->consistent(r)) return PG_KV_ERR_FRONTIER;
    // the plan covers the request's admitted step, which must still be pending
    if (r.pending == 0) return PG_KV_ERR_PENDING;
    if (step_tokens[i] != r.pending) return PG_KV_ERR_ARG;
    total += (int64_t)r.pages[family].size();
  }
  if (total > cap) return PG_KV_ERR_CAPACITY;
  if (total > 0 && !page_ids) return PG_KV_ERR_ARG;
  int64_t off = 0;
  kv_page_indptr[0] = 0;
  for (int32_t i = 0; i < n; ++i) {
    const KvRequest& r = srv->requests.find(request_ids[i])->second;
    const std::vector<int32_t>& p = r.pages[family];
    for (size_t k = 0; k < p.size(); ++k) page_ids[off + (int64_t)k] = p[k];
    off += (int64_t)p.size();
    kv_page_indptr[i + 1] = off;
    // the step's last position's slot count in its page (a ring plan does not read it)
    const int32_t end = r.frontier[family] + r.pending;
    last_page_len[i] = end - ((end - 1) / srv->page_size) * srv->page_size;
    start_pos[i] = (int64_t)r.frontier[family];
  }
  *n_page_ids = (int32_t)total;
  return PG_KV_OK;
}

}  // extern "C"
