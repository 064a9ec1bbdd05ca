// Host side of the C ABI: plan builder, checked geometry, argument checks, dispatch.
//
// Every check runs before any launch and before any write to caller memory
// ("feat(kernels): Rust wrapper for the hd256 windowed paged prefill", Description and
// Verification; "gemma4: serving prep needs pool-write forms", Proposed Plan).
#include "../../include/pg.h"
#include "pg_internal.h"

#include <atomic>
#include <climits>
#include <cmath>
#include <cstring>
#include <mutex>
#include <new>
#include <algorithm>
#include <vector>

namespace pg {

static std::atomic<int64_t> g_launches{0};
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

// Bounded waits give up after two seconds unless the test hook set a shorter limit.
constexpr uint64_t kDefaultWaitNs = 2000000000ull;
static std::atomic<uint64_t> g_wait_ns{kDefaultWaitNs};
static std::atomic<int32_t> g_test_withhold{0};
void wait_settings(uint64_t* wait_ns, int32_t* test_withhold) {
  *wait_ns = g_wait_ns.load(std::memory_order_relaxed);
  *test_withhold = g_test_withhold.load(std::memory_order_relaxed);
}

// One status word per device, allocated on first use with that device current.
static std::mutex g_status_mu;
static int* g_status_dev[128] = {nullptr};

static int* status_word(int* err) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) {
    *err = PG_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_status_mu);
  if (!g_status_dev[dev]) {
    int* p = nullptr;
    if (cudaMalloc(&p, sizeof(int)) != cudaSuccess) { *err = PG_ERR_CUDA; return nullptr; }
    if (cudaMemset(p, 0, sizeof(int)) != cudaSuccess) { cudaFree(p); *err = PG_ERR_CUDA; return nullptr; }
    g_status_dev[dev] = p;
  }
  *err = PG_OK;
  return g_status_dev[dev];
}

// ------------------------------------------------------------------ checked arithmetic
static bool mul_i64(int64_t a, int64_t b, int64_t* out) { return !__builtin_mul_overflow(a, b, out); }
static bool add_i64(int64_t a, int64_t b, int64_t* out) { return !__builtin_add_overflow(a, b, out); }
static bool fits_i32(int64_t v) { return v >= INT32_MIN && v <= INT32_MAX; }

// Query tokens per prefill CTA as the plan derives it (must agree with the kernel's):
// 128 rows on the tensor-memory path (head_dim 256/512, group dividing 128, power-of-two page
// size >= 8), else 64 (head_dim 256) or 32 (head_dim 512) rows on the mma.sync path.
static int32_t plan_cta_tile_q(int32_t head_dim, int32_t group, int32_t page_size) {
  if (group <= 0 || group > 16) return 0;
  const bool tc = (head_dim == 256 || head_dim == 512) && 128 % group == 0 && page_size >= 8 &&
                  (page_size & (page_size - 1)) == 0;
  const int32_t rows = tc ? 128 : head_dim == 256 ? 64 : head_dim == 512 ? 32 : 0;
  if (rows == 0 || rows % group != 0) return 0;
  return rows / group;
}
static int32_t plan_kv_chunk(int32_t head_dim) { return head_dim == 512 ? 512 : 256; }

}  // namespace pg

using namespace pg;

// Pinned host staging for a plan's metadata upload, two buffers used alternately: an upload from
// pageable memory can hold the host until the stream reaches it, which in a serving loop that
// rebuilds a plan while earlier calls still run would stall every later launch. Buffer k is
// rewritten only after the upload recorded on done[k] (two builds back) has completed.
struct PlanStage {
  int32_t* host[2] = {nullptr, nullptr};
  size_t cap[2] = {0, 0};
  cudaEvent_t done[2] = {nullptr, nullptr};
  int next = 0;
};

struct pg_plan {
  int32_t num_req = 0, num_tokens = 0, num_qo_heads = 0, num_kv_heads = 0, head_dim = 0,
          page_size = 0;
  int32_t max_page_id = -1, max_last_page_len = 0, max_qo_len = 0, max_kv_len = 0,
          max_pos_end = 0;
  int32_t cta_tile_q = 0, decode = 0, kv_chunk = 0, max_chunks = 0, num_work = 0, num_pairs = 0;
  int32_t num_page_ids = 0;
  int32_t ring = 0, ring_window = -1;  // ring addressing (window-crossing requests) and its window
  // key segments (cascade attention): request r's pages hold key positions
  // [kv_start_r, kv_start_r + n_r); prep_ok: every request's step tokens are its segment's tail
  int32_t segment = 0, prep_ok = 1;
  cudaStream_t stream = nullptr;
  int device = 0;
  int32_t* dev = nullptr;  // one device allocation holding every metadata array
  size_t dev_elems = 0;
  size_t dev_cap = 0;      // bytes allocated at dev
  // offsets (elements) of each array inside `dev`
  size_t o_qo = 0, o_kvp = 0, o_pages = 0, o_last = 0, o_start = 0, o_kvs = 0, o_tokreq = 0,
         o_wreq = 0, o_wtok = 0, o_pair = 0;
  PlanStage stage;  // carried over from build to build of the same plan
};

namespace {

// releases a plan's staging buffers once their uploads have completed
void free_stage(PlanStage* st) {
  for (int k = 0; k < 2; ++k) {
    if (st->done[k]) {
      cudaEventSynchronize(st->done[k]);
      cudaEventDestroy(st->done[k]);
      st->done[k] = nullptr;
    }
    if (st->host[k]) cudaFreeHost(st->host[k]);
    st->host[k] = nullptr;
    st->cap[k] = 0;
  }
}

// ring_window < 0: linear addressing (slot = position, pages cover [0, kv_len) exactly, with
// last_page_len). ring_window >= 0: ring addressing for window-crossing requests: logical page
// pos / ps lives in the request's page (pos / ps) mod (pages held), kv_len = start_pos + qo_len,
// last_page_len is not read, and the ring must hold the window plus the step
// (pages * ps >= ring_window + qo_len), so no key a query of the step can see is overwritten by
// the step's own writes.
// kv_start != null: key segments (linear addressing within the segment): request r's pages hold
// key positions [kv_start_r, kv_start_r + n_r), n_r = (pages - 1) * ps + last_page_len_r, from
// slot 0 on; the segment ends at or before the step's last position.
int build_plan(pg_plan* p, int32_t num_req, const int64_t* qo_indptr,
               const int64_t* kv_page_indptr, const int32_t* page_ids,
               const int32_t* last_page_len, const int64_t* start_pos, int32_t Hq,
               int32_t Hkv, int32_t D, int32_t ps, cudaStream_t stream,
               int32_t ring_window = -1, const int64_t* kv_start = nullptr) {
  const bool ring = ring_window >= 0;
  const bool segment = kv_start != nullptr;
  if (ring && segment) return PG_ERR_ARG;
  // The head relation is settled before anything divides by num_kv_heads.
  if (Hkv == 0) return PG_ERR_ZERO_KV_HEADS;
  if (Hkv < 0 || Hq <= 0 || Hq % Hkv != 0) return PG_ERR_HEADS;
  if (D <= 0 || D % 2 != 0 || ps <= 0) return PG_ERR_ARG;
  if (num_req < 0) return PG_ERR_ARG;
  if (num_req > 0 && (!qo_indptr || !kv_page_indptr || !page_ids || !start_pos ||
                      (!ring && !last_page_len)))
    return PG_ERR_ARG;
  const int32_t group = Hq / Hkv;

  std::vector<int32_t> qo(num_req + 1, 0), kvp(num_req + 1, 0), last(num_req), start(num_req),
      kvs(num_req, 0);
  if (num_req > 0) {
    if (qo_indptr[0] != 0 || kv_page_indptr[0] != 0) return PG_ERR_ARG;
  }
  int32_t max_page = -1, max_last = 0, max_qo = 0, max_kv = 0, max_end = 0, max_seen = 0;
  bool all_one = num_req > 0, prep_ok = true;
  for (int32_t r = 0; r < num_req; ++r) {
    const int64_t q0 = qo_indptr[r], q1 = qo_indptr[r + 1];
    const int64_t k0 = kv_page_indptr[r], k1 = kv_page_indptr[r + 1];
    if (q1 <= q0 || k1 <= k0) return PG_ERR_ARG;  // every request: >= 1 token, >= 1 page
    if (!fits_i32(q1) || !fits_i32(k1)) return PG_ERR_I32_OVERFLOW;
    const int64_t qo_len = q1 - q0;
    const int64_t sp = start_pos[r];
    if (sp < 0) return PG_ERR_ARG;
    int64_t pos_end = 0;
    if (!add_i64(sp, qo_len, &pos_end) || !fits_i32(pos_end)) return PG_ERR_I32_OVERFLOW;
    int32_t lpl = 0;
    int64_t kv_len = 0, seg0 = 0;  // kv_len: end of the keys held (exclusive); seg0: first
    if (!ring) {
      lpl = last_page_len[r];
      if (lpl < 1 || lpl > ps) return PG_ERR_LAST_PAGE_LEN;
      if (!mul_i64(k1 - k0 - 1, ps, &kv_len) || !add_i64(kv_len, lpl, &kv_len))
        return PG_ERR_I32_OVERFLOW;
      if (segment) {
        seg0 = kv_start[r];
        if (seg0 < 0) return PG_ERR_ARG;
        if (!add_i64(seg0, kv_len, &kv_len)) return PG_ERR_I32_OVERFLOW;
      }
      if (!fits_i32(kv_len)) return PG_ERR_I32_OVERFLOW;
      if (!segment && kv_len != pos_end) return PG_ERR_COVERAGE;
      // a segment holds no key past the step's last position (no query could see it)
      if (segment && kv_len > pos_end) return PG_ERR_COVERAGE;
      if (segment && !(kv_len == pos_end && sp >= seg0)) prep_ok = false;
    } else {
      int64_t cap = 0, need = 0;
      if (!mul_i64(k1 - k0, ps, &cap) || !add_i64(ring_window, qo_len, &need))
        return PG_ERR_I32_OVERFLOW;
      // a step's write can cover a key one of its queries sees only if some position wraps
      // (pos_end > cap) and the ring is shorter than the window plus the step
      if (cap < need && pos_end > cap) return PG_ERR_COVERAGE;
      kv_len = pos_end;
      // the position's slot in its (ring) page; last_page_len is not used in ring addressing
      lpl = (int32_t)(pos_end - ((pos_end - 1) / ps) * ps);
    }
    qo[r + 1] = (int32_t)q1;
    kvp[r + 1] = (int32_t)k1;
    last[r] = lpl;
    start[r] = (int32_t)sp;
    kvs[r] = (int32_t)seg0;
    if (kv_len - seg0 > max_seen) max_seen = (int32_t)(kv_len - seg0);
    if (lpl > max_last) max_last = lpl;
    if (qo_len > max_qo) max_qo = (int32_t)qo_len;
    if (kv_len > max_kv) max_kv = (int32_t)kv_len;
    if (pos_end > max_end) max_end = (int32_t)pos_end;
    if (qo_len != 1) all_one = false;
  }
  const int32_t T = num_req > 0 ? qo[num_req] : 0;
  const int32_t NP = num_req > 0 ? kvp[num_req] : 0;
  for (int32_t i = 0; i < NP; ++i) {
    if (page_ids[i] < 0) return PG_ERR_PAGE_OOB;
    if (page_ids[i] > max_page) max_page = page_ids[i];
  }

  // Tiling derived from the geometry; attention re-derives it from the kernel itself.
  const int32_t cta = plan_cta_tile_q(D, group, ps);
  const int32_t chunk = plan_kv_chunk(D);
  {
    // the chunked decode kernel holds a request's key chunks in its grid's z dimension
    const int64_t seen = ring ? std::min<int64_t>(max_kv, (int64_t)ring_window + 1) : max_seen;
    if (all_one && !attn_decode_stream_supported(D, group, ps) && (seen + chunk - 1) / chunk > 65535)
      return PG_ERR_I32_OVERFLOW;
  }
  int64_t nwork = 0;
  std::vector<int32_t> wreq, wtok, ptab;
  if (cta > 0) {
    for (int32_t r = 0; r < num_req; ++r) {
      const int32_t len = qo[r + 1] - qo[r];
      for (int32_t t = 0; t < len; t += cta) {
        wreq.push_back(r);
        wtok.push_back(t);
      }
      // the tcgen05 prefill runs query tiles in pairs (one per CTA of a cluster) that share
      // their key tiles; a request with an odd number of tiles ends with a single-tile pair
      for (int64_t t = 0; t < len; t += 2 * (int64_t)cta) {
        const int32_t kv_len =
            ring ? start[r] + len : kvs[r] + (kvp[r + 1] - kvp[r] - 1) * ps + last[r];
        const int32_t e[8] = {(int32_t)t, qo[r], len, start[r], kvp[r], kvp[r + 1], kv_len, kvs[r]};
        ptab.insert(ptab.end(), e, e + 8);
      }
    }
    nwork = (int64_t)wreq.size();
  }
  if (!fits_i32(nwork)) return PG_ERR_I32_OVERFLOW;

  // Pack everything into one int32 array and upload it on the plan's stream.
  std::vector<int32_t> host;
  auto put = [&](const int32_t* src, size_t n) {
    const size_t off = host.size();
    host.insert(host.end(), src, src + n);
    while (host.size() % 4) host.push_back(0);  // 16-byte aligned sub-arrays
    return off;
  };
  std::vector<int32_t> tokreq(T);
  for (int32_t r = 0; r < num_req; ++r)
    for (int32_t t = qo[r]; t < qo[r + 1]; ++t) tokreq[t] = r;
  std::vector<int32_t> pids(page_ids, page_ids + NP);

  pg_plan q;
  q.o_qo = put(qo.data(), qo.size());
  q.o_kvp = put(kvp.data(), kvp.size());
  q.o_pages = put(pids.data(), pids.size());
  q.o_last = put(last.data(), last.size());
  q.o_start = put(start.data(), start.size());
  q.o_kvs = put(kvs.data(), kvs.size());
  q.o_tokreq = put(tokreq.data(), tokreq.size());
  q.o_wreq = put(wreq.data(), wreq.size());
  q.o_wtok = put(wtok.data(), wtok.size());
  q.o_pair = put(ptab.data(), ptab.size());
  if (host.empty()) host.assign(4, 0);

  int err = PG_OK;
  if (!status_word(&err)) return err;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PG_ERR_CUDA;
  // the upload goes through this plan's next pinned staging buffer (see PlanStage)
  PlanStage& st = p->stage;
  const int k = st.next;
  const size_t bytes = host.size() * sizeof(int32_t);
  if (!st.done[k]) {
    if (cudaEventCreateWithFlags(&st.done[k], cudaEventDisableTiming) != cudaSuccess) {
      st.done[k] = nullptr;
      return PG_ERR_CUDA;
    }
  } else if (cudaEventSynchronize(st.done[k]) != cudaSuccess) {
    return PG_ERR_CUDA;
  }
  if (st.cap[k] < bytes) {
    if (st.host[k]) cudaFreeHost(st.host[k]);
    st.host[k] = nullptr;
    st.cap[k] = 0;
    if (cudaMallocHost((void**)&st.host[k], bytes) != cudaSuccess) {
      st.host[k] = nullptr;
      return PG_ERR_CUDA;
    }
    st.cap[k] = bytes;
  }
  std::memcpy(st.host[k], host.data(), bytes);
  // An existing plan whose device storage is large enough is updated in place: the copy is
  // ordered on the plan's stream after every call already queued with the old metadata (a plan
  // is used on its own stream only), and a CUDA graph that captured the plan keeps reading live
  // metadata. Otherwise new storage is allocated and the old freed after the commit.
  int32_t* d = nullptr;
  const bool fresh = !(p->dev && p->dev_cap >= bytes);
  if (fresh) {
    if (cudaMallocAsync((void**)&d, bytes, stream) != cudaSuccess) return PG_ERR_CUDA;
  } else {
    d = p->dev;
  }
  if (cudaMemcpyAsync(d, st.host[k], bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
      cudaEventRecord(st.done[k], stream) != cudaSuccess) {
    if (fresh) cudaFreeAsync(d, stream);
    return PG_ERR_CUDA;
  }
  st.next = k ^ 1;

  q.num_req = num_req; q.num_tokens = T; q.num_qo_heads = Hq; q.num_kv_heads = Hkv;
  q.head_dim = D; q.page_size = ps;
  q.max_page_id = max_page; q.max_last_page_len = max_last; q.max_qo_len = max_qo;
  q.max_kv_len = max_kv; q.max_pos_end = max_end;
  q.cta_tile_q = cta; q.decode = all_one ? 1 : 0; q.kv_chunk = chunk;
  // decode partials: a query sees at most window + 1 keys in ring addressing
  const int64_t seen = ring ? std::min<int64_t>(max_kv, (int64_t)ring_window + 1) : max_seen;
  q.max_chunks = seen > 0 ? (int32_t)((seen + chunk - 1) / chunk) : 0;
  q.ring = ring ? 1 : 0;
  q.ring_window = ring ? ring_window : -1;
  q.segment = segment ? 1 : 0;
  q.prep_ok = prep_ok ? 1 : 0;
  q.num_work = (int32_t)nwork; q.num_pairs = (int32_t)(ptab.size() / 8); q.num_page_ids = NP;
  q.stream = stream; q.device = dev;
  q.dev = d; q.dev_elems = host.size();
  q.dev_cap = fresh ? bytes : p->dev_cap;

  // Commit: only now does the caller's plan change.
  int32_t* old = p->dev;
  q.stage = p->stage;
  *p = q;
  if (fresh && old) cudaFreeAsync(old, stream);
  return PG_OK;
}

PlanDev plan_dev(const pg_plan* p) {
  PlanDev v;
  v.qo_indptr = p->dev + p->o_qo;
  v.kv_page_indptr = p->dev + p->o_kvp;
  v.page_ids = p->dev + p->o_pages;
  v.last_page_len = p->dev + p->o_last;
  v.start_pos = p->dev + p->o_start;
  v.kv_start = p->dev + p->o_kvs;
  v.tok_req = p->dev + p->o_tokreq;
  v.work_req = p->dev + p->o_wreq;
  v.work_tok0 = p->dev + p->o_wtok;
  v.pair_tab = p->dev + p->o_pair;
  v.num_req = p->num_req;
  v.num_tokens = p->num_tokens;
  v.num_page_ids = p->num_page_ids;
  v.num_work = p->num_work;
  v.num_pairs = p->num_pairs;
  v.ring = p->ring;
  return v;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// checked_paged_geometry: the pool descriptor must be self-consistent for head_dim D.
int check_pool(const pg_pool_t* pool, int32_t D) {
  if (!pool || !pool->base) return PG_ERR_ARG;
  if (pool->head_dim != D) return PG_ERR_LAYOUT;
  if (pool->num_layers <= 0 || pool->num_pages <= 0 || pool->page_size <= 0 ||
      pool->num_kv_heads <= 0)
    return PG_ERR_LAYOUT;
  if (!aligned16(pool->base)) return PG_ERR_ALIGN;
  int64_t s_slot = D, s_head, s_kv, s_page, s_layer, total;
  if (!mul_i64(pool->page_size, s_slot, &s_head) || !mul_i64(pool->num_kv_heads, s_head, &s_kv) ||
      !mul_i64(2, s_kv, &s_page) || !mul_i64(pool->num_pages, s_page, &s_layer) ||
      !mul_i64(pool->num_layers, s_layer, &total))
    return PG_ERR_I32_OVERFLOW;
  if (pool->stride_slot != s_slot || pool->stride_head != s_head || pool->stride_kv != s_kv ||
      pool->stride_page != s_page || pool->stride_layer != s_layer)
    return PG_ERR_LAYOUT;
  if (pool->capacity != total) return PG_ERR_LAYOUT;  // whole pages, every layer
  return PG_OK;
}

// Plan vs pool agreement plus the recorded page bounds, before every launch.
int check_plan_pool(const pg_plan* p, const pg_pool_t* pool, int32_t layer, int32_t D) {
  if (p->head_dim != D) return PG_ERR_PLAN_MISMATCH;
  int rc = check_pool(pool, D);
  if (rc) return rc;
  if (p->num_kv_heads != pool->num_kv_heads || p->page_size != pool->page_size)
    return PG_ERR_PLAN_MISMATCH;
  if (layer < 0 || layer >= pool->num_layers) return PG_ERR_LAYER;
  if (p->max_page_id >= pool->num_pages) return PG_ERR_PAGE_OOB;
  if (p->max_last_page_len > pool->page_size) return PG_ERR_LAST_PAGE_LEN;
  return PG_OK;
}

PoolDev pool_dev(const pg_pool_t* pool, int32_t layer) {
  PoolDev v;
  v.layer_base = reinterpret_cast<__nv_bfloat16*>(pool->base) + (int64_t)layer * pool->stride_layer;
  v.stride_page = pool->stride_page;
  v.stride_kv = pool->stride_kv;
  v.stride_head = pool->stride_head;
  v.num_pages = pool->num_pages;
  v.page_size = pool->page_size;
  v.num_kv_heads = pool->num_kv_heads;
  v.head_dim = pool->head_dim;
  return v;
}

int check_tok_input(const pg_bf16_t* p, int64_t stride, int32_t heads, int32_t D) {
  if (!p) return PG_ERR_ARG;
  if (stride < (int64_t)heads * D) return PG_ERR_ARG;
  if (!aligned16(p) || stride % 8 != 0) return PG_ERR_ALIGN;
  return PG_OK;
}

int prep_common(const pg_plan* plan, const pg_pool_t* pool, int32_t layer, int32_t D,
                const pg_bf16_t* q_raw, int64_t qs, const pg_bf16_t* k_raw, int64_t ks,
                const pg_bf16_t* v_raw, int64_t vs, const pg_bf16_t* w_q, const pg_bf16_t* w_k,
                float eps, const float* rc, const float* rsn, int32_t rope_rows,
                pg_bf16_t* q_out, cudaStream_t stream, PrepArgs* a) {
  if (!plan) return PG_ERR_ARG;
  if (stream != plan->stream) return PG_ERR_STREAM;
  // a key-segment plan takes prep only when every step's tokens are its segment's tail
  if (plan->segment && !plan->prep_ok) return PG_ERR_COVERAGE;
  int rc_ = check_plan_pool(plan, pool, layer, D);
  if (rc_) return rc_;
  if (!std::isfinite(eps) || !(eps > 0.0f)) return PG_ERR_NONFINITE;
  if (plan->num_tokens == 0) return PG_OK;
  if (!rc || !rsn || !w_q || !w_k || !q_out) return PG_ERR_ARG;
  if (rope_rows < 1) return PG_ERR_ARG;
  if (plan->max_pos_end > rope_rows) return PG_ERR_ROPE_RANGE;
  if ((rc_ = check_tok_input(q_raw, qs, plan->num_qo_heads, D))) return rc_;
  if ((rc_ = check_tok_input(k_raw, ks, plan->num_kv_heads, D))) return rc_;
  if (D == 256 && (rc_ = check_tok_input(v_raw, vs, plan->num_kv_heads, D))) return rc_;
  if (!aligned16(w_q) || !aligned16(w_k) || !aligned16(q_out) || !aligned16(rc) || !aligned16(rsn))
    return PG_ERR_ALIGN;
  int64_t span = 0;  // largest element offset any raw input row reaches must fit int64
  if (!mul_i64((int64_t)plan->num_tokens, qs > ks ? (qs > vs ? qs : vs) : (ks > vs ? ks : vs), &span))
    return PG_ERR_I32_OVERFLOW;
  int err = PG_OK;
  int* st = status_word(&err);
  if (!st) return err;
  a->plan = plan_dev(plan);
  a->pool = pool_dev(pool, layer);
  a->q_raw = reinterpret_cast<const __nv_bfloat16*>(q_raw);
  a->k_raw = reinterpret_cast<const __nv_bfloat16*>(k_raw);
  a->v_raw = reinterpret_cast<const __nv_bfloat16*>(v_raw);
  a->q_stride = qs; a->k_stride = ks; a->v_stride = vs;
  a->w_q = reinterpret_cast<const __nv_bfloat16*>(w_q);
  a->w_k = reinterpret_cast<const __nv_bfloat16*>(w_k);
  a->rope_cos = rc; a->rope_sin = rsn;
  a->q_out = reinterpret_cast<__nv_bfloat16*>(q_out);
  a->eps = eps;
  a->rope_rows = rope_rows;
  a->num_qo_heads = plan->num_qo_heads;
  a->status = st;
  return PG_OK;
}

size_t workspace_bytes(const pg_plan* p) {
  if (!p || !p->decode || p->num_req == 0) return 0;
  const int32_t group = p->num_qo_heads / p->num_kv_heads;
  if (attn_decode_stream_supported(p->head_dim, group, p->page_size))
    return attn_decode_stream_ws_bytes(p->num_req, group, p->head_dim);
  const size_t rows = (size_t)p->num_req * p->num_qo_heads * p->max_chunks;
  return rows * (size_t)p->head_dim * sizeof(float) + rows * 2 * sizeof(float);
}

int attn_common(const pg_plan* plan, const pg_pool_t* pool, int32_t layer, int32_t D,
                const pg_bf16_t* q, pg_bf16_t* out, float* lse, int32_t window_left,
                float sm_scale, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!plan) return PG_ERR_ARG;
  if (stream != plan->stream) return PG_ERR_STREAM;
  int rc = check_plan_pool(plan, pool, layer, D);
  if (rc) return rc;
  const int32_t group = plan->num_qo_heads / plan->num_kv_heads;
  const int32_t kernel_cta = attn_kernel_cta_tile_q(D, group, plan->page_size);
  if (kernel_cta == 0 || kernel_cta != plan->cta_tile_q) return PG_ERR_PLAN_MISMATCH;
  if (attn_kernel_kv_chunk(D) != plan->kv_chunk) return PG_ERR_PLAN_MISMATCH;
  if (window_left < -1) return PG_ERR_WINDOW;
  // ring addressing holds only the window the plan was built for
  if (plan->ring && (window_left < 0 || window_left > plan->ring_window)) return PG_ERR_WINDOW;
  if (!std::isfinite(sm_scale)) return PG_ERR_NONFINITE;
  const bool tma_rows = plan->decode ? attn_decode_stream_supported(D, group, plan->page_size)
                                     : attn_tc_supported(D, group, plan->page_size);
  // the chunked decode kernel's grid holds the key chunks of a request in its z dimension
  if (plan->decode && !attn_decode_stream_supported(D, group, plan->page_size) &&
      plan->max_chunks > 65535)
    return PG_ERR_I32_OVERFLOW;
  if (tma_rows && (int64_t)pool->num_pages * 2 * pool->num_kv_heads * pool->page_size > INT32_MAX)
    return PG_ERR_I32_OVERFLOW;  // tensor-map row coordinates are int32
  if (plan->num_tokens == 0) return PG_OK;
  if (!q || !out) return PG_ERR_ARG;
  // the tensor-core prefill kernel reads Q rows and writes output rows in 32-byte accesses
  if ((((uintptr_t)q | (uintptr_t)out) & 31u) != 0) return PG_ERR_ALIGN;
  if (lse && ((uintptr_t)lse & 3u) != 0) return PG_ERR_ALIGN;
  const size_t need = workspace_bytes(plan);
  if (need > 0) {
    if (!ws || ws_bytes < need) return PG_ERR_WORKSPACE;
    if (!aligned16(ws)) return PG_ERR_ALIGN;
  }
  int err = PG_OK;
  int* st = status_word(&err);
  if (!st) return err;
  AttnArgs a;
  a.plan = plan_dev(plan);
  a.pool = pool_dev(pool, layer);
  a.q = reinterpret_cast<const __nv_bfloat16*>(q);
  a.out = reinterpret_cast<__nv_bfloat16*>(out);
  a.lse = lse;
  a.sm_scale_log2 = sm_scale * 1.4426950408889634f;
  a.window_left = window_left;
  a.num_qo_heads = plan->num_qo_heads;
  a.group = group;
  a.cta_tile_q = plan->cta_tile_q;
  a.kv_chunk = plan->kv_chunk;
  a.max_chunks = plan->max_chunks;
  a.status = st;
  wait_settings(&a.wait_ns, &a.test_withhold);
  cudaError_t e;
  a.ws_raw = ws;
  a.ws_o = nullptr;
  a.ws_ml = nullptr;
  if (plan->decode) {
    e = launch_attn_decode(a, D, stream);
  } else {
    e = launch_attn_prefill(a, D, stream);
  }
  return e == cudaSuccess ? PG_OK : PG_ERR_CUDA;
}

// The device's status word if it already exists; never allocates.
int* status_word_existing(int* err) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) {
    *err = PG_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_status_mu);
  *err = g_status_dev[dev] ? PG_OK : PG_ERR_CUDA;
  return g_status_dev[dev];
}

}  // namespace

extern "C" {

int pg_plan_paged_prefill(pg_plan_t* plan, int32_t num_req, const int64_t* qo_indptr,
                          const int64_t* kv_page_indptr, const int32_t* page_ids,
                          const int32_t* last_page_len, const int64_t* start_pos,
                          int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                          int32_t page_size, pg_stream_t stream) {
  if (!plan) return PG_ERR_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (*plan) {
    if ((*plan)->stream != s) return PG_ERR_STREAM;
    return build_plan(*plan, num_req, qo_indptr, kv_page_indptr, page_ids, last_page_len,
                      start_pos, num_qo_heads, num_kv_heads, head_dim, page_size, s);
  }
  pg_plan* p = new (std::nothrow) pg_plan();
  if (!p) return PG_ERR_ARG;
  int rc = build_plan(p, num_req, qo_indptr, kv_page_indptr, page_ids, last_page_len, start_pos,
                      num_qo_heads, num_kv_heads, head_dim, page_size, s);
  if (rc != PG_OK) {
    free_stage(&p->stage);
    delete p;
    return rc;
  }
  *plan = p;
  return PG_OK;
}

int pg_plan_paged_prefill_ring(pg_plan_t* plan, int32_t num_req, const int64_t* qo_indptr,
                               const int64_t* kv_page_indptr, const int32_t* page_ids,
                               const int64_t* start_pos, int32_t num_qo_heads,
                               int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                               int32_t window_left, pg_stream_t stream) {
  if (!plan) return PG_ERR_ARG;
  if (window_left < 0) return PG_ERR_WINDOW;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (*plan) {
    if ((*plan)->stream != s) return PG_ERR_STREAM;
    return build_plan(*plan, num_req, qo_indptr, kv_page_indptr, page_ids, nullptr, start_pos,
                      num_qo_heads, num_kv_heads, head_dim, page_size, s, window_left);
  }
  pg_plan* p = new (std::nothrow) pg_plan();
  if (!p) return PG_ERR_ARG;
  int rc = build_plan(p, num_req, qo_indptr, kv_page_indptr, page_ids, nullptr, start_pos,
                      num_qo_heads, num_kv_heads, head_dim, page_size, s, window_left);
  if (rc != PG_OK) {
    free_stage(&p->stage);
    delete p;
    return rc;
  }
  *plan = p;
  return PG_OK;
}

int pg_plan_paged_segment(pg_plan_t* plan, int32_t num_req, const int64_t* qo_indptr,
                          const int64_t* kv_page_indptr, const int32_t* page_ids,
                          const int32_t* last_page_len, const int64_t* kv_start,
                          const int64_t* start_pos, int32_t num_qo_heads, int32_t num_kv_heads,
                          int32_t head_dim, int32_t page_size, pg_stream_t stream) {
  if (!plan) return PG_ERR_ARG;
  if (num_req > 0 && !kv_start) return PG_ERR_ARG;
  static const int64_t kNoSegments = 0;  // a non-null pointer for an empty batch
  const int64_t* ks = kv_start ? kv_start : &kNoSegments;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (*plan) {
    if ((*plan)->stream != s) return PG_ERR_STREAM;
    return build_plan(*plan, num_req, qo_indptr, kv_page_indptr, page_ids, last_page_len,
                      start_pos, num_qo_heads, num_kv_heads, head_dim, page_size, s, -1, ks);
  }
  pg_plan* p = new (std::nothrow) pg_plan();
  if (!p) return PG_ERR_ARG;
  int rc = build_plan(p, num_req, qo_indptr, kv_page_indptr, page_ids, last_page_len, start_pos,
                      num_qo_heads, num_kv_heads, head_dim, page_size, s, -1, ks);
  if (rc != PG_OK) {
    free_stage(&p->stage);
    delete p;
    return rc;
  }
  *plan = p;
  return PG_OK;
}

void pg_plan_destroy(pg_plan_t plan) {
  if (!plan) return;
  if (plan->dev) cudaFreeAsync(plan->dev, plan->stream);
  free_stage(&plan->stage);
  delete plan;
}

int pg_plan_info(const pg_plan_t p, pg_plan_info_t* info) {
  if (!p || !info) return PG_ERR_ARG;
  info->num_req = p->num_req; info->num_tokens = p->num_tokens;
  info->num_qo_heads = p->num_qo_heads; info->num_kv_heads = p->num_kv_heads;
  info->head_dim = p->head_dim; info->page_size = p->page_size;
  info->max_page_id = p->max_page_id; info->max_last_page_len = p->max_last_page_len;
  info->max_qo_len = p->max_qo_len; info->max_kv_len = p->max_kv_len;
  info->max_pos_end = p->max_pos_end; info->cta_tile_q = p->cta_tile_q;
  info->decode = p->decode; info->kv_chunk = p->kv_chunk; info->max_chunks = p->max_chunks;
  info->num_work = p->num_work;
  info->d_page_ids = p->dev + p->o_pages;
  info->stream = reinterpret_cast<pg_stream_t>(p->stream);
  info->metadata_bytes = (int64_t)p->dev_elems * (int64_t)sizeof(int32_t);
  return PG_OK;
}

int pg_rope_table(float* rope_cos, float* rope_sin, int32_t rows, int32_t head_dim, double theta,
                  pg_stream_t stream) {
  if (!rope_cos || !rope_sin || rows < 1 || head_dim < 2 || head_dim % 2) return PG_ERR_ARG;
  if (!std::isfinite(theta) || !(theta > 0.0)) return PG_ERR_NONFINITE;
  int64_t n = 0;
  if (!mul_i64(rows, head_dim / 2, &n) || !fits_i32(n)) return PG_ERR_I32_OVERFLOW;
  cudaError_t e = launch_rope_table(rope_cos, rope_sin, rows, head_dim, theta,
                                    reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PG_OK : PG_ERR_CUDA;
}

int pg_prep_paged_hd256(const pg_plan_t plan, const pg_pool_t* pool, int32_t layer,
                        const pg_bf16_t* q_raw, int64_t q_tok_stride, const pg_bf16_t* k_raw,
                        int64_t k_tok_stride, const pg_bf16_t* v_raw, int64_t v_tok_stride,
                        const pg_bf16_t* w_q, const pg_bf16_t* w_k, float eps,
                        const float* rope_cos, const float* rope_sin, int32_t rope_rows,
                        pg_bf16_t* q_out, pg_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  PrepArgs a;
  int rc = prep_common(plan, pool, layer, 256, q_raw, q_tok_stride, k_raw, k_tok_stride, v_raw,
                       v_tok_stride, w_q, w_k, eps, rope_cos, rope_sin, rope_rows, q_out, s, &a);
  if (rc != PG_OK || plan->num_tokens == 0) return rc;
  return launch_prep_hd256(a, s) == cudaSuccess ? PG_OK : PG_ERR_CUDA;
}

int pg_prep_paged_hd512(const pg_plan_t plan, const pg_pool_t* pool, int32_t layer,
                        const pg_bf16_t* q_raw, int64_t q_tok_stride, const pg_bf16_t* k_raw,
                        int64_t k_tok_stride, const pg_bf16_t* w_q, const pg_bf16_t* w_k,
                        float eps, const float* rope_cos, const float* rope_sin,
                        int32_t rope_rows, pg_bf16_t* q_out, pg_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  PrepArgs a;
  int rc = prep_common(plan, pool, layer, 512, q_raw, q_tok_stride, k_raw, k_tok_stride, nullptr,
                       0, w_q, w_k, eps, rope_cos, rope_sin, rope_rows, q_out, s, &a);
  if (rc != PG_OK || plan->num_tokens == 0) return rc;
  return launch_prep_hd512(a, s) == cudaSuccess ? PG_OK : PG_ERR_CUDA;
}

size_t pg_workspace_bytes(const pg_plan_t plan) { return workspace_bytes(plan); }

int pg_attn_paged_prefill(const pg_plan_t plan, const pg_pool_t* pool, int32_t layer,
                          const pg_bf16_t* q, pg_bf16_t* out, int32_t window_left, float sm_scale,
                          void* workspace, size_t ws_bytes, pg_stream_t stream) {
  return attn_common(plan, pool, layer, 256, q, out, nullptr, window_left, sm_scale, workspace, ws_bytes,
                     reinterpret_cast<cudaStream_t>(stream));
}

int pg_attn_paged_prefill_hd512(const pg_plan_t plan, const pg_pool_t* pool, int32_t layer,
                                const pg_bf16_t* q, pg_bf16_t* out, int32_t window_left,
                                float sm_scale, void* workspace, size_t ws_bytes,
                                pg_stream_t stream) {
  return attn_common(plan, pool, layer, 512, q, out, nullptr, window_left, sm_scale, workspace, ws_bytes,
                     reinterpret_cast<cudaStream_t>(stream));
}

int pg_attn_paged_prefill_lse(const pg_plan_t plan, const pg_pool_t* pool, int32_t layer,
                              const pg_bf16_t* q, pg_bf16_t* out, float* lse,
                              int32_t window_left, float sm_scale, void* workspace,
                              size_t ws_bytes, pg_stream_t stream) {
  if (!lse && plan && plan->num_tokens > 0) return PG_ERR_ARG;
  return attn_common(plan, pool, layer, 256, q, out, lse, window_left, sm_scale, workspace,
                     ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

int pg_attn_paged_prefill_hd512_lse(const pg_plan_t plan, const pg_pool_t* pool, int32_t layer,
                                    const pg_bf16_t* q, pg_bf16_t* out, float* lse,
                                    int32_t window_left, float sm_scale, void* workspace,
                                    size_t ws_bytes, pg_stream_t stream) {
  if (!lse && plan && plan->num_tokens > 0) return PG_ERR_ARG;
  return attn_common(plan, pool, layer, 512, q, out, lse, window_left, sm_scale, workspace,
                     ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

int pg_merge_attn_states(const pg_bf16_t* out_a, const float* lse_a, const pg_bf16_t* out_b,
                         const float* lse_b, pg_bf16_t* out, float* lse, int64_t rows,
                         int32_t head_dim, pg_stream_t stream) {
  if (rows < 0 || head_dim <= 0 || head_dim % 8 != 0) return PG_ERR_ARG;
  if (rows > INT32_MAX) return PG_ERR_I32_OVERFLOW;
  if (rows == 0) return PG_OK;
  if (!out_a || !lse_a || !out_b || !lse_b || !out) return PG_ERR_ARG;
  if (!aligned16(out_a) || !aligned16(out_b) || !aligned16(out)) return PG_ERR_ALIGN;
  if (((uintptr_t)lse_a & 3u) || ((uintptr_t)lse_b & 3u) || ((uintptr_t)lse & 3u))
    return PG_ERR_ALIGN;
  const cudaError_t e = launch_merge_states(
      reinterpret_cast<const __nv_bfloat16*>(out_a), lse_a,
      reinterpret_cast<const __nv_bfloat16*>(out_b), lse_b,
      reinterpret_cast<__nv_bfloat16*>(out), lse, (int32_t)rows, head_dim,
      reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PG_OK : PG_ERR_CUDA;
}

int pg_attn_paged_decode_noalloc(const pg_plan_t plan, const pg_pool_t* pool, int32_t layer,
                                 const pg_bf16_t* q, pg_bf16_t* out, int32_t window_left,
                                 float sm_scale, pg_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!plan) return PG_ERR_ARG;
  if (s != plan->stream) return PG_ERR_STREAM;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PG_ERR_CUDA;
  if (dev != plan->device) return PG_ERR_STREAM;
  if (!plan->decode && plan->num_req > 0) return PG_ERR_PLAN_MISMATCH;
  if (workspace_bytes(plan) > PG_NOALLOC_SCRATCH_BYTES) return PG_ERR_WORKSPACE;
  const int32_t D = plan->head_dim;
  if (D != 256 && D != 512) return PG_ERR_PLAN_MISMATCH;
  int rc = check_plan_pool(plan, pool, layer, D);
  if (rc) return rc;
  const int32_t group = plan->num_qo_heads / plan->num_kv_heads;
  const int32_t kernel_cta = attn_kernel_cta_tile_q(D, group, plan->page_size);
  if (kernel_cta == 0 || kernel_cta != plan->cta_tile_q) return PG_ERR_PLAN_MISMATCH;
  if (attn_kernel_kv_chunk(D) != plan->kv_chunk) return PG_ERR_PLAN_MISMATCH;
  if (window_left < -1) return PG_ERR_WINDOW;
  if (plan->ring && (window_left < 0 || window_left > plan->ring_window)) return PG_ERR_WINDOW;
  if (!std::isfinite(sm_scale)) return PG_ERR_NONFINITE;
  if (attn_decode_stream_supported(D, group, plan->page_size) &&
      (int64_t)pool->num_pages * 2 * pool->num_kv_heads * pool->page_size > INT32_MAX)
    return PG_ERR_I32_OVERFLOW;  // tensor-map row coordinates are int32
  if (!attn_decode_stream_supported(D, group, plan->page_size) && plan->max_chunks > 65535)
    return PG_ERR_I32_OVERFLOW;  // the chunked kernel's grid z dimension
  if (plan->num_tokens == 0) return PG_OK;
  if (!q || !out) return PG_ERR_ARG;
  if (!aligned16(q) || !aligned16(out)) return PG_ERR_ALIGN;
  int err = PG_OK;
  int* st = status_word_existing(&err);
  if (!st) return err;
  AttnArgs a;
  a.plan = plan_dev(plan);
  a.pool = pool_dev(pool, layer);
  a.q = reinterpret_cast<const __nv_bfloat16*>(q);
  a.out = reinterpret_cast<__nv_bfloat16*>(out);
  a.lse = nullptr;
  a.ws_raw = nullptr;
  a.ws_o = nullptr;
  a.ws_ml = nullptr;
  a.sm_scale_log2 = sm_scale * 1.4426950408889634f;
  a.window_left = window_left;
  a.num_qo_heads = plan->num_qo_heads;
  a.group = group;
  a.cta_tile_q = plan->cta_tile_q;
  a.kv_chunk = plan->kv_chunk;
  a.max_chunks = plan->max_chunks;
  a.status = st;
  wait_settings(&a.wait_ns, &a.test_withhold);
  return launch_attn_decode_static(a, D, s) == cudaSuccess ? PG_OK : PG_ERR_CUDA;
}

int pg_device_status(pg_stream_t stream) {
  int err = PG_OK;
  int* st = status_word(&err);
  if (!st) return err;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int h = 0;
  if (cudaMemcpyAsync(&h, st, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return PG_ERR_CUDA;
  if (cudaMemsetAsync(st, 0, sizeof(int), s) != cudaSuccess) return PG_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return PG_ERR_CUDA;
  if (h & kStatusTimeout) return PG_ERR_DEVICE_TIMEOUT;
  return h ? PG_ERR_DEVICE_BOUNDS : PG_OK;
}

int64_t pg_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int pg_test_bounded_wait(int32_t withhold, int64_t wait_limit_ns) {
  if (withhold == 0) {
    g_test_withhold.store(0, std::memory_order_relaxed);
    g_wait_ns.store(kDefaultWaitNs, std::memory_order_relaxed);
    return PG_OK;
  }
  if (withhold != 1 || wait_limit_ns < 1000000 || wait_limit_ns > (int64_t)kDefaultWaitNs)
    return PG_ERR_ARG;
  g_wait_ns.store((uint64_t)wait_limit_ns, std::memory_order_relaxed);
  g_test_withhold.store(1, std::memory_order_relaxed);
  return PG_OK;
}

const char* pg_status_string(int s) {
  switch (s) {
    case PG_OK: return "ok";
    case PG_ERR_ARG: return "invalid argument (null pointer, negative count, bad indptr)";
    case PG_ERR_PAGE_OOB: return "page id outside the pool";
    case PG_ERR_LAST_PAGE_LEN: return "last_page_len outside [1, page_size]";
    case PG_ERR_I32_OVERFLOW: return "length or offset does not fit int32 (or stride product int64)";
    case PG_ERR_ZERO_KV_HEADS: return "num_kv_heads is zero";
    case PG_ERR_HEADS: return "num_qo_heads is not a positive multiple of num_kv_heads";
    case PG_ERR_NONFINITE: return "non-finite or non-positive scale, eps or theta";
    case PG_ERR_ROPE_RANGE: return "a position is past the rotary tables";
    case PG_ERR_COVERAGE: return "pages do not cover the keys the step needs (linear: exactly [0, start_pos + qo_len))";
    case PG_ERR_LAYER: return "layer outside the pool";
    case PG_ERR_LAYOUT: return "pool layout, strides or capacity inconsistent";
    case PG_ERR_PLAN_MISMATCH: return "plan geometry or tiling disagrees with the pool or kernel";
    case PG_ERR_WINDOW: return "window_left below -1";
    case PG_ERR_WORKSPACE: return "workspace missing or too small";
    case PG_ERR_STREAM: return "stream differs from the plan's stream";
    case PG_ERR_CUDA: return "CUDA runtime error";
    case PG_ERR_DEVICE_BOUNDS: return "a kernel skipped an out-of-range access";
    case PG_ERR_ALIGN: return "pointer or stride not 16-byte aligned";
    case PG_ERR_DEVICE_TIMEOUT: return "a kernel gave up a bounded wait and returned early";
    default: return "unknown status";
  }
}

}  // extern "C"
