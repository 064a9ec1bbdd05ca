// Internal declarations shared by the library's host code and kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <mutex>

namespace pg {

// One-time, per-device set-up of a kernel's launch attributes (shared-memory opt-in, SM
// count): the attributes belong to the whole process on each device, so the first caller on a
// device runs `fn` once under std::call_once and every thread then reads the recorded result.
// Devices 0..127.
struct PerDeviceOnce {
  std::once_flag flag[128];
  cudaError_t err[128] = {};
  int value[128] = {};
  template <class F>
  cudaError_t get(int dev, F fn, int* out) {
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    std::call_once(flag[dev], [&] { err[dev] = fn(&value[dev]); });
    *out = value[dev];
    return err[dev];
  }
};

// Device view of a plan's metadata (all int32, uploaded by the plan builder).
struct PlanDev {
  const int32_t* qo_indptr;       // [R+1]
  const int32_t* kv_page_indptr;  // [R+1]
  const int32_t* page_ids;        // [num_page_ids]
  const int32_t* last_page_len;   // [R]
  const int32_t* start_pos;       // [R]
  const int32_t* kv_start;        // [R]   first key position held (0 unless a key segment)
  const int32_t* tok_req;         // [T]   request of each token row
  const int32_t* work_req;        // [num_work] prefill work item: request
  const int32_t* work_tok0;       // [num_work] prefill work item: first request-local token
  // [num_pairs][8]: two consecutive query tiles of one request, with the request's geometry so
  // a kernel reads it in one step: {first request-local token of the pair, qo_indptr[r],
  // qo_len, start_pos, kv_page_indptr[r], kv_page_indptr[r + 1], kv_end, kv_start}; the keys
  // held are positions [kv_start, kv_end)
  const int32_t* pair_tab;
  int32_t num_req, num_tokens, num_page_ids, num_work, num_pairs;
  // ring addressing: logical page pos / page_size of request r is its page
  // (pos / page_size) mod (pages of r), and kv_len = start_pos + qo_len
  int32_t ring;
};

// Device view of one family's pool, already narrowed to the called layer.
struct PoolDev {
  __nv_bfloat16* layer_base;  // pool base + layer * stride_layer
  int64_t stride_page, stride_kv, stride_head;  // elements; stride_slot == head_dim
  int32_t num_pages, page_size, num_kv_heads, head_dim;
};

struct PrepArgs {
  PlanDev plan;
  PoolDev pool;
  const __nv_bfloat16* q_raw;
  const __nv_bfloat16* k_raw;
  const __nv_bfloat16* v_raw;  // null for the head_dim-512 form
  int64_t q_stride, k_stride, v_stride;  // token strides, elements
  const __nv_bfloat16* w_q;
  const __nv_bfloat16* w_k;
  const float* rope_cos;
  const float* rope_sin;
  __nv_bfloat16* q_out;
  float eps;
  int32_t rope_rows;
  int32_t num_qo_heads;
  int* status;
};

struct AttnArgs {
  PlanDev plan;
  PoolDev pool;
  const __nv_bfloat16* q;
  __nv_bfloat16* out;
  float* lse;     // optional [T][Hq] natural-log normaliser of each row (null: not written)
  void* ws_raw;   // decode form: the caller's workspace (pg_workspace_bytes), 16-byte aligned
  float* ws_o;    // chunked decode form: partial outputs [R][Hq][max_chunks][D]
  float* ws_ml;   // chunked decode form: [R][Hq][max_chunks][2] (running max in log2 units, sum)
  float sm_scale_log2;  // sm_scale * log2(e)
  int32_t window_left;
  int32_t num_qo_heads;
  int32_t group;        // Hq / Hkv
  int32_t cta_tile_q;   // query tokens per prefill CTA
  int32_t kv_chunk;     // keys per decode chunk
  int32_t max_chunks;
  int* status;
  uint64_t wait_ns;       // limit of the kernels' bounded waits (nanoseconds)
  int32_t test_withhold;  // test hook of pg_test_bounded_wait (0: off)
};

// Bounded-wait settings for the next launches: the default limit, or the test hook's.
void wait_settings(uint64_t* wait_ns, int32_t* test_withhold);

// Device status word: set by kernels that skip an out-of-range access.
constexpr int kStatusBounds = 1;
// Device status word: a bounded wait inside a kernel ran out of time.
constexpr int kStatusTimeout = 2;

// Launch counter shared by all launchers.
void count_launch();

// ---- launchers (return cudaError_t of the launch) ----
cudaError_t launch_rope_table(float* cos_t, float* sin_t, int32_t rows, int32_t head_dim,
                              double theta, cudaStream_t stream);
cudaError_t launch_prep_hd256(const PrepArgs& a, cudaStream_t stream);
cudaError_t launch_prep_hd512(const PrepArgs& a, cudaStream_t stream);

// Query tokens per CTA of the prefill attention kernel for this geometry, or 0 when the
// kernel does not support it. Defined next to the kernels (the kernel's own derivation).
int32_t attn_kernel_cta_tile_q(int32_t head_dim, int32_t group, int32_t page_size);
// tcgen05 prefill kernel: geometry it handles, rows per CTA, launch.
bool attn_tc_supported(int32_t head_dim, int32_t group, int32_t page_size);
int32_t attn_tc_rows();
cudaError_t launch_attn_prefill_tc(const AttnArgs& a, int32_t head_dim, cudaStream_t stream);
// Keys per split-KV chunk of the decode kernel.
int32_t attn_kernel_kv_chunk(int32_t head_dim);
cudaError_t launch_attn_prefill(const AttnArgs& a, int32_t head_dim, cudaStream_t stream);
cudaError_t launch_attn_decode(const AttnArgs& a, int32_t head_dim, cudaStream_t stream);
// Decode as one balanced stream over the step's visible keys (TMA-fed, persistent): the
// geometry it handles (head_dim 256/512, group <= 16, power-of-two page size), the workspace
// it needs, and its launch (decode kernel + merge of the segments cut between CTAs).
bool attn_decode_stream_supported(int32_t head_dim, int32_t group, int32_t page_size);
size_t attn_decode_stream_ws_bytes(int32_t num_req, int32_t group, int32_t head_dim);
cudaError_t launch_attn_decode_stream(const AttnArgs& a, int32_t head_dim, cudaStream_t stream);

// Decode attention with its partials in the library's static scratch (no allocation).
// The caller has already checked the plan's workspace size against that scratch.
cudaError_t launch_attn_decode_static(AttnArgs a, int32_t head_dim, cudaStream_t stream);

// Merge of two attention states over disjoint key sets (cascade attention), row by row.
cudaError_t launch_merge_states(const __nv_bfloat16* out_a, const float* lse_a,
                                const __nv_bfloat16* out_b, const float* lse_b,
                                __nv_bfloat16* out, float* lse, int32_t rows, int32_t head_dim,
                                cudaStream_t stream);

}  // namespace pg
