// Fused QKV prep: RMSNorm + half-split rotary on Q (contiguous out) and on K, weightless
// RMSNorm on V (never rotated), with K and V scattered straight into the layer's paged
// pool ("gemma4: serving prep needs pool-write forms", Description and Proposed Plan).
//
// HBM-bound single pass. One CTA per token row; each warp owns whole head rows so the
// RMS reduction is a warp shuffle. Every lane moves 16-byte vectors; a head row of
// 256 bf16 is one 512-byte coalesced access per warp, a 512-wide row two of them.
// All loads of a warp's rows are issued before any arithmetic so each warp keeps
// several 512-byte requests in flight.
#include "pg_internal.h"

#include <cuda_bf16.h>
#include <math.h>

namespace pg {
namespace {

struct alignas(16) V8 {
  uint4 u;
};

__device__ __forceinline__ uint4 ld_stream(const __nv_bfloat16* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void unpack8(const uint4& v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint4 pack8(const float* f) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t*>(&h);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ void set_status(int* st) { atomicOr(st, kStatusBounds); }

// Per-token addressing shared by both forms. Returns false (and flags the status word)
// when metadata would put the access out of range.
struct TokenSlot {
  int32_t pos;
  __nv_bfloat16* k_row0;  // K row of kv head 0 at this token's slot (V is +stride_kv)
};

__device__ __forceinline__ bool token_slot(const PrepArgs& a, int32_t t, TokenSlot* ts) {
  const PlanDev& pl = a.plan;
  const int32_t r = pl.tok_req[t];
  if (r < 0 || r >= pl.num_req) return false;
  const int32_t q0 = pl.qo_indptr[r];
  const int32_t pos = pl.start_pos[r] + (t - q0);
  const int32_t ps = a.pool.page_size;
  const int32_t pidx = pl.kv_page_indptr[r] + pos / ps;
  if (t < q0 || t >= pl.qo_indptr[r + 1] || pos < 0 || pos >= a.rope_rows ||
      pidx >= pl.kv_page_indptr[r + 1] || pidx >= pl.num_page_ids)
    return false;
  const int32_t page = pl.page_ids[pidx];
  if (page < 0 || page >= a.pool.num_pages) return false;
  ts->pos = pos;
  ts->k_row0 = a.pool.layer_base + (int64_t)page * a.pool.stride_page +
               (int64_t)(pos % ps) * a.pool.head_dim;
  return true;
}

// ----------------------------------------------------------------------------- hd256
// Lane l holds elements [8l, 8l+8) of a 256-wide row; its rotary partner elements
// (i +/- 128) live in lane l ^ 16. Rows of a token: Hq query rows, then Hkv K rows,
// then Hkv V rows.
constexpr int kWarps256 = 8;
constexpr int kMaxRows256 = 4;  // rows per warp held in registers per pass

__global__ void __launch_bounds__(kWarps256 * 32)
prep_hd256_kernel(PrepArgs a) {
  const int32_t t = blockIdx.x;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int32_t Hq = a.num_qo_heads;
  const int32_t Hkv = a.pool.num_kv_heads;
  const int32_t nrows = Hq + 2 * Hkv;

  TokenSlot ts;
  const bool ok = token_slot(a, t, &ts);
  if (!ok) {
    if (threadIdx.x == 0) set_status(a.status);
    return;
  }
  const int half = lane >> 4;      // 0: elements [0,128), 1: [128,256)
  const int ci = (lane & 15) * 8;  // rotary table column of this lane's first element
  float c[8], s[8];
  {
    const float4* cp = reinterpret_cast<const float4*>(a.rope_cos + (int64_t)ts.pos * 128 + ci);
    const float4* sp = reinterpret_cast<const float4*>(a.rope_sin + (int64_t)ts.pos * 128 + ci);
    float4 c0 = __ldg(cp), c1 = __ldg(cp + 1), s0 = __ldg(sp), s1 = __ldg(sp + 1);
    c[0] = c0.x; c[1] = c0.y; c[2] = c0.z; c[3] = c0.w; c[4] = c1.x; c[5] = c1.y; c[6] = c1.z; c[7] = c1.w;
    s[0] = s0.x; s[1] = s0.y; s[2] = s0.z; s[3] = s0.w; s[4] = s1.x; s[5] = s1.y; s[6] = s1.z; s[7] = s1.w;
  }
  float wq[8], wk[8];
  unpack8(__ldg(reinterpret_cast<const uint4*>(a.w_q) + lane), wq);
  unpack8(__ldg(reinterpret_cast<const uint4*>(a.w_k) + lane), wk);

  for (int base = warp; base < nrows; base += kWarps256 * kMaxRows256) {
    uint4 raw[kMaxRows256];
#pragma unroll
    for (int i = 0; i < kMaxRows256; ++i) {
      const int row = base + i * kWarps256;
      if (row < nrows) {
        const __nv_bfloat16* src;
        if (row < Hq) src = a.q_raw + (int64_t)t * a.q_stride + (int64_t)row * 256;
        else if (row < Hq + Hkv) src = a.k_raw + (int64_t)t * a.k_stride + (int64_t)(row - Hq) * 256;
        else src = a.v_raw + (int64_t)t * a.v_stride + (int64_t)(row - Hq - Hkv) * 256;
        raw[i] = ld_stream(src + lane * 8);
      }
    }
#pragma unroll
    for (int i = 0; i < kMaxRows256; ++i) {
      const int row = base + i * kWarps256;
      if (row >= nrows) break;
      float x[8];
      unpack8(raw[i], x);
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
      ss = warp_sum(ss);
      const float inv = 1.0f / sqrtf(ss * (1.0f / 256.0f) + a.eps);
      const bool is_v = row >= Hq + Hkv;
      float y[8];
      if (is_v) {
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = x[e] * inv;
      } else {
        const float* w = row < Hq ? wq : wk;
        float u[8], pu[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) u[e] = x[e] * inv * w[e];
#pragma unroll
        for (int e = 0; e < 8; ++e) pu[e] = __shfl_xor_sync(0xffffffffu, u[e], 16);
        if (half == 0) {
#pragma unroll
          for (int e = 0; e < 8; ++e) y[e] = u[e] * c[e] - pu[e] * s[e];
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) y[e] = u[e] * c[e] + pu[e] * s[e];
        }
      }
      const uint4 o = pack8(y);
      __nv_bfloat16* dst;
      if (row < Hq) dst = a.q_out + ((int64_t)t * Hq + row) * 256;
      else if (!is_v) dst = ts.k_row0 + (int64_t)(row - Hq) * a.pool.stride_head;
      else dst = ts.k_row0 + a.pool.stride_kv + (int64_t)(row - Hq - Hkv) * a.pool.stride_head;
      *reinterpret_cast<uint4*>(dst + lane * 8) = o;
    }
  }
}

// ----------------------------------------------------------------------------- hd512
// Lane l holds elements [8l, 8l+8) and [256+8l, 256+8l+8): each rotary pair (i, i+256)
// sits in one lane. Rows of a token: Hq query rows, then Hkv K rows; each K row also
// produces its V row from the same registers and the same inverse RMS.
constexpr int kWarps512 = 8;
constexpr int kMaxRows512 = 2;

__global__ void __launch_bounds__(kWarps512 * 32)
prep_hd512_kernel(PrepArgs a) {
  const int32_t t = blockIdx.x;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int32_t Hq = a.num_qo_heads;
  const int32_t Hkv = a.pool.num_kv_heads;
  const int32_t nrows = Hq + Hkv;

  TokenSlot ts;
  if (!token_slot(a, t, &ts)) {
    if (threadIdx.x == 0) set_status(a.status);
    return;
  }
  const int ci = lane * 8;
  float c[8], s[8];
  {
    const float4* cp = reinterpret_cast<const float4*>(a.rope_cos + (int64_t)ts.pos * 256 + ci);
    const float4* sp = reinterpret_cast<const float4*>(a.rope_sin + (int64_t)ts.pos * 256 + ci);
    float4 c0 = __ldg(cp), c1 = __ldg(cp + 1), s0 = __ldg(sp), s1 = __ldg(sp + 1);
    c[0] = c0.x; c[1] = c0.y; c[2] = c0.z; c[3] = c0.w; c[4] = c1.x; c[5] = c1.y; c[6] = c1.z; c[7] = c1.w;
    s[0] = s0.x; s[1] = s0.y; s[2] = s0.z; s[3] = s0.w; s[4] = s1.x; s[5] = s1.y; s[6] = s1.z; s[7] = s1.w;
  }

  for (int base = warp; base < nrows; base += kWarps512 * kMaxRows512) {
    uint4 lo[kMaxRows512], hi[kMaxRows512];
#pragma unroll
    for (int i = 0; i < kMaxRows512; ++i) {
      const int row = base + i * kWarps512;
      if (row < nrows) {
        const __nv_bfloat16* src =
            row < Hq ? a.q_raw + (int64_t)t * a.q_stride + (int64_t)row * 512
                     : a.k_raw + (int64_t)t * a.k_stride + (int64_t)(row - Hq) * 512;
        lo[i] = ld_stream(src + ci);
        hi[i] = ld_stream(src + 256 + ci);
      }
    }
#pragma unroll
    for (int i = 0; i < kMaxRows512; ++i) {
      const int row = base + i * kWarps512;
      if (row >= nrows) break;
      float xa[8], xb[8];
      unpack8(lo[i], xa);
      unpack8(hi[i], xb);
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = fmaf(xa[e], xa[e], fmaf(xb[e], xb[e], ss));
      ss = warp_sum(ss);
      const float inv = 1.0f / sqrtf(ss * (1.0f / 512.0f) + a.eps);
      const bool is_q = row < Hq;
      const __nv_bfloat16* wp = is_q ? a.w_q : a.w_k;
      float wa[8], wb[8];
      unpack8(__ldg(reinterpret_cast<const uint4*>(wp + ci)), wa);
      unpack8(__ldg(reinterpret_cast<const uint4*>(wp + 256 + ci)), wb);
      float ya[8], yb[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float ua = xa[e] * inv * wa[e];
        const float ub = xb[e] * inv * wb[e];
        ya[e] = ua * c[e] - ub * s[e];
        yb[e] = ub * c[e] + ua * s[e];
      }
      __nv_bfloat16* dst = is_q ? a.q_out + ((int64_t)t * Hq + row) * 512
                                : ts.k_row0 + (int64_t)(row - Hq) * a.pool.stride_head;
      *reinterpret_cast<uint4*>(dst + ci) = pack8(ya);
      *reinterpret_cast<uint4*>(dst + 256 + ci) = pack8(yb);
      if (!is_q) {
        // V: the weightless norm of the same raw K row, same inverse RMS, no rotation.
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          ya[e] = xa[e] * inv;
          yb[e] = xb[e] * inv;
        }
        __nv_bfloat16* vdst = dst + a.pool.stride_kv;
        *reinterpret_cast<uint4*>(vdst + ci) = pack8(ya);
        *reinterpret_cast<uint4*>(vdst + 256 + ci) = pack8(yb);
      }
    }
  }
}

// ----------------------------------------------------------------------------- rotary table
__global__ void rope_table_kernel(float* cos_t, float* sin_t, int32_t rows, int32_t half,
                                  double theta) {
  const int64_t n = (int64_t)rows * half;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < n;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int32_t p = (int32_t)(idx / half);
    const int32_t i = (int32_t)(idx % half);
    const double inv_freq = pow(theta, -2.0 * (double)i / (double)(2 * half));
    double sv, cv;
    sincos((double)p * inv_freq, &sv, &cv);
    cos_t[idx] = (float)cv;
    sin_t[idx] = (float)sv;
  }
}

}  // namespace

cudaError_t launch_rope_table(float* cos_t, float* sin_t, int32_t rows, int32_t head_dim,
                              double theta, cudaStream_t stream) {
  const int32_t half = head_dim / 2;
  const int64_t n = (int64_t)rows * half;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 152 * 64) blocks = 152 * 64;
  rope_table_kernel<<<(unsigned)blocks, 256, 0, stream>>>(cos_t, sin_t, rows, half, theta);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_prep_hd256(const PrepArgs& a, cudaStream_t stream) {
  prep_hd256_kernel<<<a.plan.num_tokens, kWarps256 * 32, 0, stream>>>(a);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_prep_hd512(const PrepArgs& a, cudaStream_t stream) {
  prep_hd512_kernel<<<a.plan.num_tokens, kWarps512 * 32, 0, stream>>>(a);
  count_launch();
  return cudaGetLastError();
}

}  // namespace pg
