// Fused QKV prep: RMSNorm + half-split rotary on Q (contiguous out) and on K, weightless
// RMSNorm on V (never rotated), with K and V scattered straight into the layer's paged
// pool ("gemma4: serving prep needs pool-write forms", Description and Proposed Plan).
//
// HBM-bound single pass, one persistent CTA per (SM, slot) walking the tokens
// t = blockIdx.x + k * gridDim.x. A producer warp streams each token's raw rows (all of its
// Q rows, K rows and V rows are contiguous runs) and its rotary row into a ring of
// shared-memory stages with bulk asynchronous copies (cp.async.bulk, completion counted in
// bytes on the stage's mbarrier), several tokens ahead, so every SM keeps hundreds of KB of
// loads in flight without holding them in registers. Eight consumer warps each own whole
// head rows of the staged token: a lane reads 16-byte vectors from shared memory (a 256-wide
// row is one conflict-free 512-byte read per warp), the RMS reduction is a warp shuffle, each
// lane holds both elements of its rotary pairs, and every
// result row is one coalesced 512-byte (or 1 KB) store: q_out rows, or K/V rows at the
// token's paged slot (slot = position, wrapped over the request's pages for a ring plan, or
// counted from the segment's first position for a key-segment plan). The producer also resolves each token's request, position and page
// (32 tokens at a time, one per lane) and passes them to the consumers in the stage header.
//
// Waits are bounded (two seconds of %globaltimer); a wait that runs out sets the device
// status word and the CTA leaves the loop. Tokens whose metadata is out of range set the
// status word and are skipped (no copy, no store).
#include "pg_internal.h"

#include <cuda_bf16.h>
#include <math.h>

#include <algorithm>

namespace pg {
namespace {

constexpr int kPrepConsumerWarps = 8;
constexpr int kPrepThreads = (kPrepConsumerWarps + 1) * 32;  // + producer warp
constexpr uint64_t kPrepWaitNs = 2000000000ull;

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

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void bar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void bar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void bar_arrive_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool bar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase of the given parity; false when it (or another warp) gave up.
__device__ __noinline__ bool bar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                      int* status) {
  if (bar_try(bar, parity)) return true;
  const uint64_t t0 = gtimer();
  while (!bar_try(bar, parity)) {
    if (*abort_flag) return false;
    if (gtimer() - t0 > kPrepWaitNs) {
      atomicOr(status, kStatusTimeout);
      *abort_flag = 1;
      return false;
    }
  }
  return true;
}
// global -> shared bulk copy whose bytes complete on `bar`
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Token metadata the consumers need, written by the producer into the stage header.
struct alignas(16) TokMeta {
  int64_t slot;  // element offset of the token's K row of kv head 0 in the layer
  int32_t pos;   // absolute position (rotary row)
  int32_t ok;    // 0: out-of-range metadata, token skipped
};

// Request, position and paged slot of token t, with every index checked before use.
__device__ __forceinline__ bool token_meta(const PrepArgs& a, int32_t t, TokMeta* m) {
  const PlanDev& pl = a.plan;
  const int32_t r = pl.tok_req[t];
  if (r < 0 || r >= pl.num_req) return false;
  const int32_t q0 = pl.qo_indptr[r];
  const int32_t pos = pl.start_pos[r] + (t - q0);
  const int32_t ps = a.pool.page_size;
  const int32_t kvp0 = pl.kv_page_indptr[r], npg = pl.kv_page_indptr[r + 1] - kvp0;
  if (t < q0 || t >= pl.qo_indptr[r + 1] || pos < 0 || pos >= a.rope_rows || npg <= 0)
    return false;
  // the position's index among the keys the request holds (a key segment starts at kv_start)
  const int32_t rel = pos - pl.kv_start[r];
  if (rel < 0) return false;
  // ring addressing: logical page rel / ps lives in page (rel / ps) mod (pages held)
  const int32_t pidx = kvp0 + (pl.ring ? (rel / ps) % npg : rel / ps);
  if (pidx >= kvp0 + npg || pidx >= pl.num_page_ids) return false;
  const int32_t page = pl.page_ids[pidx];
  if (page < 0 || page >= a.pool.num_pages) return false;
  m->pos = pos;
  m->slot = (int64_t)page * a.pool.stride_page + (int64_t)(rel % ps) * a.pool.head_dim;
  m->ok = 1;
  return true;
}

// Normalise (and for Q/K rows weight and rotate) one staged row and store it. Each rotary pair
// (i, i + D/2) sits in one lane, so the rotation needs no shuffle:
//   D = 256: lane l holds elements [4l, 4l + 4) and [128 + 4l, 128 + 4l + 4);
//   D = 512: lane l holds [8l, 8l + 8) and [256 + 8l, 256 + 8l + 8).
// kind: 0 = Q, 1 = K, 2 = V (weightless, not rotated). For D = 512 a K row also writes its V
// row: the weightless norm of the same raw row with the same inverse RMS.
template <int D>
__device__ __forceinline__ void prep_row(const PrepArgs& a, const unsigned char* row_smem, int kind,
                                         int lane, const float* c, const float* s,
                                         const float* w_lo, const float* w_hi,
                                         __nv_bfloat16* dst, __nv_bfloat16* vdst) {
  if constexpr (D == 256) {
    // lane l: elements [4l, 4l + 4) and their rotary partners [128 + 4l, 128 + 4l + 4)
    float xa[4], xb[4];
    {
      const uint2 va = *reinterpret_cast<const uint2*>(row_smem + lane * 8);
      const uint2 vb = *reinterpret_cast<const uint2*>(row_smem + 256 + lane * 8);
      xa[0] = __uint_as_float(va.x << 16); xa[1] = __uint_as_float(va.x & 0xFFFF0000u);
      xa[2] = __uint_as_float(va.y << 16); xa[3] = __uint_as_float(va.y & 0xFFFF0000u);
      xb[0] = __uint_as_float(vb.x << 16); xb[1] = __uint_as_float(vb.x & 0xFFFF0000u);
      xb[2] = __uint_as_float(vb.y << 16); xb[3] = __uint_as_float(vb.y & 0xFFFF0000u);
    }
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) ss = fmaf(xa[e], xa[e], fmaf(xb[e], xb[e], ss));
    ss = warp_sum(ss);
    const float inv = 1.0f / sqrtf(ss * (1.0f / 256.0f) + a.eps);
    float ya[4], yb[4];
    if (kind == 2) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        ya[e] = xa[e] * inv;
        yb[e] = xb[e] * inv;
      }
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float ua = xa[e] * inv * w_lo[e];
        const float ub = xb[e] * inv * w_hi[e];
        ya[e] = ua * c[e] - ub * s[e];
        yb[e] = ub * c[e] + ua * s[e];
      }
    }
    uint2 oa, ob;
    {
      __nv_bfloat162 h0 = __floats2bfloat162_rn(ya[0], ya[1]), h1 = __floats2bfloat162_rn(ya[2], ya[3]);
      __nv_bfloat162 h2 = __floats2bfloat162_rn(yb[0], yb[1]), h3 = __floats2bfloat162_rn(yb[2], yb[3]);
      oa = make_uint2(*reinterpret_cast<uint32_t*>(&h0), *reinterpret_cast<uint32_t*>(&h1));
      ob = make_uint2(*reinterpret_cast<uint32_t*>(&h2), *reinterpret_cast<uint32_t*>(&h3));
    }
    *reinterpret_cast<uint2*>(dst + lane * 4) = oa;
    *reinterpret_cast<uint2*>(dst + 128 + lane * 4) = ob;
  } else {
    float xa[8], xb[8];
    unpack8(*reinterpret_cast<const uint4*>(row_smem + lane * 16), xa);
    unpack8(*reinterpret_cast<const uint4*>(row_smem + 512 + lane * 16), xb);
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) ss = fmaf(xa[e], xa[e], fmaf(xb[e], xb[e], ss));
    ss = warp_sum(ss);
    const float inv = 1.0f / sqrtf(ss * (1.0f / 512.0f) + a.eps);
    float ya[8], yb[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float ua = xa[e] * inv * w_lo[e];
      const float ub = xb[e] * inv * w_hi[e];
      ya[e] = ua * c[e] - ub * s[e];
      yb[e] = ub * c[e] + ua * s[e];
    }
    *reinterpret_cast<uint4*>(dst + lane * 8) = pack8(ya);
    *reinterpret_cast<uint4*>(dst + 256 + lane * 8) = pack8(yb);
    if (kind == 1) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        ya[e] = xa[e] * inv;
        yb[e] = xb[e] * inv;
      }
      *reinterpret_cast<uint4*>(vdst + lane * 8) = pack8(ya);
      *reinterpret_cast<uint4*>(vdst + 256 + lane * 8) = pack8(yb);
    }
  }
}

// Stage layout: raw rows [Hq Q rows][Hkv K rows][Hkv V rows (D = 256 only)] of D bf16, then the
// token's rotary row (D/2 fp32 cos, D/2 fp32 sin), then its TokMeta header; stage_bytes is a
// multiple of 128. Shared memory: 2 * nst mbarriers and the abort flag, then the stages.
template <int D>
__global__ void __launch_bounds__(kPrepThreads)
prep_kernel(PrepArgs a, int32_t nst, uint32_t stage_bytes) {
  extern __shared__ __align__(128) unsigned char psm[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int32_t Hq = a.num_qo_heads, Hkv = a.pool.num_kv_heads;
  const int32_t nrows = Hq + (D == 256 ? 2 : 1) * Hkv;
  const uint32_t rows_bytes = (uint32_t)nrows * D * 2;
  const uint32_t hdr_off = rows_bytes + D * 4;
  const uint32_t bars = smem_u32(psm);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(psm + 16 * nst);
  unsigned char* stages = psm + ((16 * nst + 4 + 127) & ~127);
  const uint32_t stages_s = smem_u32(stages);
  auto FULL = [&](int s) { return bars + 8u * s; };
  auto EMPTY = [&](int s) { return bars + 8u * (nst + s); };

  const int32_t T = a.plan.num_tokens, G = gridDim.x;
  const int32_t count = T > (int32_t)blockIdx.x ? (T - 1 - (int32_t)blockIdx.x) / G + 1 : 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < nst; ++s) {
      bar_init(FULL(s), 1);
      bar_init(EMPTY(s), kPrepConsumerWarps);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  if (warp == kPrepConsumerWarps) {
    // ---------------------------------------------------------------- producer
    const uint32_t q_bytes = (uint32_t)Hq * D * 2, kv_bytes = (uint32_t)Hkv * D * 2;
    const uint32_t tok_bytes = rows_bytes + D * 4;
    bool live = true;
    for (int32_t kb = 0; live && kb < count; kb += 32) {
      const int n = min(32, count - kb);
      // lane i resolves the metadata of this CTA's token kb + i
      TokMeta m;
      m.slot = 0;
      m.pos = 0;
      m.ok = 0;
      if (lane < n && !token_meta(a, (int32_t)blockIdx.x + (kb + lane) * G, &m)) {
        m.slot = 0;
        m.pos = 0;
        m.ok = 0;
        atomicOr(a.status, kStatusBounds);
      }
      for (int i = 0; i < n; ++i) {
        const int32_t k = kb + i;
        const int st = k % nst;
        TokMeta mi;
        mi.slot = __shfl_sync(0xffffffffu, m.slot, i);
        mi.pos = __shfl_sync(0xffffffffu, m.pos, i);
        mi.ok = __shfl_sync(0xffffffffu, m.ok, i);
        int go = 1;
        if (lane == 0) {
          // the consumers have released the stage's previous token
          if (!bar_wait(EMPTY(st), ((k / nst) & 1) ^ 1, abort_flag, a.status)) {
            go = 0;
          } else {
            unsigned char* sg = stages + (size_t)st * stage_bytes;
            *reinterpret_cast<TokMeta*>(sg + hdr_off) = mi;
            if (mi.ok) {
              const int32_t t = (int32_t)blockIdx.x + k * G;
              const uint32_t ss = stages_s + (uint32_t)st * stage_bytes;
              bar_arrive_tx(FULL(st), tok_bytes);
              bulk_g2s(ss, a.q_raw + (int64_t)t * a.q_stride, q_bytes, FULL(st));
              bulk_g2s(ss + q_bytes, a.k_raw + (int64_t)t * a.k_stride, kv_bytes, FULL(st));
              if (D == 256)
                bulk_g2s(ss + q_bytes + kv_bytes, a.v_raw + (int64_t)t * a.v_stride, kv_bytes,
                         FULL(st));
              bulk_g2s(ss + rows_bytes, a.rope_cos + (int64_t)mi.pos * (D / 2), D * 2, FULL(st));
              bulk_g2s(ss + rows_bytes + D * 2, a.rope_sin + (int64_t)mi.pos * (D / 2), D * 2,
                       FULL(st));
            } else {
              bar_arrive(FULL(st));  // skipped token: the header says so
            }
          }
        }
        if (!__shfl_sync(0xffffffffu, go, 0)) {
          live = false;
          break;
        }
      }
    }
    if (!live) {
      // copies already issued land within microseconds; let them finish before the CTA's
      // shared memory is released
      const uint64_t t0 = gtimer();
      while (gtimer() - t0 < 100000ull) {
      }
    }
  } else {
    // ---------------------------------------------------------------- consumers
    // this lane's weights (Q and K), loaded once
    float wq_lo[8], wq_hi[8], wk_lo[8], wk_hi[8];
    if (D == 512) {
      const int ci = lane * 8;
      unpack8(__ldg(reinterpret_cast<const uint4*>(a.w_q + ci)), wq_lo);
      unpack8(__ldg(reinterpret_cast<const uint4*>(a.w_k + ci)), wk_lo);
      unpack8(__ldg(reinterpret_cast<const uint4*>(a.w_q + 256 + ci)), wq_hi);
      unpack8(__ldg(reinterpret_cast<const uint4*>(a.w_k + 256 + ci)), wk_hi);
    } else {
      const int ci = lane * 4;
      auto un4 = [](uint2 v, float* f) {
        f[0] = __uint_as_float(v.x << 16); f[1] = __uint_as_float(v.x & 0xFFFF0000u);
        f[2] = __uint_as_float(v.y << 16); f[3] = __uint_as_float(v.y & 0xFFFF0000u);
      };
      un4(__ldg(reinterpret_cast<const uint2*>(a.w_q + ci)), wq_lo);
      un4(__ldg(reinterpret_cast<const uint2*>(a.w_k + ci)), wk_lo);
      un4(__ldg(reinterpret_cast<const uint2*>(a.w_q + 128 + ci)), wq_hi);
      un4(__ldg(reinterpret_cast<const uint2*>(a.w_k + 128 + ci)), wk_hi);
    }
    // rotary column of this lane's first element
    const int rc = D == 256 ? lane * 4 : lane * 8;
    for (int32_t k = 0; k < count; ++k) {
      const int st = k % nst;
      int okw = 1;
      if (lane == 0) okw = bar_wait(FULL(st), (k / nst) & 1, abort_flag, a.status) ? 1 : 0;
      if (!__shfl_sync(0xffffffffu, okw, 0)) break;
      const unsigned char* sg = stages + (size_t)st * stage_bytes;
      const TokMeta m = *reinterpret_cast<const TokMeta*>(sg + hdr_off);
      if (m.ok) {
        const int32_t t = (int32_t)blockIdx.x + k * G;
        float c[8], s[8];
        {
          const float4* cp = reinterpret_cast<const float4*>(sg + rows_bytes) + rc / 4;
          const float4* sp = reinterpret_cast<const float4*>(sg + rows_bytes + D * 2) + rc / 4;
          // D = 256 uses c[0..4), s[0..4) only
          const float4 c0 = cp[0], c1 = D == 512 ? cp[1] : c0, s0 = sp[0], s1 = D == 512 ? sp[1] : s0;
          c[0] = c0.x; c[1] = c0.y; c[2] = c0.z; c[3] = c0.w;
          c[4] = c1.x; c[5] = c1.y; c[6] = c1.z; c[7] = c1.w;
          s[0] = s0.x; s[1] = s0.y; s[2] = s0.z; s[3] = s0.w;
          s[4] = s1.x; s[5] = s1.y; s[6] = s1.z; s[7] = s1.w;
        }
        __nv_bfloat16* const kbase = a.pool.layer_base + m.slot;
        auto do_row = [&](int row) {
          const int kind = row < Hq ? 0 : (row < Hq + Hkv ? 1 : 2);
          __nv_bfloat16* dst;
          __nv_bfloat16* vdst = nullptr;
          if (kind == 0) {
            dst = a.q_out + ((int64_t)t * Hq + row) * D;
          } else if (kind == 1) {
            dst = kbase + (int64_t)(row - Hq) * a.pool.stride_head;
            vdst = dst + a.pool.stride_kv;
          } else {
            dst = kbase + a.pool.stride_kv + (int64_t)(row - Hq - Hkv) * a.pool.stride_head;
          }
          if (kind == 0)
            prep_row<D>(a, sg + (size_t)row * (D * 2), 0, lane, c, s, wq_lo, wq_hi, dst, vdst);
          else
            prep_row<D>(a, sg + (size_t)row * (D * 2), kind, lane, c, s, wk_lo, wk_hi, dst, vdst);
        };
        for (int row = warp; row < nrows; row += kPrepConsumerWarps) do_row(row);
      }
      // every lane's shared-memory reads of this stage are done
      __syncwarp();
      if (lane == 0) bar_arrive(EMPTY(st));
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

// The stages of all CTAs on an SM share about 210 KB of shared memory: the CTAs an SM holds
// (limited by registers) split it, at least two stages each, so every SM keeps ~200 KB of
// copies in flight.
template <int D>
cudaError_t launch_prep(const PrepArgs& a, cudaStream_t stream) {
  const int32_t T = a.plan.num_tokens;
  if (T <= 0) return cudaSuccess;
  const int32_t nrows = a.num_qo_heads + (D == 256 ? 2 : 1) * a.pool.num_kv_heads;
  const uint32_t stage = (uint32_t)((((int64_t)nrows * D * 2 + D * 4 + 16) + 127) & ~(int64_t)127);
  // The shared-memory opt-in is set to the kernel's maximum once per device (it is a
  // process-wide attribute); the stage count and occupancy depend on the device and the stage
  // size and are cached per thread.
  static PerDeviceOnce setup;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = setup.get(dev, [dev](int* n) {
    cudaError_t r = cudaFuncSetAttribute(prep_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         227 * 1024);
    if (r != cudaSuccess) return r;
    return cudaDeviceGetAttribute(n, cudaDevAttrMultiProcessorCount, dev);
  }, &sms);
  if (e != cudaSuccess) return e;
  static thread_local int cached_dev = -1;
  static thread_local uint32_t cached_stage = 0;
  static thread_local int per_sm = 0, nst = 0;
  static thread_local size_t smem = 0;
  if (dev != cached_dev || stage != cached_stage) {
    int by_regs = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&by_regs, prep_kernel<D>, kPrepThreads,
                                                           0)) != cudaSuccess)
      return e;
    if (by_regs < 1) by_regs = 1;
    if (by_regs > 4) by_regs = 4;
    constexpr uint32_t kSmBudget = 210 * 1024;
    int n = (int)(kSmBudget / by_regs / stage);
    if (n < 2) n = 2;
    if (n > 8) n = 8;
    const size_t sm_bytes = (size_t)((16 * n + 4 + 127) & ~127) + (size_t)n * stage;
    if (sm_bytes > 227 * 1024) return cudaErrorInvalidValue;
    int occ = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, prep_kernel<D>, kPrepThreads,
                                                           sm_bytes)) != cudaSuccess)
      return e;
    per_sm = occ < 1 ? 1 : occ;
    nst = n;
    smem = sm_bytes;
    cached_dev = dev;
    cached_stage = stage;
  }
  const int64_t ctas = std::min<int64_t>((int64_t)sms * per_sm, T);
  prep_kernel<D><<<(unsigned)ctas, kPrepThreads, smem, stream>>>(a, nst, stage);
  count_launch();
  return cudaGetLastError();
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
  return launch_prep<256>(a, stream);
}

cudaError_t launch_prep_hd512(const PrepArgs& a, cudaStream_t stream) {
  return launch_prep<512>(a, stream);
}

}  // namespace pg
