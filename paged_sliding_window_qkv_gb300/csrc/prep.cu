// Fused QKV prep: RMSNorm + half-split rotary on Q (contiguous out) and on K, weightless
// RMSNorm on V (never rotated), with K and V scattered straight into the layer's paged
// pool ("gemma4: serving prep needs pool-write forms", Description and Proposed Plan).
//
// HBM-bound single pass, one persistent CTA per (SM, slot) walking the tokens
// t = blockIdx.x + k * gridDim.x. A producer warp streams each token's raw rows (all of its
// Q rows, K rows and V rows are contiguous runs) and its rotary row into a ring of
// shared-memory stages with bulk asynchronous copies (cp.async.bulk, completion counted in
// bytes on the stage's mbarrier), several tokens ahead, so every SM keeps hundreds of KB of
// loads in flight without holding them in registers. Eight consumer warps take the staged
// token's head rows kind by kind, D / 16 lanes per row (two rows per warp at head_dim 256, one
// at 512): a lane reads two 16-byte vectors from shared memory (its elements [8j, 8j + 8) and
// their rotary partners D/2 further), the RMS reduction is a shuffle over the row's lanes, and
// the normalisation, weight and rotation run on packed fp32 pairs, so the consumers stay
// below the issue rate HBM allows. Every result row is written by coalesced 16-byte stores:
// q_out rows, or K/V rows at the token's paged slot (slot = position, wrapped over the
// request's pages for a ring plan, or counted from the segment's first position for a
// key-segment plan). The producer also resolves each token's request, position and page
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

// One staged row, normalised (and for Q/K rows weighted and rotated), stored as bf16. A row is
// handled by LPR = D / 16 lanes (a half warp at D = 256, a warp at D = 512); lane j of the row
// holds its elements [8j, 8j + 8) and their rotary partners [D/2 + 8j, D/2 + 8j + 8), so every
// rotary pair sits in one lane, and the arithmetic runs on packed fp32 pairs (f32x2), one bf16
// round-to-nearest-even at the store.
struct RowIn {
  float2 a[4], b[4];  // elements [8j, 8j + 8) and [D/2 + 8j, D/2 + 8j + 8), in fp32 pairs
};
__device__ __forceinline__ float2 bf2_to_f2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
__device__ __forceinline__ uint32_t f2_to_bf2(float2 v) {
  __nv_bfloat162 h = __float22bfloat162_rn(v);
  return *reinterpret_cast<uint32_t*>(&h);
}
// Loads lane j's 16 elements of a staged row and returns its inverse RMS (the sum of squares is
// reduced over the LPR lanes of the row).
template <int LPR>
__device__ __forceinline__ float load_row(const unsigned char* row_smem, int j, int D2, float inv_d,
                                          float eps, RowIn* x) {
  const uint4 va = *reinterpret_cast<const uint4*>(row_smem + 16 * j);
  const uint4 vb = *reinterpret_cast<const uint4*>(row_smem + D2 + 16 * j);
  x->a[0] = bf2_to_f2(va.x); x->a[1] = bf2_to_f2(va.y); x->a[2] = bf2_to_f2(va.z); x->a[3] = bf2_to_f2(va.w);
  x->b[0] = bf2_to_f2(vb.x); x->b[1] = bf2_to_f2(vb.y); x->b[2] = bf2_to_f2(vb.z); x->b[3] = bf2_to_f2(vb.w);
  float2 ss = __fmul2_rn(x->a[0], x->a[0]);
#pragma unroll
  for (int k = 1; k < 4; ++k) ss = __ffma2_rn(x->a[k], x->a[k], ss);
#pragma unroll
  for (int k = 0; k < 4; ++k) ss = __ffma2_rn(x->b[k], x->b[k], ss);
  float t = ss.x + ss.y;
#pragma unroll
  for (int o = LPR / 2; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  return rsqrtf(t * inv_d + eps);
}
// y = x * inv (weightless, never rotated)
__device__ __forceinline__ void store_plain(const RowIn& x, float inv, __nv_bfloat16* dst, int j,
                                            int D2) {
  const float2 iv = make_float2(inv, inv);
  uint4 oa, ob;
  oa.x = f2_to_bf2(__fmul2_rn(x.a[0], iv)); oa.y = f2_to_bf2(__fmul2_rn(x.a[1], iv));
  oa.z = f2_to_bf2(__fmul2_rn(x.a[2], iv)); oa.w = f2_to_bf2(__fmul2_rn(x.a[3], iv));
  ob.x = f2_to_bf2(__fmul2_rn(x.b[0], iv)); ob.y = f2_to_bf2(__fmul2_rn(x.b[1], iv));
  ob.z = f2_to_bf2(__fmul2_rn(x.b[2], iv)); ob.w = f2_to_bf2(__fmul2_rn(x.b[3], iv));
  *reinterpret_cast<uint4*>(reinterpret_cast<unsigned char*>(dst) + 16 * j) = oa;
  *reinterpret_cast<uint4*>(reinterpret_cast<unsigned char*>(dst) + D2 + 16 * j) = ob;
}
// y = rope(x * inv * w): ya = inv (a wa c - b wb s), yb = inv (b wb c + a wa s); ns = -s
__device__ __forceinline__ void store_rotated(const RowIn& x, float inv, const float2* wa,
                                              const float2* wb, const float2* c, const float2* s,
                                              const float2* ns, __nv_bfloat16* dst, int j, int D2) {
  const float2 iv = make_float2(inv, inv);
  uint32_t ya[4], yb[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 ua = __fmul2_rn(x.a[k], wa[k]), ub = __fmul2_rn(x.b[k], wb[k]);
    ya[k] = f2_to_bf2(__fmul2_rn(__ffma2_rn(ua, c[k], __fmul2_rn(ub, ns[k])), iv));
    yb[k] = f2_to_bf2(__fmul2_rn(__ffma2_rn(ub, c[k], __fmul2_rn(ua, s[k])), iv));
  }
  *reinterpret_cast<uint4*>(reinterpret_cast<unsigned char*>(dst) + 16 * j) =
      make_uint4(ya[0], ya[1], ya[2], ya[3]);
  *reinterpret_cast<uint4*>(reinterpret_cast<unsigned char*>(dst) + D2 + 16 * j) =
      make_uint4(yb[0], yb[1], yb[2], yb[3]);
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
    // LPR lanes per row: a warp holds 32 / LPR rows at a time (RPW), lane j = lane % LPR of
    // row `sub` = lane / LPR. Rows are taken kind by kind (Q rows, then K rows, then the V rows
    // of head_dim 256), RPW rows per warp at a time.
    constexpr int LPR = D / 16, RPW = 32 / LPR, D2 = D;  // D2: bytes of half a row
    const int j = lane % LPR, sub = lane / LPR;
    const float inv_d = 1.0f / (float)D;
    // this lane's weights (Q and K) as fp32 pairs, loaded once
    float2 wqa[4], wqb[4], wka[4], wkb[4];
    {
      const uint4 qa = __ldg(reinterpret_cast<const uint4*>(a.w_q) + j);
      const uint4 qb = __ldg(reinterpret_cast<const uint4*>(a.w_q + D / 2) + j);
      const uint4 ka = __ldg(reinterpret_cast<const uint4*>(a.w_k) + j);
      const uint4 kb = __ldg(reinterpret_cast<const uint4*>(a.w_k + D / 2) + j);
      wqa[0] = bf2_to_f2(qa.x); wqa[1] = bf2_to_f2(qa.y); wqa[2] = bf2_to_f2(qa.z); wqa[3] = bf2_to_f2(qa.w);
      wqb[0] = bf2_to_f2(qb.x); wqb[1] = bf2_to_f2(qb.y); wqb[2] = bf2_to_f2(qb.z); wqb[3] = bf2_to_f2(qb.w);
      wka[0] = bf2_to_f2(ka.x); wka[1] = bf2_to_f2(ka.y); wka[2] = bf2_to_f2(ka.z); wka[3] = bf2_to_f2(ka.w);
      wkb[0] = bf2_to_f2(kb.x); wkb[1] = bf2_to_f2(kb.y); wkb[2] = bf2_to_f2(kb.z); wkb[3] = bf2_to_f2(kb.w);
    }
    const int cw = warp;  // consumer warp index, 0..7
    for (int32_t k = 0; k < count; ++k) {
      const int st = k % nst;
      int okw = 1;
      if (lane == 0) okw = bar_wait(FULL(st), (k / nst) & 1, abort_flag, a.status) ? 1 : 0;
      if (!__shfl_sync(0xffffffffu, okw, 0)) break;
      const unsigned char* sg = stages + (size_t)st * stage_bytes;
      const TokMeta m = *reinterpret_cast<const TokMeta*>(sg + hdr_off);
      if (m.ok) {
        const int32_t t = (int32_t)blockIdx.x + k * G;
        // this token's rotary coefficients for the lane's 8 pairs
        float2 c[4], sn[4], ns[4];
        {
          const float4* cp = reinterpret_cast<const float4*>(sg + rows_bytes) + 2 * j;
          const float4* sp = reinterpret_cast<const float4*>(sg + rows_bytes + D * 2) + 2 * j;
          const float4 c0 = cp[0], c1 = cp[1], s0 = sp[0], s1 = sp[1];
          c[0] = make_float2(c0.x, c0.y); c[1] = make_float2(c0.z, c0.w);
          c[2] = make_float2(c1.x, c1.y); c[3] = make_float2(c1.z, c1.w);
          sn[0] = make_float2(s0.x, s0.y); sn[1] = make_float2(s0.z, s0.w);
          sn[2] = make_float2(s1.x, s1.y); sn[3] = make_float2(s1.z, s1.w);
#pragma unroll
          for (int e = 0; e < 4; ++e) ns[e] = make_float2(-sn[e].x, -sn[e].y);
        }
        __nv_bfloat16* const kbase = a.pool.layer_base + m.slot;
        // Q rows
        for (int r0 = cw * RPW; r0 < Hq; r0 += kPrepConsumerWarps * RPW) {
          const int r = r0 + sub;
          const bool live = r < Hq;
          RowIn x;
          const float inv = load_row<LPR>(sg + (size_t)(live ? r : r0) * (D * 2), j, D2, inv_d, a.eps, &x);
          if (live)
            store_rotated(x, inv, wqa, wqb, c, sn, ns, a.q_out + ((int64_t)t * Hq + r) * D, j, D2);
        }
        // K rows (head_dim 512: and the V row, the weightless norm of the same raw K)
        for (int r0 = cw * RPW; r0 < Hkv; r0 += kPrepConsumerWarps * RPW) {
          const int r = r0 + sub;
          const bool live = r < Hkv;
          RowIn x;
          const float inv =
              load_row<LPR>(sg + (size_t)(Hq + (live ? r : r0)) * (D * 2), j, D2, inv_d, a.eps, &x);
          if (live) {
            __nv_bfloat16* dst = kbase + (int64_t)r * a.pool.stride_head;
            store_rotated(x, inv, wka, wkb, c, sn, ns, dst, j, D2);
            if (D == 512) store_plain(x, inv, dst + a.pool.stride_kv, j, D2);
          }
        }
        // V rows of head_dim 256 (weightless, never rotated)
        if (D == 256) {
          for (int r0 = cw * RPW; r0 < Hkv; r0 += kPrepConsumerWarps * RPW) {
            const int r = r0 + sub;
            const bool live = r < Hkv;
            RowIn x;
            const float inv = load_row<LPR>(sg + (size_t)(Hq + Hkv + (live ? r : r0)) * (D * 2), j,
                                            D2, inv_d, a.eps, &x);
            if (live) store_plain(x, inv, kbase + a.pool.stride_kv + (int64_t)r * a.pool.stride_head, j, D2);
          }
        }
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
