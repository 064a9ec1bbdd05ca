// Paged prefill attention on the 5th-generation tensor cores (tcgen05 + TMEM + TMA)
// ("feat(kernels): Rust wrapper for the hd256 windowed paged prefill", Description:
// paged reads, explicit sm_scale, inclusive-distance window_left, GQA by integer
// division; "feat(gemma4): paged KV serving across both attention families",
// Description: hd256 local layers with a sliding window, hd512 global layers causal).
//
// One CTA owns a 128-row query tile that packs the GQA group of one KV head (rows are
// token-major, head-minor, exactly the order a 3-D TMA box of q[token][head][d] lands
// in shared memory) and walks the 64-key tiles of its visible key range, skipping
// tiles outside the causal window.
//
//   warp 0      producer: TMA loads of Q (once) and of K/V page rows into a ring of
//               32 KB slots, one box per (page, 64-wide d chunk), 128B-swizzled;
//   warp 1      MMA issuer (one thread): S = Q K^T into TMEM (M=128, N=64, K=16 steps,
//               both operands from shared memory), then O += P V with P read from TMEM
//               (M=128, N=256, K=16 steps); completion is signalled with tcgen05.commit;
//   warps 2..5  softmax: one thread per query row, S row read from TMEM, masked, online
//               softmax in log2 units with lazy rescaling (O is rescaled in TMEM only
//               when a row maximum grows by more than 2^8), P written back to TMEM as
//               bf16; then the epilogue normalises O and stores bf16 rows.
//
// TMEM (512 columns): O [0,256) fp32, S double buffer [256,384), P double buffer
// [384,448). O holds 256 output columns: for head_dim 512 each query tile runs as two
// CTAs (grid z), each computing the full 512-wide S and half of O.
//
// Every wait is bounded (two seconds of %globaltimer); a wait that runs out sets the
// device status word, makes the CTA drain and free its tensor memory, and return.
#include "pg_internal.h"

#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>

#include <mutex>

namespace pg {
namespace {

constexpr int kM = 128;            // query rows per CTA
constexpr int kBN = 64;            // keys per KV tile
constexpr int kDV = 256;           // output columns per CTA
constexpr int kSlotBytes = kBN * 256 * 2;  // 64 keys x 256 d bf16 = 32 KB
constexpr int kThreadsTc = 192;
constexpr uint32_t kTmO = 0, kTmS = 256, kTmP = 384;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

template <int DQK>
struct TcCfg {
  static constexpr int PARTS = DQK / 256 + 1;  // K slots + one V slot per tile
  static constexpr int NS = DQK == 256 ? 5 : 3;
  static constexpr int Q_BYTES = kM * DQK * 2;
  static constexpr int SMEM_DATA = Q_BYTES + NS * kSlotBytes;
  static constexpr int NBAR = 2 * NS + 11;
  static constexpr int SMEM = SMEM_DATA + NBAR * 8 + 16 + 1024;  // + barriers, tmem addr, align
};

struct TcArgs {
  PlanDev plan;
  __nv_bfloat16* out;
  int32_t num_qo_heads, group, cta_tile_q, window_left;
  int32_t page_size, num_pages, num_kv_heads, box_rows;
  float scale_log2;
  int* status;
};

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait on the phase of the given parity. Returns false when the CTA is aborting
// (another role gave up) or when this wait itself runs out of time.
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                       int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer() - t0 > kWaitLimitNs) {
      atomicOr(status, kStatusTimeout);
      *abort_flag = 1;
      return false;
    }
  }
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(tm), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* tm, int x, int y,
                                            int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(tm), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                       uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

#define PG_R8(b) "=r"(r[b + 0]), "=r"(r[b + 1]), "=r"(r[b + 2]), "=r"(r[b + 3]), \
                 "=r"(r[b + 4]), "=r"(r[b + 5]), "=r"(r[b + 6]), "=r"(r[b + 7])
#define PG_W8(b) "r"(r[b + 0]), "r"(r[b + 1]), "r"(r[b + 2]), "r"(r[b + 3]), \
                 "r"(r[b + 4]), "r"(r[b + 5]), "r"(r[b + 6]), "r"(r[b + 7])

// 32 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : PG_R8(0), PG_R8(8), PG_R8(16), PG_R8(24)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      PG_W8(0), PG_W8(8), PG_W8(16), PG_W8(24)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle. lbo/sbo in bytes.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version
  d |= (uint64_t)2 << 61;  // 128-byte swizzle
  return d;
}
// Instruction descriptor, kind::f16: bf16 A and B, fp32 accumulate.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// ------------------------------------------------------------------ kernel
template <int DQK>
__global__ void __launch_bounds__(kThreadsTc, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kv,
               TcArgs a) {
  using C = TcCfg<DQK>;
  constexpr int PARTS = C::PARTS, NS = C::NS;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* gbase = smem_raw + (base - raw);
  const uint32_t sQ = base;
  const uint32_t sSlots = base + C::Q_BYTES;
  const uint32_t bars = base + C::SMEM_DATA;
  auto FULL = [&](int s) { return bars + 8u * s; };
  auto EMPTY = [&](int s) { return bars + 8u * (NS + s); };
  const uint32_t SFULL = bars + 8u * (2 * NS), SFREE = SFULL + 16, PFULL = SFULL + 32,
                 PVDONE = SFULL + 48, QFULL = SFULL + 64, FIXB = SFULL + 72,
                 DRAIN = SFULL + 80;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::SMEM_DATA + C::NBAR * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const PlanDev& pl = a.plan;
  // longest work first: the plan lists each request's query tiles in token order
  const int32_t item = pl.num_work - 1 - (int32_t)blockIdx.x;
  const int32_t g = blockIdx.y, dh = blockIdx.z;
  const int32_t r = pl.work_req[item], tok0 = pl.work_tok0[item];
  const int32_t G = a.group, Hq = a.num_qo_heads;
  const int32_t q0 = pl.qo_indptr[r];
  const int32_t ntok = min(a.cta_tile_q, pl.qo_indptr[r + 1] - q0 - tok0);
  const int32_t kvp0 = pl.kv_page_indptr[r], kvp1 = pl.kv_page_indptr[r + 1];
  const int32_t ps = a.page_size;
  const int32_t kv_len = (kvp1 - kvp0 - 1) * ps + pl.last_page_len[r];
  const int32_t sp = pl.start_pos[r];
  const int32_t W = a.window_left;
  const int32_t p_first = sp + tok0, p_last = sp + tok0 + ntok - 1;
  const int32_t lo = W >= 0 ? max(0, p_first - W) : 0;
  const int32_t hi = min(p_last + 1, kv_len);
  const int32_t kb0 = lo & ~(kBN - 1);
  const int32_t ntiles = hi > kb0 ? (hi - kb0 + kBN - 1) / kBN : 0;

  // a CTA that finds an earlier CTA timed out returns at once (uniformly, before TMEM)
  if (threadIdx.x == 0) *abort_flag = *reinterpret_cast<volatile int*>(a.status) & kStatusTimeout;
  __syncthreads();
  if (*abort_flag) return;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(FULL(s), 1);
      mbar_init(EMPTY(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(SFULL + 8 * b, 1);
      mbar_init(SFREE + 8 * b, 4);
      mbar_init(PFULL + 8 * b, 4);
      mbar_init(PVDONE + 8 * b, 1);
    }
    mbar_init(QFULL, 1);
    mbar_init(FIXB, 1);
    mbar_init(DRAIN, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int issued = 0;
    uint32_t fix_phase = 0;
    bool ok = true;
    if (lane == 0) {
      mbar_expect_tx(QFULL, C::Q_BYTES);
      for (int c = 0; c < DQK / 64; ++c)
        tma_load_3d(sQ + c * (kM * 128), &tm_q, c * 64, g * G, q0 + tok0, QFULL);
    }
    const int BR = a.box_rows;          // rows per TMA box: min(page_size, 64)
    const int nbox = kBN / BR;          // boxes per 64-key tile per d chunk
    const int64_t head_rows = (int64_t)ps;
    for (int32_t j = 0; j < ntiles && ok; ++j) {
      const int32_t kb = kb0 + j * kBN;
      // page rows of this tile, checked against the pool (second layer of defence)
      int32_t row_k = -1;   // lane b < nbox: tensor row of box b's first K row, or -1
      bool bad = false;
      if (lane < nbox) {
        const int32_t ks = kb + lane * BR;
        if (ks < kv_len) {
          const int32_t pidx = kvp0 + ks / ps;
          const int32_t page = (pidx < kvp1 && pidx < pl.num_page_ids) ? pl.page_ids[pidx] : -1;
          if (page < 0 || page >= a.num_pages) {
            bad = true;
          } else {
            row_k = (int32_t)((((int64_t)page * 2) * a.num_kv_heads + g) * head_rows + (ks % ps));
          }
        }
      }
      const bool any_bad = __any_sync(0xffffffffu, bad);
      if (any_bad && lane == 0) atomicOr(a.status, kStatusBounds);
      const bool fix = any_bad || (kb + kBN > kv_len);
      for (int pp = 0; pp < PARTS; ++pp) {
        const int part = j * PARTS + pp;
        const int s = part % NS;
        if (!__all_sync(0xffffffffu, mbar_wait(EMPTY(s), ((part / NS) & 1) ^ 1, abort_flag, a.status))) {
          ok = false;
          break;
        }
        const bool is_v = pp == PARTS - 1;
        const int d0 = is_v ? dh * 256 : pp * 256;
        // V rows sit Hkv head-blocks after the K rows of the same page
        const int32_t vshift = is_v ? (int32_t)(a.num_kv_heads * head_rows) : 0;
        int nloaded = __popc(__ballot_sync(0xffffffffu, lane < nbox && row_k >= 0));
        const uint32_t bytes = (uint32_t)nloaded * 4u * BR * 128u;
        const uint32_t slot = sSlots + s * kSlotBytes;
        const uint32_t bar = fix ? FIXB : FULL(s);
        if (lane == 0 && bytes > 0) mbar_expect_tx(bar, bytes);
        __syncwarp();
        if (lane < nbox && row_k >= 0) {
          for (int c = 0; c < 4; ++c)
            tma_load_2d(slot + c * (kBN * 128) + lane * BR * 128, &tm_kv, d0 + c * 64,
                        row_k + vshift, bar);
        }
        ++issued;
        if (fix) {
          if (bytes > 0) {
            if (!__all_sync(0xffffffffu, mbar_wait(FIXB, fix_phase, abort_flag, a.status))) {
              ok = false;
              break;
            }
            fix_phase ^= 1u;
          }
          // zero the rows of keys the tile must not read: past kv_len or on a bad page
          for (int k = 0; k < kBN; ++k) {
            const int b = k / BR;
            const int32_t rb = __shfl_sync(0xffffffffu, row_k, b);
            if (kb + k < kv_len && rb >= 0) continue;
            // 4 chunks x 128 bytes = 32 lanes x 16 bytes
            const int c = lane >> 3, w16 = lane & 7;
            uint4* p = reinterpret_cast<uint4*>(gbase + (slot - base) + c * (kBN * 128) + k * 128) + w16;
            *p = make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async();
          __syncwarp();
          if (lane == 0) mbar_arrive(FULL(s));
        }
      }
    }
    if (!ok) {
      // drain: let every load this warp issued land before the CTA frees its memory
      for (int p = max(0, issued - NS); p < issued; ++p) {
        const int s = p % NS;
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(FULL(s), (p / NS) & 1) && globaltimer() - t0 < kWaitLimitNs) {
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_QK = idesc_bf16(kM, kBN, false);
      constexpr uint32_t IDESC_PV = idesc_bf16(kM, kDV, true);
      bool ok = mbar_wait(QFULL, 0, abort_flag, a.status);
      for (int32_t j = 0; ok && j <= ntiles; ++j) {
        if (j < ntiles) {
          const int b = j & 1, u = j >> 1;
          ok = mbar_wait(SFREE + 8 * b, (u & 1) ^ 1, abort_flag, a.status);
          uint32_t kslot[PARTS - 1];
          for (int pp = 0; ok && pp < PARTS - 1; ++pp) {
            const int part = j * PARTS + pp;
            kslot[pp] = sSlots + (part % NS) * kSlotBytes;
            ok = mbar_wait(FULL(part % NS), (part / NS) & 1, abort_flag, a.status);
          }
          if (!ok) break;
          tc_fence_after();
          const uint32_t dS = tmem + kTmS + b * kBN;
#pragma unroll 4
          for (int kk = 0; kk < DQK / 16; ++kk) {
            const uint32_t qa = sQ + (kk >> 2) * (kM * 128) + (kk & 3) * 32;
            const int kin = kk & 15;
            const uint32_t ka = kslot[kk >> 4] + (kin >> 2) * (kBN * 128) + (kin & 3) * 32;
            mma_ss(dS, sdesc(qa, 16, 1024), sdesc(ka, 16, 1024), IDESC_QK, kk > 0 ? 1u : 0u);
          }
          mma_commit(SFULL + 8 * b);
          for (int pp = 0; pp < PARTS - 1; ++pp) mma_commit(EMPTY((j * PARTS + pp) % NS));
        }
        if (j >= 1) {
          const int32_t jp = j - 1;
          const int b = jp & 1, u = jp >> 1;
          const int part = jp * PARTS + PARTS - 1;
          const int s = part % NS;
          ok = mbar_wait(FULL(s), (part / NS) & 1, abort_flag, a.status) &&
               mbar_wait(PFULL + 8 * b, u & 1, abort_flag, a.status);
          if (!ok) break;
          tc_fence_after();
          const uint32_t vs = sSlots + s * kSlotBytes;
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk) {
            mma_ts(tmem + kTmO, tmem + kTmP + b * (kBN / 2) + kk * 8,
                   sdesc(vs + kk * 2048, kBN * 128, 1024), IDESC_PV, (jp > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(EMPTY(s));
          mma_commit(PVDONE + 8 * b);
        }
      }
      // arrives once every MMA this thread issued has completed; waited on before TMEM is freed
      mma_commit(DRAIN);
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
    const bool rvalid = row < ntok * G;
    const int32_t prow = sp + tok0 + row / G;
    const int32_t rlo = W >= 0 ? max(0, prow - W) : 0;
    const int32_t rhi = min(prow + 1, kv_len);
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int32_t j = 0; ok && j < ntiles; ++j) {
      const int b = j & 1, u = j >> 1;
      if (!__all_sync(0xffffffffu, mbar_wait(SFULL + 8 * b, u & 1, abort_flag, a.status))) { ok = false; break; }
      tc_fence_after();
      uint32_t sv[kBN];
      tmem_ld32(tl + kTmS + b * kBN, sv);
      tmem_ld32(tl + kTmS + b * kBN + 32, sv + 32);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(SFREE + 8 * b);
      const int32_t kb = kb0 + j * kBN;
      float s[kBN];
      float mx = -INFINITY;
#pragma unroll
      for (int k = 0; k < kBN; ++k) {
        const int32_t key = kb + k;
        const bool vis = rvalid && key >= rlo && key < rhi;
        s[k] = vis ? __uint_as_float(sv[k]) * a.scale_log2 : -INFINITY;
        mx = fmaxf(mx, s[k]);
      }
      float alpha = 1.f;
      bool resc = false;
      if (mx > m_ref + 8.f) {
        alpha = m_ref == -INFINITY ? 0.f : exp2f(m_ref - mx);
        resc = m_ref != -INFINITY;
        l *= alpha;
        m_ref = mx;
      }
      if (j > 0 && __any_sync(0xffffffffu, resc)) {
        const int jp = j - 1;
        if (!__all_sync(0xffffffffu, mbar_wait(PVDONE + 8 * (jp & 1), (jp >> 1) & 1, abort_flag, a.status))) { ok = false; break; }
        tc_fence_after();
        for (int c = 0; c < kDV / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tl + kTmO + c * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(tl + kTmO + c * 32, o);
        }
        tmem_wait_st();
      }
      const float mu = m_ref == -INFINITY ? 0.f : m_ref;
      float sum = 0.f;
      uint32_t pk[kBN / 2];
#pragma unroll
      for (int k = 0; k < kBN / 2; ++k) {
        const float p0 = exp2f(s[2 * k] - mu), p1 = exp2f(s[2 * k + 1] - mu);
        sum += p0 + p1;
        pk[k] = pack_bf16(p0, p1);
      }
      l += sum;
      if (j >= 2 && !__all_sync(0xffffffffu, mbar_wait(PVDONE + 8 * b, ((j >> 1) & 1) ^ 1, abort_flag, a.status))) { ok = false; break; }
      tc_fence_after();
      tmem_st32(tl + kTmP + b * (kBN / 2), pk);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(PFULL + 8 * b);
    }
    if (ok && ntiles > 0) {
      const int jl = ntiles - 1;
      ok = __all_sync(0xffffffffu, mbar_wait(PVDONE + 8 * (jl & 1), (jl >> 1) & 1, abort_flag, a.status));
    }
    if (ok) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16* dst = a.out + ((int64_t)(q0 + tok0 + row / G) * Hq + g * G + row % G) * DQK +
                           dh * kDV;
      for (int c = 0; c < kDV / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tl + kTmO + c * 32, o);
        tmem_wait_ld();
        if (ntiles == 0) {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0u;
        }
        if (rvalid) {
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            w[e] = pack_bf16(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
          uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
          d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
          d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
          d4[2] = make_uint4(w[8], w[9], w[10], w[11]);
          d4[3] = make_uint4(w[12], w[13], w[14], w[15]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1 && lane == 0) {
    // every MMA has completed once the final commit has arrived
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(DRAIN, 0) && globaltimer() - t0 < kWaitLimitNs) {
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

template <int DQK>
cudaError_t launch_tc(const AttnArgs& a, cudaStream_t stream) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const int32_t G = a.group, TQ = a.cta_tile_q;
  CUtensorMap tq, tkv;
  {
    cuuint64_t dims[3] = {(cuuint64_t)DQK, (cuuint64_t)a.num_qo_heads,
                          (cuuint64_t)a.plan.num_tokens};
    cuuint64_t strides[2] = {(cuuint64_t)DQK * 2, (cuuint64_t)a.num_qo_heads * DQK * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)TQ};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, (void*)a.q, dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const int32_t ps = a.pool.page_size;
  const int32_t br = ps < 64 ? ps : 64;
  {
    const cuuint64_t rows = (cuuint64_t)a.pool.num_pages * 2 * a.pool.num_kv_heads * ps;
    cuuint64_t dims[2] = {(cuuint64_t)DQK, rows};
    cuuint64_t strides[1] = {(cuuint64_t)DQK * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)br};
    cuuint32_t es[2] = {1, 1};
    if (enc(&tkv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (void*)a.pool.layer_base, dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  TcArgs t;
  t.plan = a.plan;
  t.out = a.out;
  t.num_qo_heads = a.num_qo_heads;
  t.group = G;
  t.cta_tile_q = TQ;
  t.window_left = a.window_left;
  t.page_size = ps;
  t.num_pages = a.pool.num_pages;
  t.num_kv_heads = a.pool.num_kv_heads;
  t.box_rows = br;
  t.scale_log2 = a.sm_scale_log2;
  t.status = a.status;

  static bool configured[128] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(attn_tc_kernel<DQK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             TcCfg<DQK>::SMEM);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  dim3 grid(a.plan.num_work, a.pool.num_kv_heads, DQK / kDV);
  attn_tc_kernel<DQK><<<grid, kThreadsTc, TcCfg<DQK>::SMEM, stream>>>(tq, tkv, t);
  count_launch();
  return cudaGetLastError();
}

}  // namespace

bool attn_tc_supported(int32_t head_dim, int32_t group, int32_t page_size) {
  if (head_dim != 256 && head_dim != 512) return false;
  if (group <= 0 || kM % group != 0) return false;
  if (page_size < 8 || (page_size & (page_size - 1)) != 0) return false;
  return true;
}

cudaError_t launch_attn_prefill_tc(const AttnArgs& a, int32_t head_dim, cudaStream_t stream) {
  if (a.plan.num_work == 0) return cudaSuccess;
  return head_dim == 256 ? launch_tc<256>(a, stream) : launch_tc<512>(a, stream);
}

int32_t attn_tc_rows() { return kM; }

}  // namespace pg
