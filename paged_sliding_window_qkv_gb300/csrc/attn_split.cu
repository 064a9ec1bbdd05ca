// Paged attention over a page table with an inclusive-distance sliding window
// ("feat(kernels): Rust wrapper for the hd256 windowed paged prefill", Description;
// "feat(gemma4): paged KV serving across both attention families", Description).
//
// One CTA owns BM query rows that share one KV head (GQA: rows are (token, head)
// pairs of the head group, so each K/V tile is loaded once for the whole group) and
// walks the KV tiles of its visible key range. K/V rows are gathered row by row (one page
// lookup per key row; ring plans wrap the page index, key-segment plans offset it by the
// segment's first position) with cp.async into XOR-swizzled shared memory through NS
// stages. S = Q K^T and O += P V run on bf16 mma.sync with fp32 accumulation; the online
// softmax runs in fp32 in log2 units, and the row's log-sum-exp is written when asked.
//
// Two grid forms share the kernel:
//   prefill: one CTA per (work item = request x query tile, KV head);
//   decode (every request has one query token): one CTA per (request, KV head, key
//   chunk); each chunk writes a partial (o, m, l) and a merge kernel combines them.
//   A request whose visible keys fit one chunk is written directly.
#include "pg_internal.h"
#include "../../include/pg.h"

#include <cuda_bf16.h>
#include <math.h>

#include <mutex>

namespace pg {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = 8;
constexpr float kLn2 = 0.69314718055994531f;  // log2 units to natural log

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float* c, const uint32_t* a, const uint32_t* b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// Byte offset of 16-byte chunk c of row m in a [rows][D] bf16 tile, chunks XOR-swizzled
// by the row's low three bits so 8 consecutive rows of one chunk hit distinct banks.
template <int D>
__device__ __forceinline__ uint32_t swz(int m, int c) {
  return (uint32_t)(m * (D * 2) + ((c ^ (m & 7)) << 4));
}

template <int D_, int BM_, int BN_, int NT_, int KS_, bool DECODE_, int NS_ = 2>
struct Cfg {
  static constexpr int D = D_, BM = BM_, BN = BN_, NT = NT_, KS = KS_;
  static constexpr int NS = NS_;  // K/V tile stages: NS - 1 tiles in flight while one computes
  static constexpr bool DECODE = DECODE_;
  static constexpr int CH = D / 8;                 // 16-byte chunks per row
  // S = Q K^T warp tiling: (BM/16) m-tiles x (BN/8/NT) n-groups x KS k-splits = 8 warps
  static constexpr int WM = BM / 16;
  static constexpr int WN = BN / 8 / NT;
  static_assert(WM * WN * KS == kWarps, "S tiling must use all warps");
  static constexpr int KSTEPS = D / 16 / KS;
  // O = P V warp tiling: (BM/16) m-tiles x WNO column groups
  static constexpr int WNO = kWarps / WM;
  static constexpr int DCOLS = D / WNO;
  static constexpr int NTO = DCOLS / 8;
  static_assert(NTO % 2 == 0, "PV loads two n-tiles per ldmatrix");
  static constexpr int SLD = BN + 4;   // fp32 S row stride (floats)
  static constexpr int PLD = BN + 8;   // bf16 P row stride (elements)
  static constexpr int TPR = kThreads / BM;  // softmax threads per row
  static constexpr int VPT = BN / TPR;       // softmax values per thread
  static_assert(VPT % 2 == 0, "softmax reads float2 pairs");
  static constexpr size_t Q_BYTES = (size_t)BM * D * 2;
  static constexpr size_t KV_BYTES = (size_t)BN * D * 2;
  static constexpr size_t S_BYTES = (size_t)KS * BM * SLD * 4;
  static constexpr size_t P_BYTES = (size_t)BM * PLD * 2;
  static constexpr size_t SMEM = Q_BYTES + 2 * NS * KV_BYTES + S_BYTES + P_BYTES + 2 * BM * 4;
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

template <class C>
__global__ void __launch_bounds__(kThreads, C::D == 256 ? 2 : 1)
attn_split_kernel(AttnArgs a) {
  constexpr int D = C::D, BM = C::BM, BN = C::BN;
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* sQ = smem;
  unsigned char* sK = sQ + C::Q_BYTES;               // NS stages
  unsigned char* sV = sK + C::NS * C::KV_BYTES;      // NS stages
  float* sS = reinterpret_cast<float*>(sV + C::NS * C::KV_BYTES);
  __nv_bfloat16* sP = reinterpret_cast<__nv_bfloat16*>(reinterpret_cast<unsigned char*>(sS) + C::S_BYTES);
  float* sAlpha = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(sP) + C::P_BYTES);
  float* sL = sAlpha + BM;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const PlanDev& pl = a.plan;
  const int32_t G = a.group, Hq = a.num_qo_heads, g = blockIdx.y;

  int32_t r, tok0, ntok, chunk = 0;
  if (C::DECODE) {
    r = blockIdx.x;
    tok0 = 0;
    ntok = 1;
    chunk = blockIdx.z;
  } else {
    r = pl.work_req[blockIdx.x];
    tok0 = pl.work_tok0[blockIdx.x];
    ntok = 0;
  }
  const int32_t q0 = pl.qo_indptr[r];
  const int32_t qo_len = pl.qo_indptr[r + 1] - q0;
  if (!C::DECODE) ntok = min(a.cta_tile_q, qo_len - tok0);
  const int32_t kvp0 = pl.kv_page_indptr[r], kvp1 = pl.kv_page_indptr[r + 1];
  const int32_t ps = a.pool.page_size;
  const int32_t sp = pl.start_pos[r];
  const int32_t ks0 = pl.kv_start[r];  // first key position held (a key segment's start)
  // ring addressing (window-crossing requests): every position below start + qo_len is held
  const int32_t kv_len =
      pl.ring ? sp + qo_len : ks0 + (kvp1 - kvp0 - 1) * ps + pl.last_page_len[r];
  const int32_t p_first = sp + tok0, p_last = sp + tok0 + ntok - 1;
  const int32_t W = a.window_left;
  int32_t lo = W >= 0 ? max(ks0, p_first - W) : ks0;
  int32_t hi = min(p_last + 1, kv_len);
  int32_t nchunks = 1;
  if (C::DECODE) {
    nchunks = (hi - lo + a.kv_chunk - 1) / a.kv_chunk;
    // a row that sees no key (possible in a key segment) is still written, by chunk 0
    if (chunk >= max(nchunks, 1)) return;
    lo = lo + chunk * a.kv_chunk;
    hi = min(hi, lo + a.kv_chunk);
  }

  // ---- Q tile (rows beyond the tile's tokens are zero) ----
  {
    const uint32_t base = smem_u32(sQ);
    for (int idx = tid; idx < BM * C::CH; idx += kThreads) {
      const int m = idx / C::CH, c = idx % C::CH;
      const int tl = m / G;
      const bool valid = (m < ntok * G);
      const __nv_bfloat16* src =
          a.q + (valid ? ((int64_t)(q0 + tok0 + tl) * Hq + g * G + (m % G)) * D + c * 8 : 0);
      cp_async16(base + swz<D>(m, c), src, valid);
    }
  }
  const __nv_bfloat16* kv_base = a.pool.layer_base + (int64_t)g * a.pool.stride_head;
  // each thread copies the chunks c0, c0 + TPK, ... of one key row: one page lookup per row,
  // and the TPK threads of a row move consecutive 16-byte chunks
  constexpr int TPK = kThreads / BN;  // threads per key row
  static_assert(kThreads % BN == 0 && C::CH % TPK == 0, "key-row copy split");
  // A tile's row copies are issued in two steps: the page lookup of the thread's row (a load
  // of its page id, issued one tile ahead so that its latency overlaps a tile of compute), then
  // the checks and the copies.
  struct RowAt {
    int32_t page, off;  // page id as loaded, row within the page; off < 0: no key of the request
  };
  const int jj = tid / TPK, c0 = tid % TPK;
  auto row_fetch = [&](int32_t kb) {
    RowAt r{-1, -1};
    const int32_t j = kb + jj;
    if (j < hi) {
      const int32_t rel = j - ks0;  // index among the keys held
      const int32_t lp = rel / ps;  // logical page; ring addressing wraps it over the pages held
      const int32_t pidx = kvp0 + (pl.ring ? lp % max(kvp1 - kvp0, 1) : lp);
      r.off = rel - lp * ps;
      r.page = pidx < kvp1 ? pl.page_ids[pidx] : -1;
    }
    return r;
  };
  auto row_issue = [&](int stage, RowAt r) {
    const uint32_t bk = smem_u32(sK + stage * C::KV_BYTES);
    const uint32_t bv = smem_u32(sV + stage * C::KV_BYTES);
    bool valid = r.off >= 0;
    const __nv_bfloat16* src = a.pool.layer_base;
    if (valid) {
      if (r.page < 0 || r.page >= a.pool.num_pages) {
        if (c0 == 0) atomicOr(a.status, kStatusBounds);
        valid = false;
      } else {
        src = kv_base + (int64_t)r.page * a.pool.stride_page + (int64_t)r.off * D;
      }
    }
#pragma unroll
    for (int c = c0; c < C::CH; c += TPK) {
      cp_async16(bk + swz<D>(jj, c), src + (valid ? c * 8 : 0), valid);
      cp_async16(bv + swz<D>(jj, c), src + (valid ? a.pool.stride_kv + c * 8 : 0), valid);
    }
  };

  const int32_t ntiles = (hi - lo + BN - 1) / BN;
  // the first NS - 1 tiles (one commit group each; Q rides in the first), their lookups first
  {
    RowAt first[C::NS - 1];
#pragma unroll
    for (int st = 0; st < C::NS - 1; ++st) first[st] = row_fetch(lo + st * BN);
#pragma unroll
    for (int st = 0; st < C::NS - 1; ++st) {
      if (st < ntiles) row_issue(st, first[st]);
      cp_async_commit();
    }
  }
  RowAt pend = row_fetch(lo + (C::NS - 1) * BN);  // the tile the first iteration loads

  // S-warp coordinates
  const int s_mt = warp % C::WM;
  const int s_ng = (warp / C::WM) % C::WN;
  const int s_ks = warp / (C::WM * C::WN);
  // PV-warp coordinates
  const int o_mt = warp % C::WM;
  const int o_cg = warp / C::WM;
  // softmax coordinates
  const int sm_row = tid / C::TPR, sm_sub = tid % C::TPR;
  const int sm_tl = sm_row / G;
  const bool sm_valid = sm_row < ntok * G;
  const int32_t sm_pos = sp + tok0 + sm_tl;
  float row_m = -INFINITY, row_l = 0.f;

  float o[C::NTO][4];
#pragma unroll
  for (int i = 0; i < C::NTO; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  // a warp whose k-split spans at most 8 k-steps keeps its Q fragments in registers, loaded
  // once the first commit group (Q and the first tile) has landed
  constexpr bool kQReg = C::KSTEPS <= 8;
  uint32_t qf[kQReg ? C::KSTEPS : 1][4];

  for (int32_t it = 0; it < ntiles; ++it) {
    const int stage = it % C::NS;
    const int32_t kb = lo + it * BN;
    // tile it has landed (at most NS - 2 newer groups pending); every warp is past tile it - 1,
    // whose stage the next load reuses
    cp_async_wait<C::NS - 2>();
    __syncthreads();
    if (it + C::NS - 1 < ntiles) row_issue((it + C::NS - 1) % C::NS, pend);
    cp_async_commit();
    pend = row_fetch(kb + C::NS * BN);  // the next iteration's tile

    // ---- S = Q K^T (this warp: one m-tile, NT n-tiles, one k-split) ----
    {
      float acc[C::NT][4];
#pragma unroll
      for (int i = 0; i < C::NT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
      const uint32_t bq = smem_u32(sQ);
      const uint32_t bk = smem_u32(sK + stage * C::KV_BYTES);
      const int qrow = s_mt * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
      const int n0 = s_ng * C::NT * 8;
      if constexpr (kQReg) {
        if (it == 0) {
#pragma unroll
          for (int kk = 0; kk < C::KSTEPS; ++kk)
            ldsm_x4(bq + swz<D>(qrow, (s_ks * C::KSTEPS + kk) * 2 + (lane >> 4)), qf[kk]);
        }
      }
#pragma unroll(kQReg ? C::KSTEPS : 4)
      for (int kk = 0; kk < C::KSTEPS; ++kk) {
        const int kc = (s_ks * C::KSTEPS + kk) * 2;
        uint32_t af[4];
        if constexpr (kQReg) {
          af[0] = qf[kk][0]; af[1] = qf[kk][1]; af[2] = qf[kk][2]; af[3] = qf[kk][3];
        } else {
          ldsm_x4(bq + swz<D>(qrow, kc + (lane >> 4)), af);
        }
        if (C::NT % 2 == 0) {
#pragma unroll
          for (int nt = 0; nt < C::NT; nt += 2) {
            uint32_t bf[4];
            const int key = n0 + nt * 8 + (lane & 7) + 8 * (lane >> 4);
            ldsm_x4(bk + swz<D>(key, kc + ((lane >> 3) & 1)), bf);
            mma_bf16(acc[nt], af, bf);
            mma_bf16(acc[nt + 1], af, bf + 2);
          }
        } else {
#pragma unroll
          for (int nt = 0; nt < C::NT; ++nt) {
            uint32_t bf[2];
            const int key = n0 + nt * 8 + (lane & 7);
            ldsm_x2(bk + swz<D>(key, kc + ((lane >> 3) & 1)), bf);
            mma_bf16(acc[nt], af, bf);
          }
        }
      }
      // scale into log2 units, mask, and park in shared memory
      float* S = sS + s_ks * BM * C::SLD;
#pragma unroll
      for (int nt = 0; nt < C::NT; ++nt) {
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int m = s_mt * 16 + (lane >> 2) + h2 * 8;
          const int tl = m / G;
          const int32_t pos = sp + tok0 + tl;
          const bool rv = m < ntok * G;
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int col = n0 + nt * 8 + 2 * (lane & 3) + e;
            const int32_t j = kb + col;
            // decode: every key in [lo, hi) is visible (the range already applies the window
            // and hi <= position + 1)
            const bool vis = C::DECODE ? rv && j < hi
                                       : rv && j < hi && j <= pos && (W < 0 || pos - j <= W);
            S[m * C::SLD + col] = vis ? acc[nt][h2 * 2 + e] * a.sm_scale_log2 : -INFINITY;
          }
        }
      }
    }
    __syncthreads();

    // ---- online softmax: TPR threads per row, VPT contiguous columns each ----
    {
      float s[C::VPT];
#pragma unroll
      for (int v = 0; v < C::VPT; v += 2) {
        float2 x = *reinterpret_cast<const float2*>(sS + sm_row * C::SLD + sm_sub * C::VPT + v);
        s[v] = x.x; s[v + 1] = x.y;
#pragma unroll
        for (int k = 1; k < C::KS; ++k) {
          // k-split partials: masked entries are -inf in every partial
          float2 y = *reinterpret_cast<const float2*>(sS + k * BM * C::SLD + sm_row * C::SLD + sm_sub * C::VPT + v);
          s[v] += y.x; s[v + 1] += y.y;
        }
      }
      float mx = -INFINITY;
#pragma unroll
      for (int v = 0; v < C::VPT; ++v) mx = fmaxf(mx, s[v]);
#pragma unroll
      for (int off = C::TPR / 2; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float m_new = fmaxf(row_m, mx);
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = exp2f(row_m - m_use);
      float sum = 0.f;
      __nv_bfloat16* P = sP + sm_row * C::PLD + sm_sub * C::VPT;
#pragma unroll
      for (int v = 0; v < C::VPT; v += 2) {
        // sum the bf16-rounded weights that the PV product uses (O / l stays an exact
        // weighted average of V rows)
        const __nv_bfloat162 pb = __floats2bfloat162_rn(exp2f(s[v] - m_use), exp2f(s[v + 1] - m_use));
        sum += __bfloat162float(pb.x) + __bfloat162float(pb.y);
        *reinterpret_cast<__nv_bfloat162*>(P + v) = pb;
      }
#pragma unroll
      for (int off = C::TPR / 2; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      row_l = row_l * alpha + sum;
      row_m = m_new;
      if (sm_sub == 0) sAlpha[sm_row] = alpha;
    }
    __syncthreads();

    // ---- O = alpha * O + P V (this warp: one m-tile, DCOLS columns) ----
    {
      const int r0 = o_mt * 16 + (lane >> 2);
      const float al0 = sAlpha[r0], al1 = sAlpha[r0 + 8];
#pragma unroll
      for (int i = 0; i < C::NTO; ++i) {
        o[i][0] *= al0; o[i][1] *= al0; o[i][2] *= al1; o[i][3] *= al1;
      }
      const uint32_t bp = smem_u32(sP);
      const uint32_t bv = smem_u32(sV + stage * C::KV_BYTES);
      const int prow = o_mt * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
      for (int kk = 0; kk < BN / 16; ++kk) {
        uint32_t af[4];
        ldsm_x4(bp + (uint32_t)((prow * C::PLD + kk * 16 + (lane >> 4) * 8) * 2), af);
        const int key = kk * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
        for (int nt = 0; nt < C::NTO; nt += 2) {
          uint32_t bf[4];
          const int c = (o_cg * C::DCOLS) / 8 + nt + (lane >> 4);
          ldsm_x4_t(bv + swz<D>(key, c), bf);
          mma_bf16(o[nt], af, bf);
          mma_bf16(o[nt + 1], af, bf + 2);
        }
      }
    }
  }

  // ---- epilogue ----
  if (sm_sub == 0) sL[sm_row] = row_l;
  if (a.lse && !(C::DECODE && nchunks > 1) && sm_sub == 0 && sm_valid) {
    // natural-log normaliser of the row: row_m and row_l are in log2 units of the scores
    a.lse[(int64_t)(q0 + tok0 + sm_tl) * Hq + g * G + (sm_row % G)] =
        row_l > 0.f ? (row_m + log2f(row_l)) * kLn2 : -INFINITY;
  }
  if (C::DECODE && nchunks > 1 && sm_sub == 0 && sm_valid) {
    const int h = g * G + (sm_row % G);
    float* ml = a.ws_ml + (((int64_t)r * Hq + h) * a.max_chunks + chunk) * 2;
    ml[0] = row_m;
    ml[1] = row_l;
  }
  __syncthreads();
  (void)sm_pos;
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    const int m = o_mt * 16 + (lane >> 2) + h2 * 8;
    if (m >= ntok * G) continue;
    const float l = sL[m];
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const int tl = m / G, h = g * G + (m % G);
    if (C::DECODE && nchunks > 1) {
      float* dst = a.ws_o + (((int64_t)r * Hq + h) * a.max_chunks + chunk) * D + o_cg * C::DCOLS;
#pragma unroll
      for (int nt = 0; nt < C::NTO; ++nt) {
        const int col = nt * 8 + 2 * (lane & 3);
        *reinterpret_cast<float2*>(dst + col) = make_float2(o[nt][h2 * 2] * inv, o[nt][h2 * 2 + 1] * inv);
      }
    } else {
      __nv_bfloat16* dst = a.out + ((int64_t)(q0 + tok0 + tl) * Hq + h) * D + o_cg * C::DCOLS;
#pragma unroll
      for (int nt = 0; nt < C::NTO; ++nt) {
        const int col = nt * 8 + 2 * (lane & 3);
        *reinterpret_cast<__nv_bfloat162*>(dst + col) =
            __floats2bfloat162_rn(o[nt][h2 * 2] * inv, o[nt][h2 * 2 + 1] * inv);
      }
    }
  }
}

// Combine the decode chunks of one (request, query head) row:
// o = sum_c l_c 2^(m_c - M) o_c / sum_c l_c 2^(m_c - M).
// The chunks' (m, l) pairs are loaded once, spread over the threads, and kept in shared memory
// (256 chunks at a time); then each thread issues its loads of four columns for eight chunks at
// once, so a row waits for about two round trips to memory rather than one per chunk.
template <int D>
__global__ void __launch_bounds__(D / 4)
attn_merge_kernel(AttnArgs a) {
  constexpr int NT = D / 4, NWARP = NT / 32, CB = 256;
  __shared__ float s_m[CB], s_l[CB], s_part[NWARP];
  const int32_t r = blockIdx.x, h = blockIdx.y;
  const PlanDev& pl = a.plan;
  const int32_t kvp0 = pl.kv_page_indptr[r], kvp1 = pl.kv_page_indptr[r + 1];
  const int32_t p = pl.start_pos[r];
  const int32_t ks0 = pl.kv_start[r];
  const int32_t kv_len = pl.ring ? p + (pl.qo_indptr[r + 1] - pl.qo_indptr[r])
                                 : ks0 + (kvp1 - kvp0 - 1) * a.pool.page_size + pl.last_page_len[r];
  const int32_t W = a.window_left;
  const int32_t lo = W >= 0 ? max(ks0, p - W) : ks0;
  const int32_t hi = min(p + 1, kv_len);
  const int32_t nch = (hi - lo + a.kv_chunk - 1) / a.kv_chunk;
  if (nch <= 1) return;  // written directly by the partition kernel
  const int64_t row = ((int64_t)r * a.num_qo_heads + h) * a.max_chunks;
  const int tid = threadIdx.x, lane = tid & 31;
  // the maximum M over the chunks
  float mx = -INFINITY;
  for (int c = tid; c < nch; c += NT) {
    const float2 ml = *reinterpret_cast<const float2*>(a.ws_ml + (row + c) * 2);
    mx = fmaxf(mx, ml.x);
    if (c < CB) {
      s_m[c] = ml.x;
      s_l[c] = ml.y;
    }
  }
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  if (lane == 0) s_part[tid >> 5] = mx;
  __syncthreads();
  float M = s_part[0];
  for (int wv = 1; wv < NWARP; ++wv) M = fmaxf(M, s_part[wv]);
  const float Mr = M == -INFINITY ? 0.f : M;
  // every thread sums the same weights in the same order, so all hold the same denominator
  const int d = tid * 4;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
  for (int cb = 0; cb < nch; cb += CB) {
    const int n = min(CB, nch - cb);
    if (cb > 0) {
      __syncthreads();  // the previous block's weights have been read
      for (int c = tid; c < n; c += NT) {
        const float2 ml = *reinterpret_cast<const float2*>(a.ws_ml + (row + cb + c) * 2);
        s_m[c] = ml.x;
        s_l[c] = ml.y;
      }
      __syncthreads();
    }
    for (int c = tid; c < n; c += NT) s_l[c] = s_l[c] > 0.f ? s_l[c] * exp2f(s_m[c] - Mr) : 0.f;
    __syncthreads();
    for (int c0 = 0; c0 < n; c0 += 8) {
      float4 v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        v[k] = c0 + k < n ? *reinterpret_cast<const float4*>(a.ws_o + (row + cb + c0 + k) * D + d)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float w = c0 + k < n ? s_l[c0 + k] : 0.f;
        acc.x += w * v[k].x; acc.y += w * v[k].y; acc.z += w * v[k].z; acc.w += w * v[k].w;
        den += w;
      }
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  if (a.lse && tid == 0)
    a.lse[(int64_t)pl.qo_indptr[r] * a.num_qo_heads + h] =
        den > 0.f ? (M + log2f(den)) * kLn2 : -INFINITY;
  __nv_bfloat16* dst = a.out + ((int64_t)pl.qo_indptr[r] * a.num_qo_heads + h) * D + d;
  *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
  *reinterpret_cast<__nv_bfloat162*>(dst + 2) = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
}

using Pre256 = Cfg<256, 64, 32, 2, 1, false>;
using Pre512 = Cfg<512, 32, 32, 1, 1, false>;
// decode streams K/V from HBM: three stages keep two tiles of loads in flight behind the one
// being computed. At head_dim 512 a warp's S work is two key tiles over a quarter of d (two
// independent MMA chains of 8 k-steps) rather than one key tile over half of d (one chain of
// 16): the CTA is alone on its SM, so the chains' latency is what it waits on.
using Dec256 = Cfg<256, 16, 32, 1, 2, true, 3>;
using Dec512 = Cfg<512, 16, 32, 2, 4, true, 3>;

template <class C>
cudaError_t launch_split(const AttnArgs& a, dim3 grid, cudaStream_t stream) {
  static PerDeviceOnce setup;  // the shared-memory opt-in, once per device
  int dev = 0, unused = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = setup.get(dev, [](int*) {
    return cudaFuncSetAttribute(attn_split_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)C::SMEM);
  }, &unused);
  if (e != cudaSuccess) return e;
  attn_split_kernel<C><<<grid, kThreads, C::SMEM, stream>>>(a);
  count_launch();
  return cudaGetLastError();
}

}  // namespace

int32_t attn_kernel_cta_tile_q(int32_t head_dim, int32_t group, int32_t page_size) {
  if (group <= 0 || group > Dec256::BM) return 0;
  if (attn_tc_supported(head_dim, group, page_size)) return attn_tc_rows() / group;
  const int32_t rows = head_dim == 256 ? Pre256::BM : head_dim == 512 ? Pre512::BM : 0;
  if (rows == 0 || rows % group != 0) return 0;
  return rows / group;
}

int32_t attn_kernel_kv_chunk(int32_t head_dim) { return head_dim == 512 ? 512 : 256; }

cudaError_t launch_attn_prefill(const AttnArgs& a, int32_t head_dim, cudaStream_t stream) {
  if (a.plan.num_work == 0) return cudaSuccess;
  if (attn_tc_supported(head_dim, a.group, a.pool.page_size))
    return launch_attn_prefill_tc(a, head_dim, stream);
  dim3 grid(a.plan.num_work, a.pool.num_kv_heads, 1);
  return head_dim == 256 ? launch_split<Pre256>(a, grid, stream)
                         : launch_split<Pre512>(a, grid, stream);
}

cudaError_t launch_attn_decode(const AttnArgs& args, int32_t head_dim, cudaStream_t stream) {
  if (args.plan.num_req == 0) return cudaSuccess;
  if (attn_decode_stream_supported(head_dim, args.group, args.pool.page_size))
    return launch_attn_decode_stream(args, head_dim, stream);
  // other page sizes: fixed key chunks per (request, KV head), partials in the workspace
  AttnArgs a = args;
  const size_t rows = (size_t)a.plan.num_req * a.num_qo_heads * a.max_chunks;
  a.ws_o = reinterpret_cast<float*>(a.ws_raw);
  a.ws_ml = a.ws_o + rows * (size_t)head_dim;
  dim3 grid(a.plan.num_req, a.pool.num_kv_heads, a.max_chunks);
  cudaError_t e = head_dim == 256 ? launch_split<Dec256>(a, grid, stream)
                                  : launch_split<Dec512>(a, grid, stream);
  if (e != cudaSuccess) return e;
  dim3 mgrid(a.plan.num_req, a.num_qo_heads, 1);
  if (head_dim == 256) attn_merge_kernel<256><<<mgrid, 256 / 4, 0, stream>>>(a);
  else attn_merge_kernel<512><<<mgrid, 512 / 4, 0, stream>>>(a);
  count_launch();
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------------------
// Decode partials in library-owned scratch, for callers that cannot allocate device memory.
// The array is part of the library image; host code may not use its name as an address, so
// the device address is looked up once per device with cudaGetSymbolAddress.
namespace {
static __device__ __align__(256) unsigned char g_decode_scratch[PG_NOALLOC_SCRATCH_BYTES];
std::mutex g_decode_scratch_mu;
void* g_decode_scratch_addr[128] = {nullptr};
}  // namespace

cudaError_t launch_attn_decode_static(AttnArgs a, int32_t head_dim, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_decode_scratch_mu);
    if (!g_decode_scratch_addr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_decode_scratch);
      if (e != cudaSuccess) return e;
      g_decode_scratch_addr[dev] = p;
    }
    base = g_decode_scratch_addr[dev];
  }
  a.ws_raw = base;
  return launch_attn_decode(a, head_dim, stream);
}

}  // namespace pg
