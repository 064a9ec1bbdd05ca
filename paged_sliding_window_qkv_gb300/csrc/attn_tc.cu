// Paged prefill attention on the 5th-generation tensor cores (tcgen05 + TMEM + TMA)
// ("feat(kernels): Rust wrapper for the hd256 windowed paged prefill", Description:
// paged reads, explicit sm_scale, inclusive-distance window_left, GQA by integer
// division; "feat(gemma4): paged KV serving across both attention families",
// Description: hd256 local layers with a sliding window, hd512 global layers causal).
//
// Work unit: a pair of adjacent 128-row query tiles (rows pack the GQA group of one KV head,
// token-major, head-minor) and one 256-column part of the output, run by the two CTAs of a
// cluster; the unit walks the 64-key tiles of the pair's visible key range, skipping tiles
// outside the causal window. The kernel is persistent: one CTA per SM (its shared and tensor
// memory fill the SM), each cluster taking one unit per round (longest first), so barriers,
// tensor memory and K/V rings carry over from unit to unit: the producers fetch the next
// unit's first tiles while the current one finishes, the next unit's Q enters TMEM before
// this unit's epilogue, and the next unit's first PV waits only for every softmax warp's read
// of O.
//
//   warp 0     K producer (TMA): this CTA's 32 keys of each tile, one 4-D box per page
//              (BR rows x 256 d) into 16 KB part slots; box coordinates and page ids are
//              worked out a batch of tiles ahead, and a head_dim 512 tile's two parts go out
//              in one copy instruction; also Q into shared memory: head_dim 512 each unit's
//              columns [256,512), head_dim 256 the whole of the next unit's Q (staged while
//              this unit runs, so Q's reads do not fall in the unit transition)
//   warp 10    V producer (TMA): this CTA's 128 output columns of each tile, one 3-D box per
//              page into 16 KB slots
//   warp 1     QK issuer (leader CTA): S = Q K^T into a TMEM S buffer (2-SM MMA, M=256, N=64,
//              K=16 steps; the first 256-d part reads Q from TMEM, head_dim 512's second part
//              from shared memory)
//   warp 11    PV issuer (leader CTA): O += P V into TMEM (M=256, N=256, K=16 steps; P from
//              shared memory); MMAs are issued by lane 0, completion signalled with
//              tcgen05.commit multicast to both CTAs
//   warps 2..9 softmax: two warps per TMEM lane quarter (32 query rows), masked on boundary
//              tiles only, online softmax in log2 units with lazy rescaling (O is rescaled in
//              TMEM only when a row maximum outgrows a 2^64 headroom by more than 2^48: bf16 P
//              and fp32 O and row sums hold the range, and O / l is unchanged). head_dim 256:
//              the two warps take alternate key tiles (all 64 keys each), pass the rows'
//              running reference between them, and the one that takes the next unit's first
//              tile moves that unit's staged Q into TMEM while the other finishes the last
//              tile; the epilogue passes each warp's 32 rows x 128 output columns through its
//              quarter of its P buffer to coalesced 16-byte stores. head_dim 512: both warps read every
//              tile, each exponentiates half of its keys, each stores half of the next unit's
//              first Q part, and the epilogue stores 256 contiguous bytes of a row per thread.
//              Each thread owns half of its row's O columns.
//
// O holds 256 output columns: for head_dim 512 each query tile is two units, each computing
// the full 512-wide S and half of O. The TMEM map is described at TcCfg.
//
// Every wait is bounded (two seconds of %globaltimer unless the launch passes a shorter limit);
// a wait that runs out sets the device status word, makes the CTA drain and free its tensor
// memory, and return.
#include "pg_internal.h"

#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>

#include <algorithm>
#include <mutex>

namespace pg {
namespace {

constexpr int kM = 128;            // query rows per CTA (one query tile)
constexpr int kBN = 64;            // keys per KV tile
constexpr int kDV = 256;           // output columns per unit
constexpr int kKH = kBN / 2;       // keys of a K tile held by each CTA of the pair
constexpr int kSlotBytes = 16 * 1024;  // one ring slot: 32 keys x 256 d (K) or 64 keys x 128 d (V)
constexpr int kThreadsTc = 384;  // K producer 0; QK issuer 1; softmax 2..9; V producer 10; PV issuer 11
// Lazy rescaling: a row's reference maximum is set 2^64 above the first maximum it sees and
// O is rescaled only when a later maximum exceeds the reference by more than 2^48. P stays
// within [2^-64, 2^48] of the row's true maximum weight: inside bf16's and fp32's range, with
// the same relative precision, and O / l does not depend on the reference.
constexpr float kRescaleLog2 = 48.f;
constexpr float kHeadroomLog2 = 64.f;

// The kernel runs on clusters of two CTAs and issues its MMAs in the 2-SM form
// (tcgen05 cta_group::2, M = 256): CTA c of the pair owns query tile c of a pair of adjacent
// query tiles, its 128 rows of Q, S, P and O, and half of every K and V tile: keys
// [32c, 32c + 32) of a K tile and output columns [128c, 128c + 128) of a V tile. The leader
// (rank 0) issues every MMA; each product reads both CTAs' halves and writes each CTA's rows of
// S or O into that CTA's tensor memory. Holding half a tile per CTA doubles the depth of the
// K/V rings that the shared memory allows, which is what hides the copies' latency.
//
// TMEM map (each CTA, 512 columns): O [0,256) (the unit's 256 output columns), Q columns
// [256,384) (this unit's first 256-d part of Q; QK reads A from TMEM), two S buffers
// [384,448) and [448,512). The softmax writes P(j) to a 16 KB shared-memory buffer (NPB of
// them; PV is SS), so QK(j + 2) waits only for both CTAs' reads of S(j). head_dim 512 also keeps Q
// columns [256,512) in shared memory (64 KB; QK's second part is SS); head_dim 256 uses the same
// 64 KB to stage the next unit's Q. K streams through NKS 256-d part slots (a tile is KP parts),
// V through NVR tile slots.
template <int DQK>
struct TcCfg {
  static constexpr int KP = DQK / 256;                // K parts per tile (256 d each)
  static constexpr int NKS = DQK == 256 ? 3 : 6;      // K part slots
  static constexpr int NVR = DQK == 256 ? 4 : 3;      // V tile slots
  static constexpr int NS = NKS + NVR;
  // 128 rows x 256 d of Q in shared memory: head_dim 512 keeps the unit's Q columns [256,512)
  // there (QK's second part reads them); head_dim 256 stages the next unit's Q there, loaded by
  // TMA during this unit and moved into TMEM at the unit's end
  static constexpr int QS_BYTES = kM * 256 * 2;
  static constexpr int P_BUF = kM * kBN * 2;          // one P buffer: 128 rows x 64 keys bf16
  // P buffers: head_dim 512 keeps one (PV(j) has long completed when the softmax of tile j + 1
  // writes P) and gives the 16 KB to the K ring
  static constexpr int NPB = DQK == 256 ? 2 : 1;
  static constexpr int SMEM_DATA = QS_BYTES + NS * kSlotBytes + NPB * P_BUF;
  // final row-sum exchange between warp pairs; head_dim 256 also passes the rows' running
  // reference from tile to tile ([tile parity][128 rows])
  static constexpr int XM_FLOATS = DQK == 256 ? 2 * kM : 0;
  static constexpr int XL_BYTES = 2 * kM * 4 + XM_FLOATS * 4;
  // ..., QFREE, (head_dim 256: 8 reference handoffs, Q staging full / free), 4 per-producer
  // fix-up barriers last
  static constexpr int NBAR = 2 * NS + 22 + (DQK == 256 ? 10 : 0);
  static constexpr int SMEM = SMEM_DATA + XL_BYTES + NBAR * 8 + 16 + 1024;
  static constexpr int NSB = 2;                 // S buffers (and PFULL / PVDONE barrier pairs)
  // softmax warps (of both CTAs) that read each S buffer and write each P buffer: head_dim 256
  // gives each tile to one warp of a lane quarter, head_dim 512 to both
  static constexpr int SMW = DQK == 256 ? 8 : 16;
  static constexpr uint32_t TM_O = 0, TM_Q = 256, TM_S = 384;
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

struct TcArgs {
  PlanDev plan;
  const __nv_bfloat16* q;
  __nv_bfloat16* out;
  const __nv_bfloat16* pool_layer;  // pool base of the called layer
  int64_t stride_page, stride_kv, stride_head;
  int32_t num_qo_heads, group, cta_tile_q, window_left;
  int32_t page_size, num_pages, num_kv_heads, box_rows_k, box_rows_v;
  float scale_log2;
  float* lse;  // optional [T][Hq] natural-log normaliser of each row (null: not written)
  int* status;
  uint64_t wait_ns;       // limit of every bounded wait
  int32_t test_withhold;  // test hook: the leader's K producer withholds its first arrival
};

// What a bounded wait needs: the CTA's abort flag (set by whichever role gives up first), the
// device status word, and the limit.
struct WaitCtx {
  volatile int* abort_flag;
  int* status;
  uint64_t limit_ns;
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
__device__ __forceinline__ bool mbar_wait_body(uint32_t bar, uint32_t parity, const WaitCtx& w) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    // plain try_wait: with an explicit suspend-time hint, waiters woke measurably later
    if (mbar_try_wait(bar, parity)) return true;
    if (*w.abort_flag) return false;
    if (globaltimer() - t0 > w.limit_ns) {
      atomicOr(w.status, kStatusTimeout);
      *w.abort_flag = 1;
      return false;
    }
  }
}
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, WaitCtx w) {
  return mbar_wait_body(bar, parity, w);
}
// The same wait inlined, for the MMA-issuing warps.
__device__ __forceinline__ bool mbar_wait_inline(uint32_t bar, uint32_t parity, const WaitCtx& w) {
  return mbar_wait_body(bar, parity, w);
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// ---- the CTA pair
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// the address of the same shared-memory location in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t mapa(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
// arrivals on a barrier given by its cluster address (either CTA of the pair). What they
// publish is read only by the tensor cores, from the arriving CTA's own shared or tensor memory
// (ordered by fence.proxy.async / tcgen05 fences before the arrival), so the default release
// (CTA scope) suffices; cluster scope measured several times slower here.
__device__ __forceinline__ void mbar_arrive_cl(uint32_t cbar) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cbar) : "memory");
}
// An arrival with an expected byte count, without release semantics: it publishes no data of
// its own (the TMA's byte count completes the phase), and a release arrive would first wait for
// every earlier load of the thread, which in a producer loop means the next page-id lookup.
__device__ __forceinline__ void mbar_expect_tx_cl_relaxed(uint32_t cbar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.relaxed.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(cbar),
               "r"(bytes)
               : "memory");
}

// TMA loads into this CTA's shared memory whose bytes count on `bar`, a cluster address that may
// be the leader's barrier
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* tm, int c0, int c1,
                                            int c2, int c3, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(tm), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
      : "memory");
}
// L2 prefetch of a 3-D box (no shared-memory destination, no completion)
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap* tm, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global [%0, {%1, %2, %3}];" ::"l"(tm), "r"(x),
               "r"(y), "r"(z)
               : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* tm, int x, int y,
                                            int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
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
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// The MMA and commit helpers below are executed by the whole issuing warp of the leader CTA
// and act from lane 0 only; the MMAs are the 2-SM form and each commit arrives on the barrier
// at the same offset in both CTAs. The instruction descriptor is an immediate. Measured on this kernel: with the
// descriptor in a register, or with the issuing lane picked by elect.sync, M128 MMAs issued at
// one per ~220-290 cycles in many tiles; predicated on lane 0 with an immediate descriptor they
// keep the tensor pipe full (32-48 cycles per M128 x N64 x K16 instruction).
template <uint32_t IDESC>
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred e, p;\n .reg .u32 ln;\n mov.u32 ln, %%laneid;\n setp.eq.u32 e, ln, 0;\n setp.ne.b32 p, %3, 0;\n"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %4, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(acc), "n"(IDESC)
      : "memory");
}
template <uint32_t IDESC>
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred e, p;\n .reg .u32 ln;\n mov.u32 ln, %%laneid;\n setp.eq.u32 e, ln, 0;\n setp.ne.b32 p, %3, 0;\n"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %4, p;\n}\n" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(acc), "n"(IDESC)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "{\n .reg .pred e;\n .reg .u32 ln;\n mov.u32 ln, %%laneid;\n setp.eq.u32 e, ln, 0;\n"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n}\n"
      ::"r"(bar), "h"((uint16_t)3)
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

// 2^x with the hardware exponential (ex2.approx; -inf gives 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// ------------------------------------------------------------------ kernel
// One work unit = (pair of adjacent query tiles of one request, KV head, 256-column part of the
// output). Units are numbered longest first (the plan lists each request's tile pairs in token
// order, so the last pairs come first); cluster i takes one unit per round of clusters.
struct TcUnit {
  int32_t q0, tok0, ntok;  // this CTA's query tile: request's first token, tile start, tokens (0: none)
  // keys held: positions [kv_start, kv_len); key tiles start kb0 + 64 t, 64-aligned from kv_start
  int32_t kvp0, kvp1, kv_len, kv_start, sp, kb0, ntiles, g, dh;
};
__device__ __forceinline__ TcUnit tc_unit(const TcArgs& a, int32_t w, int32_t ndh, int32_t rank) {
  const PlanDev& pl = a.plan;
  TcUnit u;
  const int32_t pr = pl.num_pairs - 1 - w / (a.num_kv_heads * ndh);
  u.g = (w / ndh) % a.num_kv_heads;
  u.dh = w % ndh;
  // the pair's entry of the plan's pair table: two 16-byte loads, no dependent lookups
  const int4 e0 = __ldg(reinterpret_cast<const int4*>(pl.pair_tab) + 2 * pr);
  const int4 e1 = __ldg(reinterpret_cast<const int4*>(pl.pair_tab) + 2 * pr + 1);
  const int32_t t0 = e0.x, len = e0.z;
  const int32_t TQ = a.cta_tile_q;
  u.q0 = e0.y;
  u.sp = e0.w;
  u.tok0 = t0 + rank * TQ;
  u.ntok = max(0, min(TQ, len - u.tok0));
  u.kvp0 = e1.x;
  u.kvp1 = e1.y;
  u.kv_len = e1.z;
  u.kv_start = e1.w;
  // the pair's key range: the keys some row of either tile sees
  const int32_t W = a.window_left;
  const int32_t p_first = u.sp + t0, p_last = u.sp + min(t0 + 2 * TQ, len) - 1;
  const int32_t lo = W >= 0 ? max(u.kv_start, p_first - W) : u.kv_start;
  const int32_t hi = min(p_last + 1, u.kv_len);
  // tiles are aligned from the first key held, so a box of page rows never straddles a page
  u.kb0 = u.kv_start + ((lo - u.kv_start) & ~(kBN - 1));
  u.ntiles = hi > u.kb0 ? (hi - u.kb0 + kBN - 1) / kBN : 0;
  return u;
}
// L2 prefetch of unit w's pair-table entry, so tc_unit finds it there later
__device__ __forceinline__ void tc_unit_prefetch(const TcArgs& a, int32_t w, int32_t ndh) {
  const int32_t pr = a.plan.num_pairs - 1 - w / (a.num_kv_heads * ndh);
  asm volatile("prefetch.global.L2 [%0];" ::"l"(a.plan.pair_tab + 8 * pr));
}

template <int DQK>
__global__ void __launch_bounds__(kThreadsTc, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kv,
               const __grid_constant__ CUtensorMap tm_v, TcArgs a) {
  using C = TcCfg<DQK>;
  constexpr int KP = C::KP, NKS = C::NKS, NVR = C::NVR, NS = C::NS;
  constexpr int NSB = C::NSB;
  constexpr int32_t NDH = DQK / kDV;
  constexpr uint32_t kTmO = C::TM_O, kTmQ = C::TM_Q, kTmS = C::TM_S;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* gbase = smem_raw + (base - raw);
  const uint32_t sQ = base;
  const uint32_t sSlots = base + C::QS_BYTES;
  const uint32_t sP = sSlots + NS * kSlotBytes;  // NPB P buffers
  float* xl = reinterpret_cast<float*>(gbase + C::SMEM_DATA);  // [2 halves][128 rows]
  const uint32_t bars = base + C::SMEM_DATA + C::XL_BYTES;
  auto FULL = [&](int s) { return bars + 8u * s; };
  auto EMPTY = [&](int s) { return bars + 8u * (NS + s); };
  // Barriers named here exist in both CTAs. FULL, SFREE, PFULL and QFULL are waited on in the
  // leader only and count both CTAs' arrivals; EMPTY, SFULL, PVDONE, QFREE and DRAIN receive
  // the leader's commits in both CTAs; PAIRB and the fix-up barriers are local.
  const uint32_t SFULL = bars + 8u * (2 * NS), SFREE = SFULL + 16, PFULL = SFULL + 32,
                 PVDONE = SFULL + 56, QFULL = SFULL + 80,
                 OFREE = SFULL + 88,  // head_dim 256: every softmax warp has read the unit's O
                 DRAIN = SFULL + 96,
                 PAIRB = SFULL + 104,  // 4 barriers, one per lane quarter
                 QFREE = SFULL + 136,  // head_dim 512: the unit's QK MMAs have read Q's shared part
                 PAIRX = SFULL + 144,  // head_dim 256: [tile parity][lane quarter] reference handoffs
                 QSFULL = SFULL + 208,  // head_dim 256: the next unit's Q has landed in shared memory
                 QSFREE = SFULL + 216;  // head_dim 256: ... and has been moved into TMEM
  // ring slots, by the CTA's running tile count J: K part pp of tile J is the (J KP + pp)-th part
  // through the NKS K slots; V tile J uses V slot J mod NVR
  auto KSLOT = [&](int32_t j, int pp) { return (int)((j * KP + pp) % NKS); };
  auto KROUND = [&](int32_t j, int pp) { return (int)((j * KP + pp) / NKS); };
  auto VSLOT = [&](int32_t j) { return NKS + (int)(j % NVR); };
  uint32_t* tmem_slot =
      reinterpret_cast<uint32_t*>(gbase + C::SMEM_DATA + C::XL_BYTES + C::NBAR * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const WaitCtx wc{abort_flag, a.status, a.wait_ns};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();  // 0: the leader, which issues the pair's MMAs
  const bool leader = rank == 0;
  auto LEAD = [&](uint32_t bar) { return mapa(bar, 0); };  // the leader's copy of a barrier
  const PlanDev& pl = a.plan;
  const int32_t G = a.group, Hq = a.num_qo_heads;
  const int32_t ps = a.page_size;
  const int32_t W = a.window_left;
  const int32_t nunits = pl.num_pairs * a.num_kv_heads * NDH;
  // the cluster's k-th unit: rounds of (number of clusters) units, walked forwards in even
  // rounds and backwards in odd ones, so the long and the short units of the longest-first
  // order even out
  const int32_t ncl = (int32_t)gridDim.x / 2, ci = (int32_t)blockIdx.x / 2;
  auto unit_at = [&](int32_t k) -> int32_t { return k * ncl + ((k & 1) ? ncl - 1 - ci : ci); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(FULL(s), 2);  // one arrival (with its byte count) from each CTA's producer
      mbar_init(EMPTY(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(SFULL + 8 * b, 1);
      mbar_init(SFREE + 8 * b, C::SMW);  // the softmax warps of both CTAs that read S have
    }
    for (int b = 0; b < 3; ++b) {
      mbar_init(PFULL + 8 * b, C::SMW);
      mbar_init(PVDONE + 8 * b, 1);
    }
    // per unit: head_dim 256: the four softmax warps of each CTA that take the unit's first tile
    // store its Q into TMEM; head_dim 512: all sixteen store Q columns [0,256), and each CTA's
    // K producer loads the rest by TMA
    mbar_init(QFULL, DQK == 256 ? 8 : 18);
    mbar_init(OFREE, 16);
    mbar_init(QFREE, 1);
    for (int f = 0; f < 4; ++f) mbar_init(bars + 8u * (C::NBAR - 4 + f), 1);
    mbar_init(DRAIN, 2);  // one final commit from each MMA-issuing warp of the leader
    for (int q = 0; q < 4; ++q) mbar_init(PAIRB + 8 * q, 2);
    if (DQK == 256) {
      for (int q = 0; q < 8; ++q) mbar_init(PAIRX + 8 * q, 1);
      mbar_init(QSFULL, 1);  // the K producer's arrival with the staged bytes
      mbar_init(QSFREE, 4);  // the four softmax warps (one per lane quarter) that move it
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before either CTA signals the other
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 || warp == 10) {
    // ------------------------------------------------------------ producers
    // Each CTA loads its half of every tile: warp 0 the keys [32 rank, 32 rank + 32) of each K
    // part, warp 10 the output columns [128 rank, 128 rank + 128) of each V tile, in boxes of BR
    // key rows (one page each), counted on the leader's FULL barrier. K lands as
    // [key / 8][64-d chunk][8 rows][128 B] (a 4-D box), so every 8-key atom of QK's K-major
    // B operand sits 4096 bytes after the previous one across pages; V lands page-major as
    // [chunk][BR rows][128 B] (a 3-D box of two chunks), which PV's MN-major B operand reads with
    // a chunk stride of BR*128 bytes. Warp 0 also loads each unit's Q columns [256,512).
    const bool is_v = warp == 10;
    const uint32_t FIX = bars + 8u * (C::NBAR - 4 + (is_v ? 1 : 0));
    uint32_t fix_phase = 0;
    bool ok = true;
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(is_v ? &tm_v : &tm_kv) : "memory");
      if (!is_v) asm volatile("prefetch.tensormap [%0];" ::"l"(&tm_q) : "memory");
      if (!is_v && unit_at(1) < nunits) tc_unit_prefetch(a, unit_at(1), NDH);
    }
    const int BR = is_v ? a.box_rows_v : a.box_rows_k;  // key rows per box
    const int nbox = (is_v ? kBN : kKH) / BR;            // boxes per tile half
    const int key_off = is_v ? 0 : (int)rank * kKH;      // this CTA's first key of a tile
    const uint32_t row_bytes = is_v ? 256u : 512u;       // bytes of one key row in a slot
    const int64_t head_rows = (int64_t)ps;
    // head_dim 256: Q of the cluster's k-th unit goes into the staging buffer once the softmax
    // warps have moved Q of unit k - 1 out of it (QSFREE phase k - 1); one lane issues it
    auto stage_q = [&](int32_t k) -> bool {
      if (lane != 0) return true;
      if (k > 0 && !mbar_wait(QSFREE, (k - 1) & 1, wc)) return false;
      const TcUnit v = tc_unit(a, unit_at(k), NDH, (int32_t)rank);
      mbar_expect_tx(QSFULL, v.ntok > 0 ? (uint32_t)C::QS_BYTES : 0u);
      if (v.ntok > 0)
        for (int c = 0; c < 4; ++c)
          tma_load_3d(sQ + c * (kM * 128), &tm_q, c * 64, v.g * G, v.q0 + v.tok0, mapa(QSFULL, rank));
      return true;
    };
    if (DQK == 256 && !is_v && unit_at(0) < nunits) ok = __shfl_sync(0xffffffffu, stage_q(0) ? 1 : 0, 0) != 0;
    int32_t J = 0;  // tiles of this cluster's earlier units
    int32_t ui = 0;
    for (int32_t w = unit_at(0); ok && w < nunits; w = unit_at(++ui)) {
      const TcUnit u = tc_unit(a, w, NDH, (int32_t)rank);
      // head_dim 256: the next unit's Q is staged after this unit's fourth K tile has been issued:
      // that tile's slot wait shows this unit's first QK complete, so its Q has left the staging
      // buffer and the wait for it does not hold up the ring (in units of up to four tiles it
      // comes after the last tile)
      const bool stage_next = DQK == 256 && !is_v && unit_at(ui + 1) < nunits;
      const int32_t stage_at = min(u.ntiles, 4);
      if (!is_v && lane == 0) {
        // a unit ahead, bring the next unit's pair-table entry and this CTA's Q rows of it into
        // L2, so the softmax warps' move to that unit waits on L2 rather than DRAM
        if (unit_at(ui + 2) < nunits) tc_unit_prefetch(a, unit_at(ui + 2), NDH);
        if (DQK != 256 && unit_at(ui + 1) < nunits) {
          const TcUnit un = tc_unit(a, unit_at(ui + 1), NDH, (int32_t)rank);
          if (un.ntok > 0)
            for (int c = 0; c < DQK / 64; ++c) tma_prefetch_3d(&tm_q, c * 64, un.g * G, un.q0 + un.tok0);
        }
      }
      if (DQK == 512 && !is_v) {
        // Q columns [256,512) of this CTA's tile, once the previous unit's QK MMAs have read them
        int go = 1;
        if (lane == 0) {
          if (ui > 0 && !mbar_wait(QFREE, (ui - 1) & 1, wc)) {
            go = 0;
          } else {
            mbar_expect_tx_cl_relaxed(LEAD(QFULL), u.ntok > 0 ? (uint32_t)C::QS_BYTES : 0u);
            if (u.ntok > 0)
              for (int c = 0; c < (DQK - 256) / 64; ++c)
                tma_load_3d(sQ + c * (kM * 128), &tm_q, 256 + c * 64, u.g * G, u.q0 + u.tok0,
                            LEAD(QFULL));
          }
        }
        if (!__shfl_sync(0xffffffffu, go, 0)) {
          ok = false;
          break;
        }
      }
      // Box coordinates are worked out a batch of TB tiles at a time, one box per lane: lane i
      // holds box i mod nbox of tile (batch start + i / nbox). Page ids are read a batch ahead,
      // so the per-tile path is a slot wait, one byte-count arrival and the copies.
      const int TB = 32 / nbox;
      const int my_t = lane / nbox, my_b = lane % nbox;
      auto lookup = [&](int32_t t0) -> int32_t {  // page id of this lane's box in the batch at t0
        const int32_t tt = t0 + my_t;
        if (tt >= u.ntiles) return -1;
        const int32_t ks = u.kb0 + tt * kBN + key_off + my_b * BR;
        if (ks >= u.kv_len) return -1;
        const int32_t lp = (ks - u.kv_start) / ps;  // logical page; a ring wraps it over its pages
        const int32_t pidx = u.kvp0 + (pl.ring ? lp % max(u.kvp1 - u.kvp0, 1) : lp);
        return (pidx < u.kvp1 && pidx < pl.num_page_ids) ? pl.page_ids[pidx] : a.num_pages;
      };
      int32_t pg_next = lookup(0);
      int32_t my_page = -1, my_row = 0;
      uint32_t bm_load = 0u, bm_fix = 0u;
      const uint32_t box_mask = nbox >= 32 ? 0xffffffffu : ((1u << nbox) - 1u);
      const uint32_t box_bytes = (uint32_t)BR * row_bytes;
      for (int32_t t = 0; ok && t < u.ntiles; ++t) {
        const int32_t JJ = J + t;
        if (stage_next && t == stage_at && !__shfl_sync(0xffffffffu, stage_q(ui + 1) ? 1 : 0, 0)) {
          ok = false;
          break;
        }
        const int tb = t % TB;
        if (tb == 0) {
          my_page = pg_next;
          pg_next = lookup(t + TB);  // used TB tiles from now
          const int32_t tt = t + my_t;
          const int32_t ks = u.kb0 + tt * kBN + key_off + my_b * BR;
          const bool live = tt < u.ntiles;
          const bool past = !live || ks >= u.kv_len;
          const bool bad = !past && (my_page < 0 || my_page >= a.num_pages);
          const bool load = !past && !bad;
          // V rows past kv_len (partial last page) must read as zeros; K rows there are masked
          const bool fixb = live && (bad || (is_v && ks + BR > u.kv_len));
          bm_load = __ballot_sync(0xffffffffu, load);
          bm_fix = __ballot_sync(0xffffffffu, fixb);
          if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(a.status, kStatusBounds);
          my_row = load ? (int32_t)((((int64_t)my_page * 2 + (is_v ? 1 : 0)) * a.num_kv_heads + u.g) *
                                        head_rows + ((ks - u.kv_start) & (ps - 1)))
                        : 0;
        }
        // test hook: the leader's K producer issues neither the arrival nor the copies of its
        // first tile, so the QK issuer's wait on that slot runs out
        if (!is_v && leader && a.test_withhold && ui == 0 && t == 0) continue;
        const int sh = tb * nbox;
        const bool fix = ((bm_fix >> sh) & box_mask) != 0u;
        const uint32_t bytes = (uint32_t)__popc((bm_load >> sh) & box_mask) * box_bytes;
        const bool issue = my_t == tb && ((bm_load >> lane) & 1u);
        const int nparts = is_v ? 1 : KP;
        if (!is_v && KP > 1 && !fix) {
          // every K part of the tile in one copy instruction (each warp-level copy instruction
          // costs the producer hundreds of cycles, whatever its box count): lane i copies box
          // i mod nbox of part i / nbox, after lane 0 has seen every part's slot free and
          // announced each part's bytes
          int r = 1;
          if (lane == 0) {
            for (int pp = 0; r && pp < KP; ++pp)
              r = mbar_wait_inline(EMPTY(KSLOT(JJ, pp)), (KROUND(JJ, pp) & 1) ^ 1, wc) ? 1 : 0;
            if (r)
              for (int pp = 0; pp < KP; ++pp) mbar_expect_tx_cl_relaxed(LEAD(FULL(KSLOT(JJ, pp))), bytes);
          }
          if (!__shfl_sync(0xffffffffu, r, 0)) {
            ok = false;
            break;
          }
          const int pp = lane / nbox, b = lane % nbox;
          const int32_t row = __shfl_sync(0xffffffffu, my_row, sh + b);
          const bool go = pp < KP && ((bm_load >> (sh + b)) & 1u);
          if (go) {
            const int s = KSLOT(JJ, pp);
            tma_load_4d(sSlots + s * kSlotBytes + b * (BR * 512), &tm_kv, 0, 0, pp * 4, row / 8,
                        LEAD(FULL(s)));
          }
          continue;
        }
        for (int pp = 0; ok && pp < nparts; ++pp) {
          const int s = is_v ? VSLOT(JJ) : KSLOT(JJ, pp);
          const int round = is_v ? (int)(JJ / NVR) : KROUND(JJ, pp);
          const int c0 = is_v ? u.dh * 4 + (int)rank * 2 : pp * 4;
          int r = 1;
          if (lane == 0) r = mbar_wait_inline(EMPTY(s), (round & 1) ^ 1, wc) ? 1 : 0;
          if (!__shfl_sync(0xffffffffu, r, 0)) {
            ok = false;
            break;
          }
          const uint32_t slot = sSlots + s * kSlotBytes;
          const uint32_t bar = fix ? FIX : LEAD(FULL(s));
          if (lane == 0) {
            if (!fix) mbar_expect_tx_cl_relaxed(bar, bytes);
            else if (bytes > 0) mbar_expect_tx(FIX, bytes);
          }
          __syncwarp();
          if (issue) {
            if (is_v) tma_load_3d(slot + my_b * (BR * 256), &tm_v, 0, my_row, c0, bar);
            else tma_load_4d(slot + my_b * (BR * 512), &tm_kv, 0, 0, c0, my_row / 8, bar);
          }
          if (fix) {
            if (bytes > 0) {
              if (!__all_sync(0xffffffffu, mbar_wait(FIX, fix_phase, wc))) {
                ok = false;
                break;
              }
              fix_phase ^= 1u;
            }
            // zero this warp's rows that must not be read: keys past kv_len, keys on bad pages
            const int32_t kb = u.kb0 + t * kBN + key_off;  // first key of this CTA's half
            for (int b = 0; b < nbox; ++b) {
              const int32_t pb = __shfl_sync(0xffffffffu, my_page, sh + b);
              for (int rr = 0; rr < BR; ++rr) {
                const int32_t key = kb + b * BR + rr;
                if (key < u.kv_len && pb >= 0 && pb < a.num_pages) continue;
                const int c = lane >> 3, w16 = lane & 7;  // chunk c, 16-byte piece w16 of a 128-B row
                const int kt = b * BR + rr;  // key within this CTA's half
                if (is_v && c >= 2) continue;  // V rows are two chunks (256 B) here
                const uint32_t off = is_v ? b * (BR * 256) + c * (BR * 128) + rr * 128
                                          : (kt >> 3) * 4096 + c * 1024 + (kt & 7) * 128;
                *(reinterpret_cast<uint4*>(gbase + (slot - base) + off) + w16) = make_uint4(0u, 0u, 0u, 0u);
              }
            }
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive_cl(LEAD(FULL(s)));
          }
        }
      }
      if (ok && stage_next && stage_at == u.ntiles)
        ok = __shfl_sync(0xffffffffu, stage_q(ui + 1) ? 1 : 0, 0) != 0;
      J += u.ntiles;
    }
    if (!ok) {
      // aborting: give the copies this warp already issued time to land (they complete within
      // microseconds) before the CTA releases its shared memory
      const uint64_t t0 = globaltimer();
      while (globaltimer() - t0 < 100000ull) {
      }
    }
  } else if (warp == 1 || warp == 11) {
    // ------------------------------------------------------------ MMA issuers (the leader's)
    // QK (warp 1) and PV (warp 11) are issued by two warps of the leader CTA; they accumulate
    // into disjoint TMEM (S and O) of both CTAs and are ordered against each other only through
    // the barriers. Lane 0 waits on the barriers and issues; the other lanes follow it.
    constexpr uint32_t IDESC_QK = idesc_bf16(2 * kM, kBN, false);
    constexpr uint32_t IDESC_PV = idesc_bf16(2 * kM, kDV, true);
    auto wait1 = [&](uint32_t bar, uint32_t parity) -> bool {
      const bool r = lane == 0 ? mbar_wait_inline(bar, parity, wc) : false;
      return __shfl_sync(0xffffffffu, r ? 1 : 0, 0) != 0;
    };
    bool ok = true;
    int32_t J = 0;  // tiles of this cluster's earlier units
    int32_t ui = 0;
    int32_t nof = 0;  // head_dim 256: units with tiles whose PVs this warp has issued
    for (int32_t w = unit_at(0); leader && ok && w < nunits; w = unit_at(++ui)) {
      const int32_t ntiles = tc_unit(a, w, NDH, 0).ntiles;
      if (warp == 1) {
        ok = wait1(QFULL, ui & 1);  // this unit's Q is in place in both CTAs
        for (int32_t j = 0; ok && j < ntiles; ++j) {
          const int32_t JJ = J + j;
          const int sb = JJ % NSB;
          // S buffer sb is free once both CTAs' softmax warps have read S(JJ - 2)
          ok = wait1(SFREE + 8 * sb, ((JJ / NSB) & 1) ^ 1);
          if (!ok) break;
          const uint32_t dS = tmem + kTmS + sb * kBN;
          for (int pp = 0; ok && pp < KP; ++pp) {
            const int sidx = KSLOT(JJ, pp);
            ok = wait1(FULL(sidx), KROUND(JJ, pp) & 1);
            if (!ok) break;
            tc_fence_after();
            // descriptors advance by 32 B per K step inside a 128-byte swizzle row and by one
            // 64-column chunk every 4 steps: 1024 B in a K slot (8-key atoms 4096 B apart),
            // kM x 128 B in shared-memory Q
            const uint64_t kd0 = sdesc(sSlots + sidx * kSlotBytes, 16, 4096);
            if (pp == 0) {
#pragma unroll
              for (int kk = 0; kk < 16; ++kk) {
                const uint64_t kd = kd0 + (uint64_t)(((kk >> 2) * 1024 + (kk & 3) * 32) >> 4);
                mma_ts<IDESC_QK>(dS, tmem + kTmQ + kk * 8, kd, kk > 0 ? 1u : 0u);
              }
            } else {
              // an opaque copy of Q's base descriptor keeps the compiler from hoisting the 16
              // derived descriptors out of the loop
              uint64_t qd0 = sdesc(sQ, 16, 1024);
              asm volatile("mov.b64 %0, %0;" : "+l"(qd0));
#pragma unroll
              for (int kk = 0; kk < 16; ++kk) {
                const uint64_t kd = kd0 + (uint64_t)(((kk >> 2) * 1024 + (kk & 3) * 32) >> 4);
                const uint64_t qd = qd0 + (uint64_t)(((kk >> 2) * (kM * 128) + (kk & 3) * 32) >> 4);
                mma_ss<IDESC_QK>(dS, qd, kd, 1u);
              }
            }
            // this part's slots are free once its MMAs (and all earlier ones) complete
            mma_commit(EMPTY(sidx));
          }
          if (!ok) break;
          mma_commit(SFULL + 8 * sb);
        }
        // Q's shared-memory parts may be replaced once this unit's QK MMAs have completed
        if (ok && DQK == 512) mma_commit(QFREE);
      } else {
        const int BR = a.box_rows_v;
        const uint32_t lbo = (uint32_t)BR * 128u, sbo = BR >= 16 ? 1024u : (uint32_t)BR * 256u;
        if (DQK == 256 && ntiles > 0) {
          // the unit's first PV starts O afresh: only once every softmax warp (both CTAs) has
          // read the previous unit's O (a tile's P comes from one warp of each pair here, so
          // PFULL alone does not say that the other warp's epilogue is done)
          if (nof > 0) ok = wait1(OFREE, (nof - 1) & 1);
          ++nof;
        }
        for (int32_t jp = 0; ok && jp < ntiles; ++jp) {
          const int32_t JJ = J + jp;
          const int pb = JJ % NSB;
          const int sidx = VSLOT(JJ);
          ok = wait1(FULL(sidx), (JJ / NVR) & 1) && wait1(PFULL + 8 * pb, (JJ / NSB) & 1);
          if (!ok) break;
          tc_fence_after();
          const uint32_t vs = sSlots + sidx * kSlotBytes;
          // V slot: page-major boxes of BR rows, each [2 chunks][BR rows][128 B]
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk) {
            const uint32_t key = 16u * kk;
            const uint32_t va = vs + (key / BR) * (BR * 256u) + (key % BR) * 128u;
            // P buffer: K-major, 128-byte swizzled rows of 64 keys; a K step is 32 bytes. The
            // unit's first MMA starts O afresh.
            mma_ss<IDESC_PV>(tmem + kTmO, sdesc(sP + (JJ % C::NPB) * C::P_BUF + kk * 32, 16, 1024),
                             sdesc(va, lbo, sbo), (jp > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(EMPTY(sidx));
          mma_commit(PVDONE + 8 * pb);
        }
      }
      J += ntiles;
    }
    // arrives (in both CTAs) once every MMA this warp issued has completed; waited on before
    // the pair frees its tensor memory
    if (leader) mma_commit(DRAIN);
  } else if (warp >= 2 && warp <= 9) {
    // ------------------------------------------------------------ softmax + epilogue
    // Two warps per TMEM lane quarter: half h = 0 owns key columns [0,32) of each tile and
    // output columns [0,128), half h = 1 the other halves. Each half keeps its own partial row
    // sum. At the end of a unit the warps store the next unit's Q columns into TMEM (the QK
    // MMAs of this unit are complete), so its first QK products overlap this unit's epilogue.
    // Arrivals that the leader's MMA warps wait on go to the leader's barriers.
    const int quarter = warp & 3;
    const int h = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t pair_bar = PAIRB + 8 * quarter;  // meeting point of the two warps sharing these rows
    uint32_t pair_phase = 0;
    bool ok = true;
    constexpr int HC = kBN / 2;  // key columns per half
    // head_dim 256: this warp's quarter of its own P buffer (its 32 rows x 128 bytes, rows
    // 128-byte swizzled) is free between its P writes and serves to transpose the epilogue's
    // output from the row-per-lane layout of TMEM to coalesced global stores (eight lanes per
    // 128-byte piece of a row, four rows per instruction: lane l takes row 4 i + l / 8, piece
    // l mod 8).
    unsigned char* const tbuf = gbase + (sP - base) + h * C::P_BUF + quarter * 4096;
    const int crow = lane >> 3, cpc = lane & 7;
    // G divides the 128 rows of a tile, so it is a power of two: rows split into (token, head)
    // by shift and mask
    const int gsh = __ffs(G) - 1;
    const int32_t gmask = G - 1;
    // Q rows into TMEM (bf16 pairs, the A operand layout of QK). head_dim 512: this warp's d
    // columns [128h, 128h + 128) of the first 256-d part, one 32-byte load per row and lane.
    auto load_q128 = [&](const TcUnit& v, int d0) {
      const bool valid = row < v.ntok * G;
      const uint4* src = reinterpret_cast<const uint4*>(
          a.q + ((int64_t)(v.q0 + v.tok0 + (row >> gsh)) * Hq + v.g * G + (row & gmask)) * DQK + d0);
      // all loads in flight before the first store; 32-byte loads halve the instructions, each
      // of which touches 32 rows (one per lane)
      uint32_t w[64];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (valid) {
          asm volatile("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                       : "=r"(w[8 * q]), "=r"(w[8 * q + 1]), "=r"(w[8 * q + 2]), "=r"(w[8 * q + 3]),
                         "=r"(w[8 * q + 4]), "=r"(w[8 * q + 5]), "=r"(w[8 * q + 6]), "=r"(w[8 * q + 7])
                       : "l"(src + 2 * q));
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) w[8 * q + e] = 0u;
        }
      }
      tmem_st32(tl + kTmQ + d0 / 2, w);
      tmem_st32(tl + kTmQ + d0 / 2 + 32, w + 32);
      tmem_wait_st();
    };
    // head_dim 256: Q of the cluster's k-th unit from the staging buffer (TMA-written as four
    // 64-d pieces of [128 rows][128 swizzled bytes]) into TMEM, this warp's 32 rows; then the
    // buffer is released to the K producer
    auto copy_q256 = [&](int32_t k) -> bool {
      if (!__all_sync(0xffffffffu, mbar_wait(QSFULL, k & 1, wc))) return false;
      const unsigned char* src = gbase + (sQ - base) + row * 128;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t w[32];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint4 y = *reinterpret_cast<const uint4*>(src + c * (kM * 128) + ((q ^ (row & 7)) << 4));
          w[4 * q] = y.x;
          w[4 * q + 1] = y.y;
          w[4 * q + 2] = y.z;
          w[4 * q + 3] = y.w;
        }
        tmem_st32(tl + kTmQ + c * 32, w);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(QSFREE);
      tmem_wait_st();
      return true;
    };
    auto q_stored = [&]() {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cl(LEAD(QFULL));
    };
    // head_dim 256: the warp of each pair that takes the unit's first tile moves all 256 Q
    // columns of the cluster's k-th unit in from the staging buffer; head_dim 512: each warp
    // loads its 128 columns of Q's first part
    auto store_q = [&](const TcUnit& v, int32_t k) -> bool {
      tc_fence_after();  // after the wait that showed the previous QK MMAs complete
      if (DQK == 256) {
        if (!copy_q256(k)) return false;
      } else {
        load_q128(v, h * 128);
      }
      q_stored();
      return true;
    };
    int32_t J = 0;  // tiles of this cluster's earlier units
    TcUnit u;
    int32_t ui = 0;
    if (unit_at(0) < nunits) {
      u = tc_unit(a, unit_at(0), NDH, (int32_t)rank);
      if (DQK != 256 || h == 0) ok = store_q(u, 0);
    }
    for (int32_t w = unit_at(0); ok && w < nunits; w = unit_at(++ui)) {
      const int32_t ntiles = u.ntiles;
      const bool rvalid = row < u.ntok * G;
      const int32_t prow = u.sp + u.tok0 + (row >> gsh);
      const int32_t rlo = W >= 0 ? max(u.kv_start, prow - W) : u.kv_start;
      const int32_t rhi = min(prow + 1, u.kv_len);
      float m_ref = -INFINITY, l = 0.f;
      if constexpr (DQK == 256) {
        // Tile-parity softmax: the two warps of a lane quarter take alternate key tiles (warp h
        // the tiles with JJ mod 2 == h, all 64 keys of each), so one warp's exponentials overlap
        // the other's loads and maximum. The rows' running reference passes from tile to tile
        // between the two warps through shared memory (hm[tile parity][row], one mbarrier per
        // parity and quarter, bounded waits); each warp keeps its own partial row sum, and the
        // two are brought to the unit's final reference and added at the end of the unit. The
        // warp whose tile raises the reference rescales all of O's columns for its rows.
        float* hm = xl + 2 * kM;  // [tile parity][row]
        float m_mine = -INFINITY;  // the reference this warp's last tile used
        for (int32_t j = 0; ok && j < ntiles; ++j) {
          const int32_t JJ = J + j;
          if ((JJ & 1) != h) continue;
          const int b = JJ & 1;  // this warp's S and P buffers
          if (!__all_sync(0xffffffffu, mbar_wait_inline(SFULL + 8 * b, (JJ >> 1) & 1, wc))) { ok = false; break; }
          tc_fence_after();
          uint32_t sv[kBN];
          tmem_ld32(tl + kTmS + b * kBN, sv);
          tmem_ld32(tl + kTmS + b * kBN + 32, sv + 32);
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          // this warp has read S(JJ): the S buffer is free for QK(JJ + 2) once all have
          if (lane == 0) mbar_arrive_cl(LEAD(SFREE + 8 * b));
          const int32_t kb = u.kb0 + j * kBN;
          const bool interior = __all_sync(0xffffffffu, rvalid && kb >= rlo && kb + kBN <= rhi);
          if (!interior) {
#pragma unroll
            for (int k = 0; k < kBN; ++k) {
              const int32_t key = kb + k;
              const bool vis = rvalid && key >= rlo && key < rhi;
              sv[k] = vis ? sv[k] : 0xFF800000u;  // -inf
            }
          }
          // this tile's row maximum in log2 units; t holds the values the exponent scales
          float t[kBN];
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
          float mx;
          const float tscale = a.scale_log2 > 0.f ? a.scale_log2 : 1.f;
          if (a.scale_log2 > 0.f) {
#pragma unroll
            for (int k = 0; k < kBN; ++k) {
              t[k] = __uint_as_float(sv[k]);
              m4[k & 3] = fmaxf(m4[k & 3], t[k]);
            }
            mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * a.scale_log2;
          } else {
#pragma unroll
            for (int k = 0; k < kBN; ++k) {
              t[k] = sv[k] == 0xFF800000u ? -INFINITY : __uint_as_float(sv[k]) * a.scale_log2;
              m4[k & 3] = fmaxf(m4[k & 3], t[k]);
            }
            mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
          }
          // the reference after the previous tile (the other warp's), then this tile's
          float m_prev = -INFINITY;
          if (j > 0) {
            const int32_t jp = JJ - 1;
            if (!__all_sync(0xffffffffu, mbar_wait_inline(PAIRX + 8 * ((jp & 1) * 4 + quarter), (jp >> 1) & 1, wc))) {
              ok = false;
              break;
            }
            m_prev = hm[(jp & 1) * kM + row];
          }
          // new reference with headroom above this maximum, so later growth rarely rescales
          const float m_new = mx > m_prev + kRescaleLog2 ? mx + kHeadroomLog2 : m_prev;
          hm[(JJ & 1) * kM + row] = m_new;
          __syncwarp();
          if (lane == 0) mbar_arrive(PAIRX + 8 * ((JJ & 1) * 4 + quarter));
          if (m_mine != m_new) {
            if (m_mine != -INFINITY) l *= ex2(m_mine - m_new);
            m_mine = m_new;
          }
          const float mu = m_new == -INFINITY ? 0.f : m_new;
          uint32_t pk[kBN / 2];
          {
            // exponents and row sums on fp32 pairs; the row sum adds the bf16-rounded weights the
            // PV product uses, so O / l is an exact weighted average of V rows
            const float2 ts2 = make_float2(tscale, tscale), nmu2 = make_float2(-mu, -mu);
            float2 sa = make_float2(0.f, 0.f), sb2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int k = 0; k < kBN / 2; ++k) {
              const float2 e = __ffma2_rn(make_float2(t[2 * k], t[2 * k + 1]), ts2, nmu2);
              pk[k] = pack_bf16(ex2(e.x), ex2(e.y));
              const float2 wv = make_float2(__uint_as_float(pk[k] << 16), __uint_as_float(pk[k] & 0xFFFF0000u));
              if (k & 1) sb2 = __fadd2_rn(sb2, wv);
              else sa = __fadd2_rn(sa, wv);
            }
            l += (sa.x + sb2.x) + (sa.y + sb2.y);
          }
          // P buffer b is free once PV(JJ - 2) has read it
          if (!__all_sync(0xffffffffu, mbar_wait_inline(PVDONE + 8 * b, ((JJ >> 1) & 1) ^ 1, wc))) { ok = false; break; }
          {
            // the row's 64 keys: eight 16-byte chunks of its 128-byte row, swizzled by the row
            // within its 8-row atom
            unsigned char* prow_p = gbase + (sP - base) + b * C::P_BUF + (row >> 3) * 1024 + (row & 7) * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<uint4*>(prow_p + ((c ^ (row & 7)) << 4)) =
                  make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
          }
          // (after P is written, so the exponents' registers are free)
          const bool resc = m_prev != -INFINITY && m_new != m_prev;
          if (__any_sync(0xffffffffu, resc)) {
            // O holds PV(0 .. JJ - 1) at the old reference: rescale all its columns before PV(JJ)
            const float alpha = resc ? ex2(m_prev - m_new) : 1.f;
            const int32_t jp = JJ - 1;
            if (!__all_sync(0xffffffffu, mbar_wait(PVDONE + 8 * (jp % NSB), (jp / NSB) & 1, wc))) { ok = false; break; }
            tc_fence_after();
            for (int c = 0; c < kDV / 32; ++c) {
              uint32_t o[32];
              const uint32_t col = kTmO + c * 32;
              tmem_ld32(tl + col, o);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
              tmem_st32(tl + col, o);
            }
            tmem_wait_st();
          }
          fence_proxy_async();  // the PV MMA reads P through the async proxy
          tc_fence_before();    // and after any rescaling of O in TMEM above
          __syncwarp();
          if (lane == 0) mbar_arrive_cl(LEAD(PFULL + 8 * b));
        }
        // the unit's final reference is its last tile's; this warp's partial sum follows it
        if (ok && ntiles > 0) {
          const int32_t jl = J + ntiles - 1;
          float m_fin = m_mine;
          if ((jl & 1) != h) {
            if (!__all_sync(0xffffffffu, mbar_wait_inline(PAIRX + 8 * ((jl & 1) * 4 + quarter), (jl >> 1) & 1, wc)))
              ok = false;
            else
              m_fin = hm[(jl & 1) * kM + row];
          }
          if (ok && m_fin != m_mine) {
            if (m_mine != -INFINITY) l *= ex2(m_mine - m_fin);
            m_mine = m_fin;
          }
        }
        m_ref = m_mine;
      } else {
      for (int32_t j = 0; ok && j < ntiles; ++j) {
        const int32_t JJ = J + j;
        const int b = JJ % NSB;
        if (!__all_sync(0xffffffffu, mbar_wait_inline(SFULL + 8 * b, (JJ / NSB) & 1, wc))) { ok = false; break; }
        tc_fence_after();
        float mx;
        // this thread's 32 keys (masked keys: -inf); log2 units are t * tscale
        float t[HC];
        const float tscale = a.scale_log2 > 0.f ? a.scale_log2 : 1.f;
        const int32_t kb = u.kb0 + j * kBN;
        {
        // both warps of the pair read the whole 64-key row: the row maximum needs no exchange
        uint32_t sv[kBN];
        tmem_ld32(tl + kTmS + b * kBN, sv);
        tmem_ld32(tl + kTmS + b * kBN + 32, sv + 32);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        // this warp has read S(JJ): the S buffer is free for QK(JJ + 2) once all have
        if (lane == 0) mbar_arrive_cl(LEAD(SFREE + 8 * b));
        const bool interior = __all_sync(0xffffffffu, rvalid && kb >= rlo && kb + kBN <= rhi);
        if (!interior) {
#pragma unroll
          for (int k = 0; k < kBN; ++k) {
            const int32_t key = kb + k;
            const bool vis = rvalid && key >= rlo && key < rhi;
            sv[k] = vis ? sv[k] : 0xFF800000u;  // -inf
          }
        }
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (a.scale_log2 > 0.f) {
          // a positive scale keeps the maximum where it was, and masked keys at -inf
#pragma unroll
          for (int k = 0; k < kBN; ++k) m4[k & 3] = fmaxf(m4[k & 3], __uint_as_float(sv[k]));
          mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * a.scale_log2;
#pragma unroll
          for (int k = 0; k < HC; ++k) t[k] = __uint_as_float(h ? sv[HC + k] : sv[k]);  // scaled below
        } else {
#pragma unroll
          for (int k = 0; k < kBN; ++k)
            m4[k & 3] = fmaxf(m4[k & 3], sv[k] == 0xFF800000u ? -INFINITY : __uint_as_float(sv[k]) * a.scale_log2);
          mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
#pragma unroll
          for (int k = 0; k < HC; ++k) {
            const uint32_t v = h ? sv[HC + k] : sv[k];
            t[k] = v == 0xFF800000u ? -INFINITY : __uint_as_float(v) * a.scale_log2;
          }
        }
        }
        float alpha = 1.f;
        bool resc = false;
        if (mx > m_ref + kRescaleLog2) {
          // new reference with headroom above this maximum, so later growth rarely rescales
          const float m_new = mx + kHeadroomLog2;
          alpha = m_ref == -INFINITY ? 0.f : ex2(m_ref - m_new);
          resc = m_ref != -INFINITY;
          l *= alpha;
          m_ref = m_new;
        }
        if (j > 0 && __any_sync(0xffffffffu, resc)) {
          const int32_t jp = JJ - 1;
          if (!__all_sync(0xffffffffu, mbar_wait(PVDONE + 8 * (jp % NSB), (jp / NSB) & 1, wc))) { ok = false; break; }
          tc_fence_after();
          for (int c = 0; c < kDV / 64; ++c) {
            uint32_t o[32];
            const uint32_t col = kTmO + h * (kDV / 2) + c * 32;
            tmem_ld32(tl + col, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(tl + col, o);
          }
          tmem_wait_st();
        }
        const float mu = m_ref == -INFINITY ? 0.f : m_ref;
        uint32_t pk[HC / 2];
        {
          // exponents and row sums on fp32 pairs; the row sum adds the bf16-rounded weights the
          // PV product uses, so O / l is an exact weighted average of V rows (a dominant key's
          // rounding cancels)
          const float2 ts2 = make_float2(tscale, tscale), nmu2 = make_float2(-mu, -mu);
          float2 sa = make_float2(0.f, 0.f), sb2 = make_float2(0.f, 0.f);
#pragma unroll
          for (int k = 0; k < HC / 2; ++k) {
            const float2 e = __ffma2_rn(make_float2(t[2 * k], t[2 * k + 1]), ts2, nmu2);
            pk[k] = pack_bf16(ex2(e.x), ex2(e.y));
            const float2 w = make_float2(__uint_as_float(pk[k] << 16), __uint_as_float(pk[k] & 0xFFFF0000u));
            if (k & 1) sb2 = __fadd2_rn(sb2, w);
            else sa = __fadd2_rn(sa, w);
          }
          l += (sa.x + sb2.x) + (sa.y + sb2.y);
        }
        // P buffer JJ mod NPB is free once PV(JJ - NPB) has read it
        if (C::NPB == 2) {
          if (!__all_sync(0xffffffffu, mbar_wait_inline(PVDONE + 8 * b, ((JJ / NSB) & 1) ^ 1, wc))) { ok = false; break; }
        } else if (JJ > 0) {
          const int32_t jp = JJ - 1;
          if (!__all_sync(0xffffffffu, mbar_wait_inline(PVDONE + 8 * (jp % NSB), (jp / NSB) & 1, wc))) { ok = false; break; }
        }
        {
          // this row's 32 keys: four 16-byte chunks h*4 .. h*4+3 of its 128-byte row, at
          // positions swizzled by the row within its 8-row atom
          unsigned char* prow_p = gbase + (sP - base) + (JJ % C::NPB) * C::P_BUF + (row >> 3) * 1024 + (row & 7) * 128;
#pragma unroll
          for (int c = 0; c < 4; ++c)
            *reinterpret_cast<uint4*>(prow_p + (((h * 4 + c) ^ (row & 7)) << 4)) =
                make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        }
        fence_proxy_async();  // the PV MMA reads P through the async proxy
        tc_fence_before();    // and after any rescaling of O in TMEM above
        __syncwarp();
        if (lane == 0) mbar_arrive_cl(LEAD(PFULL + 8 * b));
      }
      }
      if (!ok) break;
      const int32_t wn = unit_at(ui + 1);
      TcUnit un;
      if (wn < nunits) un = tc_unit(a, wn, NDH, (int32_t)rank);
      if constexpr (DQK == 256) {
        // The row sum is the sum of the two warps' partial sums, swapped through shared memory.
        // The warp that wrote the last tile's P waits for that tile's PV before publishing (its
        // own earlier waits keep that PVDONE barrier at most a phase behind); the other warp
        // publishes at once, so the partner's epilogue does not wait for its Q load, and waits
        // for the last PV after the exchange (before it, the barrier of the other parity can be
        // two phases behind this warp's view and a parity wait would pass early). A warp has
        // read the partner's value before the partner writes its next one: that write follows
        // the next unit's first PV, or the other warp's next tile, and both wait for this
        // warp's epilogue (OFREE, the reference handoff).
        const int32_t jl = J + ntiles - 1;
        const bool last = ntiles > 0 && (jl & 1) == h;
        if (last) ok = __all_sync(0xffffffffu, mbar_wait(PVDONE + 8 * (jl % NSB), (jl / NSB) & 1, wc));
        if (ok && ntiles > 0) {
          xl[h * kM + row] = l;
          __syncwarp();
          if (lane == 0) mbar_arrive(pair_bar);
        }
        // The warp that takes the next unit's first tile stores its Q now: this unit's QK MMAs
        // have completed, since that warp has seen the last tile's S through the reference
        // handoff (or, in a unit without tiles, at the end of an earlier unit).
        if (ok && wn < nunits && ((J + ntiles) & 1) == h) ok = store_q(un, ui + 1);
        if (ok && ntiles > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait(pair_bar, pair_phase, wc));
          pair_phase ^= 1u;
          if (ok && !last) ok = __all_sync(0xffffffffu, mbar_wait(PVDONE + 8 * (jl % NSB), (jl / NSB) & 1, wc));
          if (ok) l = xl[row] + xl[kM + row];
        }
      } else {
        // the next unit's Q columns: this unit's QK MMAs are complete (every S was read)
        if (wn < nunits) store_q(un, ui + 1);
        if (ntiles > 0) {
          const int32_t jl = J + ntiles - 1;
          ok = __all_sync(0xffffffffu, mbar_wait(PVDONE + 8 * (jl % NSB), (jl / NSB) & 1, wc));
          // the row sum is the sum of both halves' partial sums, swapped through shared memory.
          // The partner has read this unit's value before this warp writes the next one: that
          // write waits for the next unit's last PV, which needs the partner's P of that tile,
          // which it writes after this unit's epilogue.
          if (ok) {
            xl[h * kM + row] = l;
            __syncwarp();
            if (lane == 0) mbar_arrive(pair_bar);
            ok = __all_sync(0xffffffffu, mbar_wait(pair_bar, pair_phase, wc));
            pair_phase ^= 1u;
            if (ok) l = xl[row] + xl[kM + row];
          }
        }
      }
      if (ok) {
        // epilogue: normalise this thread's 128 output columns [128h, 128h + 128) of the row
        tc_fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        if (a.lse && rvalid && h == 0 && u.dh == 0)  // both output halves of hd512 agree
          a.lse[(int64_t)(u.q0 + u.tok0 + (row >> gsh)) * Hq + u.g * G + (row & gmask)] =
              l > 0.f ? (m_ref + log2f(l)) * 0.69314718055994531f : -INFINITY;
        if (DQK == 256) {
          // each 64-column half of this warp's 128 columns goes through the transposition
          // buffer (free: every PV of the unit has completed) and out in coalesced 16-byte
          // stores, four rows per instruction; rows past the tile's tokens are not written
          const int32_t nvalid = u.ntok * G;
          __nv_bfloat16* const obase = a.out + (int64_t)(u.q0 + u.tok0) * Hq * DQK + (int64_t)u.g * G * DQK +
                                       u.dh * kDV + h * (kDV / 2) + cpc * 8;
#pragma unroll 1
          for (int bx = 0; bx < 2; ++bx) {
            uint32_t wv[32];
            if (ntiles > 0) {
              uint32_t o[64];
              tmem_ld32(tl + kTmO + h * (kDV / 2) + bx * 64, o);
              tmem_ld32(tl + kTmO + h * (kDV / 2) + bx * 64 + 32, o + 32);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e)
                wv[e] = pack_bf16(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
            } else {
#pragma unroll
              for (int e = 0; e < 32; ++e) wv[e] = 0u;
            }
#pragma unroll
            for (int k = 0; k < 8; ++k)
              *reinterpret_cast<uint4*>(tbuf + lane * 128 + ((k ^ (lane & 7)) << 4)) =
                  make_uint4(wv[4 * k], wv[4 * k + 1], wv[4 * k + 2], wv[4 * k + 3]);
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int r = 4 * i + crow;
              const int32_t R = quarter * 32 + r;
              if (R < nvalid) {
                const uint4 x = *reinterpret_cast<const uint4*>(tbuf + r * 128 + ((cpc ^ (r & 7)) << 4));
                *reinterpret_cast<uint4*>(obase + ((int64_t)(R >> gsh) * Hq + (R & gmask)) * DQK + bx * 64) = x;
              }
            }
            __syncwarp();  // read before the next half overwrites the buffer
          }
        } else {
          // head_dim 512: 256 contiguous bytes of the row per thread
          __nv_bfloat16* dst = a.out + ((int64_t)(u.q0 + u.tok0 + (row >> gsh)) * Hq + u.g * G + (row & gmask)) * DQK +
                               u.dh * kDV + h * (kDV / 2);
          for (int c2 = 0; c2 < kDV / 64; c2 += 2) {
            // two 32-column loads in flight per wait
            uint32_t o[64];
            tmem_ld32(tl + kTmO + h * (kDV / 2) + c2 * 32, o);
            tmem_ld32(tl + kTmO + h * (kDV / 2) + c2 * 32 + 32, o + 32);
            tmem_wait_ld();
            if (rvalid) {
#pragma unroll
              for (int c = 0; c < 2; ++c) {
                uint32_t wv[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                  wv[e] = ntiles == 0 ? 0u
                                      : pack_bf16(__uint_as_float(o[32 * c + 2 * e]) * inv,
                                                  __uint_as_float(o[32 * c + 2 * e + 1]) * inv);
                // 32-byte stores: each instruction touches 32 rows (one per lane)
                __nv_bfloat16* d = dst + (c2 + c) * 32;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
                  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(d + 16 * hh),
                               "r"(wv[8 * hh]), "r"(wv[8 * hh + 1]), "r"(wv[8 * hh + 2]), "r"(wv[8 * hh + 3]),
                               "r"(wv[8 * hh + 4]), "r"(wv[8 * hh + 5]), "r"(wv[8 * hh + 6]), "r"(wv[8 * hh + 7])
                               : "memory");
              }
            }
          }
        }
        // the next unit's first PV overwrites O only after these reads
        tc_fence_before();
        if (DQK == 256 && ntiles > 0) {
          __syncwarp();
          if (lane == 0) mbar_arrive_cl(LEAD(OFREE));
        }
      }
      J += ntiles;
      u = un;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1 && lane == 0) {
    // every MMA of the pair has completed once the leader's final commits have arrived (in
    // both CTAs); a wait that runs out is reported like any other
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(DRAIN, 0)) {
      if (globaltimer() - t0 > a.wait_ns) {
        atomicOr(a.status, kStatusTimeout);
        break;
      }
    }
  }
  __syncthreads();
  // neither CTA frees its tensor memory or leaves while the other may still use the pair's
  cluster_sync();
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
  CUtensorMap tq, tkv, tv;
  // Q: dims (d, head, token); a box is 64 d x G heads x TQ tokens
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
  const int32_t brk = ps < kKH ? ps : kKH;  // K rows per box: a page, or a CTA's 32-key half of one
  const int32_t brv = ps < kBN ? ps : kBN;  // V rows per box
  {
    // K: dims (64 d, row within an 8-row group, d chunk, 8-row group); one box = brk rows x
    // 256 d of one page, landing as [group][chunk][8 rows][128 B]
    const cuuint64_t rows = (cuuint64_t)a.pool.num_pages * 2 * a.pool.num_kv_heads * ps;
    cuuint64_t dims[4] = {64, 8, (cuuint64_t)DQK / 64, rows / 8};
    cuuint64_t strides[3] = {(cuuint64_t)DQK * 2, 128, (cuuint64_t)DQK * 2 * 8};
    cuuint32_t box[4] = {64, 8, 4, (cuuint32_t)brk / 8};
    cuuint32_t es[4] = {1, 1, 1, 1};
    if (enc(&tkv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, (void*)a.pool.layer_base, dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    // V: dims (64 d, row, d chunk); one box = brv rows x 2 chunks (a CTA's 128 d) of one page
    const cuuint64_t rows = (cuuint64_t)a.pool.num_pages * 2 * a.pool.num_kv_heads * ps;
    cuuint64_t dims[3] = {64, rows, (cuuint64_t)DQK / 64};
    cuuint64_t strides[2] = {(cuuint64_t)DQK * 2, 128};
    cuuint32_t box[3] = {64, (cuuint32_t)brv, 2};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, (void*)a.pool.layer_base, dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  TcArgs t;
  t.plan = a.plan;
  t.q = a.q;
  t.out = a.out;
  t.num_qo_heads = a.num_qo_heads;
  t.group = G;
  t.cta_tile_q = TQ;
  t.window_left = a.window_left;
  t.page_size = ps;
  t.num_pages = a.pool.num_pages;
  t.num_kv_heads = a.pool.num_kv_heads;
  t.box_rows_k = brk;
  t.box_rows_v = brv;
  t.pool_layer = a.pool.layer_base;
  t.stride_page = a.pool.stride_page;
  t.stride_kv = a.pool.stride_kv;
  t.stride_head = a.pool.stride_head;
  t.scale_log2 = a.sm_scale_log2;
  t.lse = a.lse;
  t.status = a.status;
  t.wait_ns = a.wait_ns;
  t.test_withhold = a.test_withhold;

  // the shared-memory opt-in and the SM count, once per device
  static PerDeviceOnce setup;
  int dev = 0, nsm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = setup.get(dev, [dev](int* n) {
    cudaError_t r = cudaFuncSetAttribute(attn_tc_kernel<DQK>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, TcCfg<DQK>::SMEM);
    if (r != cudaSuccess) return r;
    r = cudaDeviceGetAttribute(n, cudaDevAttrMultiProcessorCount, dev);
    if (*n < 1) *n = 1;
    return r;
  }, &nsm);
  if (e != cudaSuccess) return e;
  // one persistent CTA per SM (its shared and tensor memory fill the SM), in clusters of two;
  // cluster i walks the units (pair of query tiles, KV head, 256-column output part) of its
  // rounds
  const int64_t units = (int64_t)a.plan.num_pairs * a.pool.num_kv_heads * (DQK / kDV);
  if (units == 0) return cudaSuccess;
  const int64_t clusters = std::min<int64_t>(units, nsm / 2 > 0 ? nsm / 2 : 1);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * clusters), 1, 1);
  cfg.blockDim = dim3(kThreadsTc, 1, 1);
  cfg.dynamicSmemBytes = TcCfg<DQK>::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, attn_tc_kernel<DQK>, tq, tkv, tv, t);
  if (e != cudaSuccess) return e;
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
