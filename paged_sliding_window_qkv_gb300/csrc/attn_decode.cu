// Decode attention (every request has one query token) as one balanced stream over the step's
// visible keys ("feat(gemma4): paged KV serving across both attention families", Description:
// decode runs the prefill entry at one token per request; "feat(kernels): Rust wrapper for the
// hd256 windowed paged prefill", Description: paged reads, explicit sm_scale, inclusive-distance
// window_left, GQA by integer division, and the split-KV decode form left to measurement).
//
// Work units. The keys one request's query sees under the window, [lo, hi), are cut into units
// of 16 positions aligned from the first key the request holds; one (request, KV head) pair is a
// segment, and the segments in (request, head) order give the step's U units. CTA s of S takes
// units [s U / S, (s + 1) U / S): every CTA streams the same number of units (to one), so the
// split needs no length-dependent tuning, and a segment that starts and ends inside one CTA's
// range is written directly. A segment cut by a range boundary leaves one fp32 record (O / l,
// running maximum m, sum l) per CTA that holds part of it; the merge kernel combines them.
//
// Inside a CTA (persistent: S = SMs x CTAs per SM):
//   warp NW    producer: per unit, one TMA box of 16 key rows x head_dim for K and one for V
//              (a page's rows of one KV head are contiguous; 128-byte swizzle, so the
//              consumers' ldmatrix reads are conflict-free) into a ring of NS stages, with the
//              unit's geometry in a stage header; each segment's Q rows (the G rows of its
//              head group) by a bulk copy into one of NQ Q slots (2 to 8, as many as the Q
//              region holds),
//              which the consumers release when they finish the segment (a slot is read until
//              then). Page ids are resolved 32 boxes at a time, one per lane, each checked
//              against the plan and the pool (a bad id marks the unit skipped and sets the
//              status word; nothing is read through it).
//   consumers, in one of two forms:
//     group up to 4: one warp takes whole units with the products transposed (S^T = K Q^T,
//              O^T = V^T P^T on bf16 mma.sync): the unit's 16 keys, and then 16 output columns at
//              a time, are the MMA rows and the group's query rows are the 8 MMA columns, so no
//              MMA row is padding and no partial sums cross warps;
//     larger groups: NW = D / 128 warps, one per 128 output columns: S = Q K^T partial over the
//              warp's 128 d, partial S exchanged through shared memory (an mbarrier per buffer),
//              the sum taken in one fixed order by every warp (so every warp holds the same S,
//              maximum and weights), O += P V for the warp's columns.
//   Both run the online softmax in log2 units and end a segment with its output or record.
// Decode is bound by HBM: per unit the CTA moves 16 K and 16 V rows of one head (16 KB at
// head_dim 256, 32 KB at 512) and does 4 * 16 * G * D flop on them. A unit's consumer work is a
// chain of dependent steps, so what keeps HBM busy is the number of units in flight per SM: the
// rings are short (3 stages at head_dim 256, 2 at 512) so that 4 (transposed form), 3 or 2
// CTAs share each SM, each with its own producer and consumers.
//
// Every wait is bounded (two seconds of %globaltimer unless the launch passes a shorter limit);
// a wait that runs out sets the device status word and the CTA leaves its loop; a producer that
// gives up waits 100 us for its issued copies to land before the CTA's shared memory is released.
#include "pg_internal.h"

#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>

#include <algorithm>

namespace pg {
namespace {

constexpr int kUnit = 16;                      // keys per unit
constexpr int kMaxDecodeCtas = 608;            // records are sized for this many CTAs (4 per SM)
constexpr float kLn2 = 0.69314718055994531f;

// unit header flags
constexpr int kFirst = 1;   // first unit of its segment in this CTA
constexpr int kLast = 2;    // last unit of its segment in this CTA
constexpr int kSplit = 4;   // the segment also has units in another CTA: write a record
constexpr int kBad = 8;     // out-of-range metadata: the unit was not loaded, skip it
constexpr int kEnd = 16;    // the CTA's last unit

// TR selects the consumer form. false: NW = D / 128 warps share each unit, warp w owning
// columns [128w, 128w + 128) (any group up to 16). true (group up to 4): one warp takes whole
// units with the products transposed, S^T = K Q^T and O^T = V^T P^T, so the keys and the output
// columns fill the 16 MMA rows and the group sits in the 8 MMA columns; with a small Q region
// the CTA fits 4 to an SM.
template <int D, bool TR>
struct DecCfg {
  static constexpr int NW = TR ? 1 : D / 128;    // consumer warps
  static constexpr int NC = D / 64;              // 128-byte chunks of one row
  static constexpr int THREADS = (NW + 1) * 32;
  static constexpr int HALF = kUnit * D * 2;     // K (or V) bytes of one unit
  static constexpr int STAGE = 2 * HALF;         // K, then V
  static constexpr int NS = D == 256 ? 3 : 2;    // stages
  static constexpr int MIN_CTAS = TR ? 4 : D == 256 ? 3 : 2;  // CTAs per SM
  // Q slots share QROWS rows of D: NQ = QROWS / G slots of G rows each (a power of two, 2 to 8
  // slots); MMA rows (or columns) past the group read one zero row
  static constexpr int QROWS = TR ? 8 : 32;
  static constexpr int QBYTES = QROWS * D * 2;
  static constexpr int NQMAX = 8;
  static constexpr int XBUF = TR ? 0 : NW * 32 * 8 * 4;  // partial S of every consumer warp
  static constexpr int OFF_Q = NS * STAGE;
  static constexpr int OFF_ZROW = OFF_Q + QBYTES;  // one row of D zeros
  static constexpr int OFF_X = OFF_ZROW + D * 2;
  static constexpr int OFF_HDR = OFF_X + 2 * XBUF;
  static constexpr int HDR = 32;
  static constexpr int OFF_BAR = OFF_HDR + NS * HDR;
  // FULL[NS], EMPTY[NS], QFULL[NQMAX], QEMPTY[NQMAX], XFULL[2]
  static constexpr int NBAR = 2 * NS + 2 * NQMAX + 2;
  static constexpr int SMEM_USED = OFF_BAR + NBAR * 8 + 16;
  static constexpr int SMEM = SMEM_USED + 1024;  // + alignment of the stage base
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

// Geometry of one unit, written by the producer into the stage header.
struct alignas(16) DecUnit {
  int32_t r, g;       // segment: request, KV head
  int32_t k0;         // position of the unit's first key
  int32_t klo, khi;   // visible positions [klo, khi) of the unit
  int32_t vz;         // V rows [vz, 16) hold no key of the request: they must read as zero
  int32_t flags;
  int32_t rec;        // record slot (0: the CTA's first segment, 1: its last) when split
};

struct DecArgs {
  PlanDev plan;
  const __nv_bfloat16* q;
  __nv_bfloat16* out;
  float* lse;                // optional
  float* rec_o;              // [kMaxDecodeCtas][2][G][D] fp32 (O / l of a split segment)
  float* rec_ml;             // [kMaxDecodeCtas][2][G][2] (m in log2 units, l)
  int64_t* prefix;           // [R + 1] units before request r (all heads); [R] = U
  int32_t num_qo_heads, num_kv_heads, group, page_size, num_pages, window_left;
  int32_t box_rows;          // key rows per TMA box: min(page_size, 16)
  int32_t box_lg, page_lg;   // log2 of box_rows and of page_size (both powers of two)
  float scale_log2;
  int* status;
  uint64_t wait_ns;
};

// ------------------------------------------------------------------ PTX helpers
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
struct Wait {
  volatile int* abort_flag;
  int* status;
  uint64_t limit_ns;
};
// Bounded wait for the phase of the given parity; false when it ran out (or another warp gave up).
__device__ __noinline__ bool bar_wait(uint32_t bar, uint32_t parity, Wait w) {
  if (bar_try(bar, parity)) return true;
  const uint64_t t0 = gtimer();
  while (!bar_try(bar, parity)) {
    if (*w.abort_flag) return false;
    if (gtimer() - t0 > w.limit_ns) {
      atomicOr(w.status, kStatusTimeout);
      *w.abort_flag = 1;
      return false;
    }
  }
  return true;
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_3d(uint32_t dst, const CUtensorMap* tm, int x, int y, int z,
                                       uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(tm), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void mma_bf16(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Byte offset in a unit's K or V half of 16-byte piece u (0..7) of chunk c of key row k: the
// unit lands as 16 / box_rows boxes, each [chunk][box_rows rows][128 B] with the 128-byte
// swizzle (piece index XOR the row's 128-byte line index within the 1024-byte-aligned stage);
// box_rows br is a power of two.
template <int NC>
__device__ __forceinline__ uint32_t kv_off(int k, int c, int u, int br) {
  const int lo = k & (br - 1);
  const uint32_t row = (uint32_t)((k - lo) * (NC * 128) + c * (br * 128) + lo * 128);
  return row + (uint32_t)((u ^ ((row >> 7) & 7)) << 4);
}

// Units of request r's visible keys (one KV head), the unit index of its first visible key and
// the visible range, from the plan's per-request entry (pair table: for a decode plan entry r
// is request r: {0, qo_indptr[r], 1, start_pos, kvp0, kvp1, kv_end, kv_start}).
struct ReqUnits {
  int32_t n, j0, lo, hi, tok, kvp0, kvp1, kv_len, ks0;
};
__device__ __forceinline__ ReqUnits req_units(const DecArgs& a, int32_t r) {
  const int4 e0 = __ldg(reinterpret_cast<const int4*>(a.plan.pair_tab) + 2 * r);
  const int4 e1 = __ldg(reinterpret_cast<const int4*>(a.plan.pair_tab) + 2 * r + 1);
  ReqUnits u;
  const int32_t p = e0.w;  // the query's position
  u.tok = e0.y;
  u.kvp0 = e1.x;
  u.kvp1 = e1.y;
  u.kv_len = e1.z;
  u.ks0 = e1.w;
  u.lo = a.window_left >= 0 ? max(u.ks0, p - a.window_left) : u.ks0;
  u.hi = min(p + 1, u.kv_len);
  if (u.hi > u.lo) {
    u.j0 = (u.lo - u.ks0) / kUnit;
    u.n = (u.hi - 1 - u.ks0) / kUnit - u.j0 + 1;
  } else {
    u.j0 = 0;
    u.n = 0;
  }
  return u;
}

template <int D, bool TR>
__global__ void __launch_bounds__(DecCfg<D, TR>::THREADS, DecCfg<D, TR>::MIN_CTAS)
attn_decode_kernel(const __grid_constant__ CUtensorMap tm_kv, DecArgs a) {
  using C = DecCfg<D, TR>;
  constexpr int NW = C::NW, NS = C::NS, NC = C::NC;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* gb = smem_raw + (base - raw);
  const uint32_t bars = base + C::OFF_BAR;
  auto FULL = [&](int s) { return bars + 8u * s; };
  auto EMPTY = [&](int s) { return bars + 8u * (NS + s); };
  auto QFULL = [&](int q) { return bars + 8u * (2 * NS + q); };
  auto QEMPTY = [&](int q) { return bars + 8u * (2 * NS + C::NQMAX + q); };
  auto XFULL = [&](int x) { return bars + 8u * (2 * NS + 2 * C::NQMAX + x); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gb + C::OFF_BAR + C::NBAR * 8);
  const Wait wt{abort_flag, a.status, a.wait_ns};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t G = a.group, Hq = a.num_qo_heads, Hkv = a.num_kv_heads;
  // Q slots: G rows each, a power of two of them (2 to 8) in the Q region
  const int32_t qslot = G * D * 2;
  const int32_t lnq = (C::QROWS / G) >= 8 ? 3 : (C::QROWS / G) >= 4 ? 2 : 1;
  const int32_t NQ = 1 << lnq;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      bar_init(FULL(s), 1);
      bar_init(EMPTY(s), NW);
    }
    for (int q = 0; q < C::NQMAX; ++q) {
      bar_init(QFULL(q), 1);
      bar_init(QEMPTY(q), NW);
    }
    for (int x = 0; x < 2; ++x) bar_init(XFULL(x), NW);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // the zero row that MMA rows past the group read
  for (int i = threadIdx.x; i < D / 8; i += blockDim.x)
    *reinterpret_cast<uint4*>(gb + C::OFF_ZROW + i * 16) = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();
  // the merge kernel may launch now; it waits for this grid's completion before reading
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp == NW) {
    // ------------------------------------------------------------ producer
    const int32_t R = a.plan.num_req;
    const int32_t S = (int32_t)gridDim.x, s = (int32_t)blockIdx.x;
    // Units of every request (all heads), in warp-wide scans of 32 requests: the total U, and
    // (CTA 0) the prefix for the merge kernel. The first kHeld chunks' counts are loaded at
    // once (one round trip to memory) and stay in registers for the second scan.
    constexpr int kHeld = 8;
    auto units_of = [&](int32_t r) -> int64_t { return r < R ? (int64_t)req_units(a, r).n * Hkv : 0; };
    auto scan32 = [&](int64_t v) {  // inclusive prefix over the warp
      int64_t incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      return incl;
    };
    int64_t held[kHeld];
#pragma unroll
    for (int j = 0; j < kHeld; ++j) held[j] = units_of(32 * j + lane);
    int64_t run = 0;
#pragma unroll
    for (int j = 0; j < kHeld; ++j) {
      if (32 * j < R) {
        const int64_t incl = scan32(held[j]);
        if (s == 0 && 32 * j + lane < R) a.prefix[32 * j + lane] = run + incl - held[j];
        run += __shfl_sync(0xffffffffu, incl, 31);
      }
    }
    for (int32_t c = 32 * kHeld; c < R; c += 32) {
      const int64_t v = units_of(c + lane);
      const int64_t incl = scan32(v);
      if (s == 0 && c + lane < R) a.prefix[c + lane] = run + incl - v;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    const int64_t U = run;
    if (s == 0 && lane == 0) a.prefix[R] = U;
    const int64_t u0 = (int64_t)s * U / S, u1 = (int64_t)(s + 1) * U / S;
    // the request holding unit u0, and the units before it
    int32_t r = 0;
    int64_t rbase = 0;
    run = 0;
    bool found = false;
#pragma unroll
    for (int j = 0; j < kHeld; ++j) {
      if (!found && 32 * j < R) {
        const int64_t incl = scan32(held[j]);
        const uint32_t past = __ballot_sync(0xffffffffu, run + incl > u0);
        if (past) {
          const int f = __ffs(past) - 1;
          r = 32 * j + f;
          rbase = run + __shfl_sync(0xffffffffu, incl - held[j], f);
          found = true;
        } else {
          run += __shfl_sync(0xffffffffu, incl, 31);
        }
      }
    }
    for (int32_t c = 32 * kHeld; !found && c < R; c += 32) {
      const int64_t v = units_of(c + lane);
      const int64_t incl = scan32(v);
      const uint32_t past = __ballot_sync(0xffffffffu, run + incl > u0);
      if (past) {
        const int f = __ffs(past) - 1;
        r = c + f;
        rbase = run + __shfl_sync(0xffffffffu, incl - v, f);
        found = true;
      } else {
        run += __shfl_sync(0xffffffffu, incl, 31);
      }
    }
    const int32_t ps = a.page_size, BR = a.box_rows, LNB = 4 - a.box_lg, NB = 1 << LNB;  // boxes per unit
    const uint32_t box_bytes = (uint32_t)BR * D * 2;
    const int32_t UB = 32 >> LNB;  // units per lookup batch
    int64_t u = u0;
    int32_t i = 0;     // units issued by this CTA
    int32_t nseg = 0;  // segments started by this CTA
    bool ok = true;
    while (ok && u < u1) {
      const ReqUnits q = req_units(a, r);
      const int64_t in_req = u - rbase;
      if (q.n == 0 || in_req >= (int64_t)q.n * Hkv) {  // next request
        rbase += (int64_t)q.n * Hkv;
        ++r;
        continue;
      }
      const int32_t g = (int32_t)(in_req / q.n);
      const int64_t seg0 = rbase + (int64_t)g * q.n;   // the segment's first unit
      const int64_t seg_end = seg0 + q.n;
      const int64_t stop = min(seg_end, u1);
      const bool split = seg0 < u0 || seg_end > u1;
      const int32_t rec = nseg == 0 ? 0 : 1;
      // the segment's query rows into Q slot nseg mod NQ, once the consumers have finished the
      // segment that used it before
      {
        const int qs = nseg & (NQ - 1), use = nseg >> lnq;
        int go = 1;
        if (lane == 0) {
          if (use >= 1 && !bar_wait(QEMPTY(qs), (use - 1) & 1, wt)) {
            go = 0;
          } else {
            bar_arrive_tx(QFULL(qs), (uint32_t)qslot);
            bulk_g2s(base + C::OFF_Q + qs * qslot, a.q + ((int64_t)q.tok * Hq + g * G) * D,
                     (uint32_t)qslot, QFULL(qs));
          }
        }
        if (!__shfl_sync(0xffffffffu, go, 0)) {
          ok = false;
          break;
        }
      }
      const int32_t npg = q.kvp1 - q.kvp0;
      for (int64_t ub = u; ok && ub < stop; ub += UB) {
        // lane l resolves box l % NB of unit ub + l / NB: its page id (or -1 past the keys held,
        // or num_pages when the metadata is out of range)
        const int32_t jl = (int32_t)(ub - seg0) + (lane >> LNB);  // unit within the segment
        const int32_t rel = (q.j0 + jl) * kUnit + (lane & (NB - 1)) * BR;  // key index among those held
        int32_t page = -1, row = 0;
        if (ub + (lane >> LNB) < stop && q.ks0 + rel < q.kv_len) {
          const int32_t lp = rel >> a.page_lg;
          const int32_t pidx = q.kvp0 + (a.plan.ring ? lp % max(npg, 1) : lp);
          page = (pidx < q.kvp1 && pidx < a.plan.num_page_ids) ? a.plan.page_ids[pidx] : a.num_pages;
          if (page < 0 || page >= a.num_pages) page = a.num_pages;
          else row = ((page * 2) * Hkv + g) * ps + (rel & (ps - 1));  // K row; V is Hkv * ps rows later
        }
        const int32_t nb_units = (int32_t)(stop - ub < UB ? stop - ub : UB);
        for (int32_t t = 0; t < nb_units; ++t, ++i) {
          const int st = i % NS;
          const int32_t jj = (int32_t)(ub - seg0) + t;
          const int32_t k0 = q.ks0 + (q.j0 + jj) * kUnit;
          const bool lane_box = (lane >> LNB) == t;
          const bool bad = __any_sync(0xffffffffu, lane_box && page == a.num_pages);
          const uint32_t nload = __popc(__ballot_sync(0xffffffffu, lane_box && page >= 0 &&
                                                                       page < a.num_pages));
          int go = 1;
          if (lane == 0) {
            if (!bar_wait(EMPTY(st), ((i / NS) & 1) ^ 1, wt)) {
              go = 0;
            } else {
              DecUnit h;
              h.r = r;
              h.g = g;
              h.k0 = k0;
              h.klo = max(q.lo, k0);
              h.khi = min(q.hi, k0 + kUnit);
              h.vz = min(max(q.kv_len - k0, 0), kUnit);
              const int64_t uu = ub + t;
              h.flags = (uu == u ? kFirst : 0) | (uu + 1 == stop ? kLast : 0) |
                        (split ? kSplit : 0) | (bad ? kBad : 0) | (uu + 1 == u1 ? kEnd : 0);
              h.rec = rec;
              *reinterpret_cast<DecUnit*>(gb + C::OFF_HDR + st * C::HDR) = h;
              if (bad) {
                atomicOr(a.status, kStatusBounds);
                bar_arrive(FULL(st));
              } else {
                bar_arrive_tx(FULL(st), nload * box_bytes * 2);
              }
            }
          }
          if (!__shfl_sync(0xffffffffu, go, 0)) {
            ok = false;
            break;
          }
          if (!bad && lane_box && page >= 0 && page < a.num_pages) {
            const uint32_t dst = base + st * C::STAGE + (lane & (NB - 1)) * box_bytes;
            tma_3d(dst, &tm_kv, 0, row, 0, FULL(st));                      // K rows
            tma_3d(dst + C::HALF, &tm_kv, 0, row + Hkv * ps, 0, FULL(st));  // V rows
          }
        }
      }
      u = stop;
      ++nseg;
    }
    if (ok && u0 == u1 && lane == 0) {
      // no unit for this CTA (more CTAs than units): one empty unit ends the consumers' loop
      DecUnit h{};
      h.flags = kBad | kEnd;
      *reinterpret_cast<DecUnit*>(gb + C::OFF_HDR) = h;
      bar_arrive(FULL(0));
    }
    if (!ok) {
      const uint64_t t0 = gtimer();
      while (gtimer() - t0 < 100000ull) {
      }
    }
  } else if constexpr (TR) {
    // ------------------------------------------------------------ consumer (whole units)
    // Fragments (m16n8k16): S^T = K Q^T has the unit's 16 keys as rows and the group's query
    // rows as the 8 columns; lane (gid, tig) holds S of keys gid and gid + 8 for query rows 2 tig
    // and 2 tig + 1. O^T = V^T P^T has output columns d as rows: o[mt] holds columns 16 mt + gid
    // and 16 mt + gid + 8 for the same two query rows.
    const int gid = lane >> 2, tig = lane & 3;
    const int BR = a.box_rows;
    float o[16][4];
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    uint32_t qf[16][2];
    int32_t nseg = 0;
    // P as the B operand: lane (gid, tig) needs query row gid at keys 2 tig, 2 tig + 1 (+ 8),
    // which lanes 8 tig + gid / 2 and 8 tig + 4 + gid / 2 hold, in the half gid & 1
    const int src0 = 8 * tig + (gid >> 1), src1 = src0 + 4;
    const uint32_t psel = (gid & 1) ? 0x7632u : 0x5410u;
    for (int32_t i = 0;; ++i) {
      const int st = i % NS;
      if (!bar_wait(FULL(st), (i / NS) & 1, wt)) break;
      const DecUnit h = *reinterpret_cast<const DecUnit*>(gb + C::OFF_HDR + st * C::HDR);
      if (h.flags & kFirst) {
        const int qs = nseg & (NQ - 1);
        if (!bar_wait(QFULL(qs), (nseg >> lnq) & 1, wt)) break;
        // B fragments of Q^T over all D: query row lane & 7 (rows past the group read the zero
        // row), four 8-wide pieces of d per load
        const int qrow = lane & 7;
        const uint32_t qb = qrow < G ? base + C::OFF_Q + qs * qslot + qrow * (D * 2)
                                     : base + C::OFF_ZROW;
#pragma unroll
        for (int pq = 0; pq < D / 32; ++pq) {
          uint32_t r4[4];
          ldsm_x4(qb + (uint32_t)((32 * pq + 8 * (lane >> 3)) * 2), r4);
          qf[2 * pq][0] = r4[0];
          qf[2 * pq][1] = r4[1];
          qf[2 * pq + 1][0] = r4[2];
          qf[2 * pq + 1][1] = r4[3];
        }
        ++nseg;
#pragma unroll
        for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
        m[0] = m[1] = -INFINITY;
        l[0] = l[1] = 0.f;
      }
      const uint32_t kb = base + st * C::STAGE, vb = kb + C::HALF;
      if (!(h.flags & kBad)) {
        // ---- S^T over all D in 16 k-steps, four independent accumulator chains
        float sa[4][4] = {};
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          uint32_t kf[8][4];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int ks = 8 * hb + j;
            ldsm_x4(kb + kv_off<NC>(lane & 15, ks >> 2, 2 * (ks & 3) + (lane >> 4), BR), kf[j]);
          }
#pragma unroll
          for (int j = 0; j < 8; ++j)
            mma_bf16(sa[j & 3], kf[j], qf[8 * hb + j][0], qf[8 * hb + j][1]);
        }
        // ---- mask, scale (log2 units), online softmax per query row (a column here); element
        // e is key k0 + gid + 8 (e >> 1) of query row 2 tig + (e & 1)
        float t[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float sv = (sa[0][e] + sa[1][e]) + (sa[2][e] + sa[3][e]);
          const int32_t key = h.k0 + gid + 8 * (e >> 1);
          t[e] = (key >= h.klo && key < h.khi) ? sv * a.scale_log2 : -INFINITY;
        }
        float mx0 = fmaxf(t[0], t[2]), mx1 = fmaxf(t[1], t[3]);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float n0 = fmaxf(m[0], mx0), n1 = fmaxf(m[1], mx1);
        // a row that has seen no visible key yet keeps weight 0 (reference 0, not -inf)
        const float r0 = n0 == -INFINITY ? 0.f : n0, r1 = n1 == -INFINITY ? 0.f : n1;
        const float al0 = ex2(m[0] - r0), al1 = ex2(m[1] - r1);
        m[0] = n0;
        m[1] = n1;
        const uint32_t plo = pack_bf16(ex2(t[0] - r0), ex2(t[1] - r1));  // key gid
        const uint32_t phi = pack_bf16(ex2(t[2] - r0), ex2(t[3] - r1));  // key gid + 8
        // the row sums add the bf16-rounded weights the PV product uses (this lane's two keys;
        // summed over the lanes at the segment's end)
        auto lo16 = [](uint32_t v) { return __uint_as_float(v << 16); };
        auto hi16 = [](uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); };
        l[0] = l[0] * al0 + (lo16(plo) + lo16(phi));
        l[1] = l[1] * al1 + (hi16(plo) + hi16(phi));
        if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
          for (int n = 0; n < 16; ++n) {
            o[n][0] *= al0; o[n][1] *= al1;
            o[n][2] *= al0; o[n][3] *= al1;
          }
        }
        const uint32_t pb0 = __byte_perm(__shfl_sync(0xffffffffu, plo, src0),
                                         __shfl_sync(0xffffffffu, plo, src1), psel);
        const uint32_t pb1 = __byte_perm(__shfl_sync(0xffffffffu, phi, src0),
                                         __shfl_sync(0xffffffffu, phi, src1), psel);
        // V rows past the keys the request holds may be anything: they read as zero
        if (h.vz < kUnit) {
          for (int idx = lane; idx < (kUnit - h.vz) * NC * 8; idx += 32) {
            const int k = h.vz + idx / (NC * 8);
            *reinterpret_cast<uint4*>(gb + (vb - base) + kv_off<NC>(k, (idx >> 3) % NC, idx & 7, BR)) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          __syncwarp();
        }
        // ---- O^T += V^T P^T: 16 row tiles of 16 output columns, one k-step of 16 keys
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          uint32_t vf[8][4];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int mt = 8 * hb + j;
            ldsm_x4_t(vb + kv_off<NC>((lane & 7) + 8 * (lane >> 4), mt >> 2,
                                      2 * (mt & 3) + ((lane >> 3) & 1), BR),
                      vf[j]);
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) mma_bf16(o[8 * hb + j], vf[j], pb0, pb1);
        }
        if (h.vz < kUnit) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      }
      if (h.flags & kLast) {
        // ---- the segment's output (or this CTA's record of it): query rows 2 tig + j < G
        float lt[2] = {l[0], l[1]};
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          lt[0] += __shfl_xor_sync(0xffffffffu, lt[0], off);
          lt[1] += __shfl_xor_sync(0xffffffffu, lt[1], off);
        }
        const float iv[2] = {lt[0] > 0.f ? 1.f / lt[0] : 0.f, lt[1] > 0.f ? 1.f / lt[1] : 0.f};
        if (h.flags & kSplit) {
          const int64_t rb = ((int64_t)blockIdx.x * 2 + h.rec) * G;
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int row = 2 * tig + j;
            if (row < G) {
              float* dst = a.rec_o + (rb + row) * D + gid;
#pragma unroll
              for (int n = 0; n < 16; ++n) {
                dst[16 * n] = o[n][j] * iv[j];
                dst[16 * n + 8] = o[n][2 + j] * iv[j];
              }
              if (gid == 0)
                *reinterpret_cast<float2*>(a.rec_ml + (rb + row) * 2) = make_float2(m[j], lt[j]);
            }
          }
        } else {
          const int32_t tok = a.plan.qo_indptr[h.r];
          const int64_t row0 = (int64_t)tok * Hq + (int64_t)h.g * G;
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int row = 2 * tig + j;
            if (row < G) {
              __nv_bfloat16* dst = a.out + (row0 + row) * D + gid;
#pragma unroll
              for (int n = 0; n < 16; ++n) {
                dst[16 * n] = __float2bfloat16_rn(o[n][j] * iv[j]);
                dst[16 * n + 8] = __float2bfloat16_rn(o[n][2 + j] * iv[j]);
              }
              if (a.lse && gid == 0)
                a.lse[row0 + row] = lt[j] > 0.f ? (m[j] + log2f(lt[j])) * kLn2 : -INFINITY;
            }
          }
        }
      }
      // the stage (and its header) is released only now; at the segment's end so is its Q slot
      __syncwarp();
      if (lane == 0) {
        bar_arrive(EMPTY(st));
        if (h.flags & kLast) bar_arrive(QEMPTY((nseg - 1) & (NQ - 1)));
      }
      if (h.flags & kEnd) break;
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int w = warp;
    const int gid = lane >> 2, tig = lane & 3;
    const int BR = a.box_rows;
    float o[16][4];
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    uint32_t qa[8][4];
    int32_t nseg = 0;
    int32_t xi = 0;  // exchanges so far (skipped units exchange nothing)
    for (int32_t i = 0;; ++i) {
      const int st = i % NS;
      if (!bar_wait(FULL(st), (i / NS) & 1, wt)) break;
      const DecUnit h = *reinterpret_cast<const DecUnit*>(gb + C::OFF_HDR + st * C::HDR);
      if (h.flags & kFirst) {
        const int qs = nseg & (NQ - 1);
        if (!bar_wait(QFULL(qs), (nseg >> lnq) & 1, wt)) break;
        // this warp's A fragments: rows 0..15 (rows past the group read the zero row), d
        // [128w, 128w + 128) in eight 16-wide k-steps; the slot stays held until the segment ends
        const int qrow = lane & 15;
        const uint32_t qb = qrow < G ? base + C::OFF_Q + qs * qslot + qrow * (D * 2)
                                     : base + C::OFF_ZROW;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          ldsm_x4(qb + (uint32_t)((128 * w + 16 * ks + 8 * (lane >> 4)) * 2), qa[ks]);
        ++nseg;
#pragma unroll
        for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
        m0 = m1 = -INFINITY;
        l0 = l1 = 0.f;
      }
      const uint32_t kb = base + st * C::STAGE, vb = kb + C::HALF;
      if (!(h.flags & kBad)) {
        // ---- partial S over this warp's 128 d (chunks 2w, 2w + 1): keys 0..7 and 8..15
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          uint32_t b[4];
          const int key = (lane & 7) + 8 * (lane >> 4);
          ldsm_x4(kb + kv_off<NC>(key, 2 * w + (ks >> 2), 2 * (ks & 3) + ((lane >> 3) & 1), BR), b);
          mma_bf16(acc[0], qa[ks], b[0], b[1]);
          mma_bf16(acc[1], qa[ks], b[2], b[3]);
        }
        // ---- exchange: every warp sums the NW partials in the same order
        float* xb = reinterpret_cast<float*>(gb + C::OFF_X + (xi & 1) * C::XBUF);
        *reinterpret_cast<float4*>(xb + (w * 32 + lane) * 8) =
            make_float4(acc[0][0], acc[0][1], acc[0][2], acc[0][3]);
        *reinterpret_cast<float4*>(xb + (w * 32 + lane) * 8 + 4) =
            make_float4(acc[1][0], acc[1][1], acc[1][2], acc[1][3]);
        __syncwarp();
        if (lane == 0) bar_arrive(XFULL(xi & 1));
        if (!bar_wait(XFULL(xi & 1), (xi >> 1) & 1, wt)) break;
        ++xi;
        float sv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ww = 0; ww < NW; ++ww) {
          const float4 x0 = *reinterpret_cast<const float4*>(xb + (ww * 32 + lane) * 8);
          const float4 x1 = *reinterpret_cast<const float4*>(xb + (ww * 32 + lane) * 8 + 4);
          sv[0] += x0.x; sv[1] += x0.y; sv[2] += x0.z; sv[3] += x0.w;
          sv[4] += x1.x; sv[5] += x1.y; sv[6] += x1.z; sv[7] += x1.w;
        }
        // ---- mask, scale (log2 units), online softmax; element e of n-tile nt is key
        // k0 + 8 nt + 2 tig + (e & 1) of row gid + 8 (e >> 1)
        float t[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int32_t key = h.k0 + 8 * (e >> 2) + 2 * tig + (e & 1);
          t[e] = (key >= h.klo && key < h.khi) ? sv[e] * a.scale_log2 : -INFINITY;
        }
        float mx0 = fmaxf(fmaxf(t[0], t[1]), fmaxf(t[4], t[5]));
        float mx1 = fmaxf(fmaxf(t[2], t[3]), fmaxf(t[6], t[7]));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
        const float al0 = ex2(m0 - n0), al1 = ex2(m1 - n1);  // -inf - finite: 0
        m0 = n0;
        m1 = n1;
        uint32_t pa[4];
        pa[0] = pack_bf16(ex2(t[0] - n0), ex2(t[1] - n0));
        pa[1] = pack_bf16(ex2(t[2] - n1), ex2(t[3] - n1));
        pa[2] = pack_bf16(ex2(t[4] - n0), ex2(t[5] - n0));
        pa[3] = pack_bf16(ex2(t[6] - n1), ex2(t[7] - n1));
        // the row sums add the bf16-rounded weights the PV product uses
        auto lo16 = [](uint32_t v) { return __uint_as_float(v << 16); };
        auto hi16 = [](uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); };
        l0 = l0 * al0 + ((lo16(pa[0]) + hi16(pa[0])) + (lo16(pa[2]) + hi16(pa[2])));
        l1 = l1 * al1 + ((lo16(pa[1]) + hi16(pa[1])) + (lo16(pa[3]) + hi16(pa[3])));
        if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
          for (int n = 0; n < 16; ++n) {
            o[n][0] *= al0; o[n][1] *= al0;
            o[n][2] *= al1; o[n][3] *= al1;
          }
        }
        // V rows past the keys the request holds may be anything: this warp's two chunks of
        // them read as zero
        if (h.vz < kUnit) {
          for (int idx = lane; idx < (kUnit - h.vz) * 16; idx += 32) {
            const int k = h.vz + idx / 16;
            *reinterpret_cast<uint4*>(gb + (vb - base) +
                                      kv_off<NC>(k, 2 * w + ((idx >> 3) & 1), idx & 7, BR)) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          __syncwarp();
        }
        // ---- O += P V over this warp's 128 columns
#pragma unroll
        for (int np = 0; np < 8; ++np) {
          uint32_t b[4];
          const int key = (lane & 7) + 8 * ((lane >> 3) & 1);
          ldsm_x4_t(vb + kv_off<NC>(key, 2 * w + (np >> 2), 2 * (np & 3) + (lane >> 4), BR), b);
          mma_bf16(o[2 * np], pa, b[0], b[1]);
          mma_bf16(o[2 * np + 1], pa, b[2], b[3]);
        }
        if (h.vz < kUnit) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      }
      if (h.flags & kLast) {
        // ---- the segment's output (or this CTA's record of it)
        float lt0 = l0 + __shfl_xor_sync(0xffffffffu, l0, 1);
        float lt1 = l1 + __shfl_xor_sync(0xffffffffu, l1, 1);
        lt0 += __shfl_xor_sync(0xffffffffu, lt0, 2);
        lt1 += __shfl_xor_sync(0xffffffffu, lt1, 2);
        const float i0 = lt0 > 0.f ? 1.f / lt0 : 0.f, i1 = lt1 > 0.f ? 1.f / lt1 : 0.f;
        if (h.flags & kSplit) {
          const int64_t rb = ((int64_t)blockIdx.x * 2 + h.rec) * G;
#pragma unroll
          for (int n = 0; n < 16; ++n) {
            const int col = 128 * w + 8 * n + 2 * tig;
            if (gid < G)
              *reinterpret_cast<float2*>(a.rec_o + (rb + gid) * D + col) =
                  make_float2(o[n][0] * i0, o[n][1] * i0);
            if (gid + 8 < G)
              *reinterpret_cast<float2*>(a.rec_o + (rb + gid + 8) * D + col) =
                  make_float2(o[n][2] * i1, o[n][3] * i1);
          }
          if (w == 0 && tig == 0) {
            if (gid < G) *reinterpret_cast<float2*>(a.rec_ml + (rb + gid) * 2) = make_float2(m0, lt0);
            if (gid + 8 < G)
              *reinterpret_cast<float2*>(a.rec_ml + (rb + gid + 8) * 2) = make_float2(m1, lt1);
          }
        } else {
          const int32_t tok = a.plan.qo_indptr[h.r];
          const int64_t row0 = (int64_t)tok * Hq + (int64_t)h.g * G;
#pragma unroll
          for (int n = 0; n < 16; ++n) {
            const int col = 128 * w + 8 * n + 2 * tig;
            if (gid < G)
              *reinterpret_cast<uint32_t*>(a.out + (row0 + gid) * D + col) =
                  pack_bf16(o[n][0] * i0, o[n][1] * i0);
            if (gid + 8 < G)
              *reinterpret_cast<uint32_t*>(a.out + (row0 + gid + 8) * D + col) =
                  pack_bf16(o[n][2] * i1, o[n][3] * i1);
          }
          if (a.lse && w == 0 && tig == 0) {
            if (gid < G) a.lse[row0 + gid] = lt0 > 0.f ? (m0 + log2f(lt0)) * kLn2 : -INFINITY;
            if (gid + 8 < G) a.lse[row0 + gid + 8] = lt1 > 0.f ? (m1 + log2f(lt1)) * kLn2 : -INFINITY;
          }
        }
      }
      // the stage (and its header) is released only now; at the segment's end so is its Q slot
      __syncwarp();
      if (lane == 0) {
        bar_arrive(EMPTY(st));
        if (h.flags & kLast) bar_arrive(QEMPTY((nseg - 1) & (NQ - 1)));
      }
      if (h.flags & kEnd) break;
    }
  }
}

// Combine the records of each segment cut by CTA range boundaries, write the rows of segments
// that see no key (out = 0, lse = -inf); segments inside one CTA's range were written directly.
// One CTA per (request, KV head). The request's entry and the unit prefixes are loaded together,
// then each thread loads the (m, l) and columns of up to four records at once and folds them
// in with a running maximum: about two round trips to memory per segment.
template <int D>
__global__ void __launch_bounds__(128) attn_decode_merge_kernel(DecArgs a, int32_t S) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int32_t Hkv = a.num_kv_heads, G = a.group, Hq = a.num_qo_heads;
  const int32_t r = (int32_t)blockIdx.x / Hkv, g = (int32_t)blockIdx.x % Hkv;
  const int64_t U = a.prefix[a.plan.num_req];
  const int64_t pre = a.prefix[r];
  const ReqUnits q = req_units(a, r);
  const int64_t row0 = (int64_t)q.tok * Hq + (int64_t)g * G;
  if (q.n == 0) {
    for (int i = threadIdx.x; i < G * D / 2; i += blockDim.x)
      reinterpret_cast<uint32_t*>(a.out + row0 * D)[i] = 0u;
    if (a.lse && (int)threadIdx.x < G) a.lse[row0 + threadIdx.x] = -INFINITY;
    return;
  }
  const int64_t first = pre + (int64_t)g * q.n, last = first + q.n - 1;  // U > 0 here
  auto cta_of = [&](int64_t x) { return (int32_t)(((x + 1) * S - 1) / U); };
  const int32_t sa = cta_of(first), sb = cta_of(last);
  if (sa == sb) return;
  // the record slot of CTA s: a segment that started before CTA s's range is its first (slot 0);
  // in CTA sa the segment is the first only when the range starts inside it
  const int32_t slot_a = (int64_t)sa * U / S < first ? 1 : 0;
  for (int idx = threadIdx.x; idx < G * (D / 4); idx += blockDim.x) {
    const int row = idx / (D / 4), c4 = idx % (D / 4);
    float M = -INFINITY, den = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int32_t s0 = sa; s0 <= sb; s0 += 4) {
      float2 ml[4];
      float4 v[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int32_t s = s0 + k;
        // CTAs with an empty range (more CTAs than units) hold no record
        const bool holds = s <= sb && (int64_t)s * U / S < (int64_t)(s + 1) * U / S;
        const int64_t rb = ((int64_t)s * 2 + (s == sa ? slot_a : 0)) * G + row;
        ml[k] = holds ? *reinterpret_cast<const float2*>(a.rec_ml + rb * 2) : make_float2(-INFINITY, 0.f);
        v[k] = holds ? *reinterpret_cast<const float4*>(a.rec_o + rb * D + 4 * c4)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (!(ml[k].y > 0.f)) continue;
        const float mn = fmaxf(M, ml[k].x);
        const float so = exp2f(M - mn), w = ml[k].y * exp2f(ml[k].x - mn);  // M = -inf: so = 0
        acc.x = acc.x * so + w * v[k].x; acc.y = acc.y * so + w * v[k].y;
        acc.z = acc.z * so + w * v[k].z; acc.w = acc.w * so + w * v[k].w;
        den = den * so + w;
        M = mn;
      }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    __nv_bfloat16* dst = a.out + (row0 + row) * D + 4 * c4;
    *reinterpret_cast<uint32_t*>(dst) = pack_bf16(acc.x * inv, acc.y * inv);
    *reinterpret_cast<uint32_t*>(dst + 2) = pack_bf16(acc.z * inv, acc.w * inv);
    if (a.lse && c4 == 0) a.lse[row0 + row] = den > 0.f ? (M + log2f(den)) * kLn2 : -INFINITY;
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn_dec() {
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

size_t align16(size_t n) { return (n + 15) & ~(size_t)15; }

template <int D, bool TR>
cudaError_t launch_dec(const AttnArgs& a, cudaStream_t stream) {
  using C = DecCfg<D, TR>;
  EncodeTiledFn enc = encode_fn_dec();
  if (!enc) return cudaErrorNotSupported;
  const int32_t ps = a.pool.page_size, Hkv = a.pool.num_kv_heads, G = a.group;
  const int32_t br = ps < kUnit ? ps : kUnit;
  CUtensorMap tm;
  {
    // rows of D elements: (page, K/V, head, slot) flattened; a box = br rows x D (all chunks)
    const cuuint64_t rows = (cuuint64_t)a.pool.num_pages * 2 * Hkv * ps;
    cuuint64_t dims[3] = {64, rows, (cuuint64_t)D / 64};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, 128};
    cuuint32_t box[3] = {64, (cuuint32_t)br, (cuuint32_t)D / 64};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, (void*)a.pool.layer_base, dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  DecArgs d;
  d.plan = a.plan;
  d.q = a.q;
  d.out = a.out;
  d.lse = a.lse;
  const int32_t R = a.plan.num_req;
  unsigned char* ws = reinterpret_cast<unsigned char*>(a.ws_raw);
  d.prefix = reinterpret_cast<int64_t*>(ws);
  d.rec_ml = reinterpret_cast<float*>(ws + align16((size_t)(R + 1) * 8));
  d.rec_o = d.rec_ml + (size_t)kMaxDecodeCtas * 2 * G * 2;
  d.num_qo_heads = a.num_qo_heads;
  d.num_kv_heads = Hkv;
  d.group = G;
  d.page_size = ps;
  d.num_pages = a.pool.num_pages;
  d.window_left = a.window_left;
  d.box_rows = br;
  d.box_lg = 31 - __builtin_clz((unsigned)br);
  d.page_lg = 31 - __builtin_clz((unsigned)ps);
  d.scale_log2 = a.sm_scale_log2;
  d.status = a.status;
  d.wait_ns = a.wait_ns;

  static PerDeviceOnce setup;  // the shared-memory opt-in and the occupancy, once per device
  int dev = 0, slots = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = setup.get(dev, [dev](int* n) {
    cudaError_t rr = cudaFuncSetAttribute(attn_decode_kernel<D, TR>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (rr != cudaSuccess) return rr;
    int sms = 0, per = 0;
    rr = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (rr != cudaSuccess) return rr;
    rr = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, attn_decode_kernel<D, TR>, C::THREADS,
                                                       C::SMEM);
    if (rr != cudaSuccess) return rr;
    *n = std::max(1, sms * std::max(per, 1));
    return cudaSuccess;
  }, &slots);
  if (e != cudaSuccess) return e;
  // one persistent CTA per slot; CTAs beyond the step's units run an empty range
  const int32_t grid = std::min(slots, kMaxDecodeCtas);
  attn_decode_kernel<D, TR><<<(unsigned)grid, C::THREADS, C::SMEM, stream>>>(tm, d);
  count_launch();
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // the merge: launched with programmatic stream serialisation, so its launch overlaps the
  // decode kernel's tail (it waits for the decode grid's completion before reading)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((int64_t)R * Hkv), 1, 1);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, attn_decode_merge_kernel<D>, d, grid);
  if (e != cudaSuccess) return e;
  count_launch();
  return cudaGetLastError();
}

}  // namespace

bool attn_decode_stream_supported(int32_t head_dim, int32_t group, int32_t page_size) {
  // Measured on the 64-request decode step (existing KV U[1,1024] at head_dim 256, U[1,16384]
  // at 512): this kernel streams head_dim 256 at 3.78 TB/s against 3.60 for the chunked
  // kernel, but head_dim 512 at 3.1-3.3 TB/s whatever its ring depth or CTAs per SM, against
  // 4.33 for the chunked kernel, which therefore serves head_dim 512.
  if (head_dim != 256) return false;
  if (group < 1 || group > 16) return false;
  if (page_size < 1 || (page_size & (page_size - 1)) != 0) return false;
  // every TMA box starts on a 1024-byte boundary of its stage (the 128-byte swizzle's period)
  return ((page_size < kUnit ? page_size : kUnit) * head_dim * 2) % 1024 == 0;
}

size_t attn_decode_stream_ws_bytes(int32_t num_req, int32_t group, int32_t head_dim) {
  return align16((size_t)(num_req + 1) * 8) + (size_t)kMaxDecodeCtas * 2 * group * 2 * 4 +
         (size_t)kMaxDecodeCtas * 2 * group * head_dim * 4;
}

cudaError_t launch_attn_decode_stream(const AttnArgs& a, int32_t head_dim, cudaStream_t stream) {
  if (a.plan.num_req == 0) return cudaSuccess;
  if (head_dim == 256)
    return a.group <= 4 ? launch_dec<256, true>(a, stream) : launch_dec<256, false>(a, stream);
  return launch_dec<512, false>(a, stream);
}

}  // namespace pg
