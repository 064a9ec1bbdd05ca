// Merge of two attention states over disjoint key sets, for cascade attention (requests
// that share a key prefix attend to it once as a segment and to their own keys as another).
// With w_x = exp(lse_x - M), M = max(lse_a, lse_b):
//   out = (w_a out_a + w_b out_b) / (w_a + w_b),  lse = M + log(w_a + w_b);
// the state (anything, -inf) of a row that saw no key contributes nothing. The softmax over
// the union of the key sets is the two softmaxes reweighted by their normalisers, so the
// merge is exact up to the rounding of the bf16 inputs. Declared in include/pg.h.
#include "pg_internal.h"

#include <math.h>

namespace pg {
namespace {

constexpr int kMergeRowsPerBlock = 8;  // one warp per row

__global__ void __launch_bounds__(32 * kMergeRowsPerBlock)
merge_states_kernel(const __nv_bfloat16* out_a, const float* lse_a, const __nv_bfloat16* out_b,
                    const float* lse_b, __nv_bfloat16* out, float* lse, int32_t rows,
                    int32_t head_dim) {
  // out may alias out_a or out_b (and lse either input): each thread reads its 16 bytes of
  // both inputs before it writes the same 16 bytes of out
  const int32_t row = blockIdx.x * kMergeRowsPerBlock + (int32_t)(threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float la = lse_a[row], lb = lse_b[row];
  const float M = fmaxf(la, lb);
  float wa = 0.f, wb = 0.f, l = -INFINITY;
  if (M != -INFINITY) {
    wa = la == -INFINITY ? 0.f : expf(la - M);
    wb = lb == -INFINITY ? 0.f : expf(lb - M);
    l = M + logf(wa + wb);
    const float inv = 1.f / (wa + wb);
    wa *= inv;
    wb *= inv;
  }
  const int64_t base = (int64_t)row * head_dim;
  for (int c = lane * 8; c < head_dim; c += 32 * 8) {
    const uint4 va = *reinterpret_cast<const uint4*>(out_a + base + c);
    const uint4 vb = *reinterpret_cast<const uint4*>(out_b + base + c);
    const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&va);
    const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&vb);
    uint4 vo;
    __nv_bfloat162* po = reinterpret_cast<__nv_bfloat162*>(&vo);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 fa = __bfloat1622float2(pa[e]), fb = __bfloat1622float2(pb[e]);
      // a side with zero weight contributes nothing, whatever its bits
      const float x = (wa > 0.f ? wa * fa.x : 0.f) + (wb > 0.f ? wb * fb.x : 0.f);
      const float y = (wa > 0.f ? wa * fa.y : 0.f) + (wb > 0.f ? wb * fb.y : 0.f);
      po[e] = __floats2bfloat162_rn(x, y);
    }
    *reinterpret_cast<uint4*>(out + base + c) = vo;
  }
  __syncwarp();  // every lane has read lse_a / lse_b before lane 0 may overwrite them
  if (lse && lane == 0) lse[row] = l;
}

}  // namespace

cudaError_t launch_merge_states(const __nv_bfloat16* out_a, const float* lse_a,
                                const __nv_bfloat16* out_b, const float* lse_b,
                                __nv_bfloat16* out, float* lse, int32_t rows, int32_t head_dim,
                                cudaStream_t stream) {
  const int32_t blocks = (rows + kMergeRowsPerBlock - 1) / kMergeRowsPerBlock;
  merge_states_kernel<<<blocks, 32 * kMergeRowsPerBlock, 0, stream>>>(out_a, lse_a, out_b, lse_b,
                                                                     out, lse, rows, head_dim);
  count_launch();
  return cudaGetLastError();
}

}  // namespace pg
