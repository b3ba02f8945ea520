// combine.cu -- log-sum-exp merge of the split-K partials of cut heads.
//
// A head the ahead-of-time plan cut into k items ("Tangram: Unlocking
// Non-Uniform KV Cache for Efficient Multi-turn LLM Serving", AOT Load
// Balancing, Fig. 13) has k partials (m_i, l_i, o_i) with m_i the running
// maximum in log2 units, l_i the sum of 2^(s - m_i) and o_i the un-normalised
// weighted value sum. The merged output is
//     M = max_i m_i,   out = sum_i 2^(m_i - M) o_i / sum_i 2^(m_i - M) l_i,
// which equals softmax attention over the head's whole kept set. The merge
// runs in slot order, so the result is deterministic.
#include <math.h>

#include "kvx_internal.h"
#include "ptx.cuh"

namespace kvx {
namespace {

template <int D>
__global__ void __launch_bounds__(KVX_MAX_GQA * 32)
    combine_kernel(const __grid_constant__ CombineParams p) {
  constexpr int DL = D / 32;
  const SplitHead sh = p.heads[blockIdx.x];
  const int qi = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (qi >= p.g) return;
  const int b = sh.bh / p.Hkv, h = sh.bh - b * p.Hkv;
  float M = -INFINITY;
  for (int s = 0; s < sh.count; ++s)
    M = fmaxf(M, p.part_ml[(size_t)(sh.slot_begin + s) * p.g + qi].x);
  float L = 0.f, acc[DL];
#pragma unroll
  for (int i = 0; i < DL; ++i) acc[i] = 0.f;
  for (int s = 0; s < sh.count; ++s) {
    const size_t slot = (size_t)(sh.slot_begin + s);
    const float2 ml = p.part_ml[slot * p.g + qi];
    const float f = ex2(ml.x - M);
    L += f * ml.y;
    const float *po = p.part_o + (slot * p.g + qi) * D;
#pragma unroll
    for (int i = 0; i < DL; ++i) acc[i] += f * po[lane + 32 * i];
  }
  float *out = p.out + ((size_t)b * p.Hq + (size_t)h * p.g + qi) * D;
#pragma unroll
  for (int i = 0; i < DL; ++i) out[lane + 32 * i] = acc[i] / L;
}

}  // namespace

cudaError_t launch_combine(const CombineParams &p, cudaStream_t st) {
  if (p.num_heads <= 0) return cudaSuccess;
  const dim3 grid(p.num_heads), block(p.g * 32);
  if (p.D == 128)
    combine_kernel<128><<<grid, block, 0, st>>>(p);
  else
    combine_kernel<64><<<grid, block, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace kvx
