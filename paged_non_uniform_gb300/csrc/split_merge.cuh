// split_merge.cuh -- log-sum-exp merge of a split head's partials, done
// inside the attention kernels by the block that finishes the head's last
// piece (so no separate combine launch is needed).
//
// A head the ahead-of-time plan cut into k pieces ("Tangram: Unlocking
// Non-Uniform KV Cache for Efficient Multi-turn LLM Serving", AOT Load
// Balancing, Fig. 13) leaves k partials (m_i, l_i, o_i): m_i the running
// maximum of its scores in log2 units, l_i the sum of 2^(s - m_i), o_i the
// un-normalised weighted value sum. Softmax attention over the whole kept set
// is
//     M = max_i m_i,  out = sum_i 2^(m_i - M) o_i / sum_i 2^(m_i - M) l_i.
// The partials are folded in slot order, so the result does not depend on
// which block finishes last.
#pragma once

#include <math.h>

#include "kvx_internal.h"
#include "ptx.cuh"

namespace kvx {

// Called by the NT merging threads of a block (tid in [0, NT)). Each thread
// owns up to V float4 groups of the head's g x D outputs and keeps R = V *
// BATCH (slot, group) loads in flight per L2 round trip: BATCH slots of each
// of its V groups, or, when the outputs need only one group per thread,
// R slots of that group. Partials are folded in slot order with a running
// maximum.
template <int D, int NT>
__device__ __forceinline__ void merge_split(const AttnParams &p, const SplitHead &sh, int tid) {
  constexpr int V = (KVX_MAX_GQA * D / 4 + NT - 1) / NT;
  constexpr int BATCH = V == 1 ? 4 : 2;
  constexpr int R = V * BATCH;
  const int g = p.g, cnt = sh.count, n4 = g * D / 4;
  const bool one = n4 <= NT;      // one float4 group per thread
  const int per = one ? R : BATCH;  // slots per round trip
  const int b = sh.bh / p.Hkv, h = sh.bh - b * p.Hkv;
  const float2 *ml = p.part_ml + (size_t)sh.slot_begin * g;
  const float4 *po = reinterpret_cast<const float4 *>(p.part_o + (size_t)sh.slot_begin * g * D);
  float M[V], L[V];
  float4 O[V];
#pragma unroll
  for (int k = 0; k < V; ++k) {
    M[k] = -INFINITY;
    L[k] = 0.f;
    O[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int s0 = 0; s0 < cnt; s0 += per) {
    float2 mv[R];
    float4 ov[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int k = one ? 0 : r % V, j = one ? r : r / V;
      const int q4 = tid + k * NT;
      if (s0 + j < cnt && q4 < n4) {
        mv[r] = __ldcg(ml + (size_t)(s0 + j) * g + (4 * q4) / D);
        ov[r] = __ldcg(po + (size_t)(s0 + j) * n4 + q4);
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
#pragma unroll
      for (int k = 0; k < V; ++k) {
        const bool mine = one ? (k == 0) : (r % V == k);
        const int j = one ? r : r / V;
        const int q4 = tid + k * NT;
        if (mine && s0 + j < cnt && q4 < n4) {
          const float mn = fmaxf(M[k], mv[r].x);
          const float a = ex2(M[k] - mn), f = ex2(mv[r].x - mn);
          L[k] = L[k] * a + f * mv[r].y;
          O[k].x = O[k].x * a + f * ov[r].x;
          O[k].y = O[k].y * a + f * ov[r].y;
          O[k].z = O[k].z * a + f * ov[r].z;
          O[k].w = O[k].w * a + f * ov[r].w;
          M[k] = mn;
        }
      }
    }
  }
  float4 *out = reinterpret_cast<float4 *>(p.out + ((size_t)b * p.Hq + (size_t)h * g) * D);
#pragma unroll
  for (int k = 0; k < V; ++k) {
    const int q4 = tid + k * NT;
    if (q4 < n4) {
      const float r = 1.f / L[k];
      out[q4] = make_float4(O[k].x * r, O[k].y * r, O[k].z * r, O[k].w * r);
    }
  }
}

}  // namespace kvx
