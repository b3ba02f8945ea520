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

// One merging thread of NT (tid in [0, NT)) owns the float4 groups q4 = tid,
// tid + NT, ... (V of them) of the head's g x D outputs. It issues the loads
// of S = PAIRS / V slots of every group it owns before folding any of them,
// so that a head of up to S pieces costs one L2 round trip. Each group folds
// its slots in slot order with a running maximum. The caller picks V so that
// V * NT float4 groups cover g x D.
template <int D, int NT, int V, int PAIRS>
__device__ __forceinline__ void merge_split(const AttnParams &p, const SplitHead &sh, int tid) {
  static_assert(V >= 1 && V <= 3 && PAIRS >= V, "merge: one to three groups per thread");
  constexpr int S = (PAIRS + V - 1) / V;  // slots per round trip
  const int g = p.g, cnt = sh.count, n4 = g * D / 4;
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
  for (int s0 = 0; s0 < cnt; s0 += S) {
    float2 mv[S][V];
    float4 ov[S][V];
#pragma unroll
    for (int j = 0; j < S; ++j) {
#pragma unroll
      for (int k = 0; k < V; ++k) {
        const int q4 = tid + k * NT;
        if (s0 + j < cnt && q4 < n4) {
          mv[j][k] = __ldcg(ml + (size_t)(s0 + j) * g + (4 * q4) / D);
          ov[j][k] = __ldcg(po + (size_t)(s0 + j) * n4 + q4);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < S; ++j) {
#pragma unroll
      for (int k = 0; k < V; ++k) {
        const int q4 = tid + k * NT;
        if (s0 + j < cnt && q4 < n4) {
          const float mn = fmaxf(M[k], mv[j][k].x);
          const float a = ex2(M[k] - mn), f = ex2(mv[j][k].x - mn);
          L[k] = L[k] * a + f * mv[j][k].y;
          O[k].x = O[k].x * a + f * ov[j][k].x;
          O[k].y = O[k].y * a + f * ov[j][k].y;
          O[k].z = O[k].z * a + f * ov[j][k].z;
          O[k].w = O[k].w * a + f * ov[j][k].w;
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
