// attn_simt.cu -- split decode attention over head-group pages on the CUDA
// cores (fp32 or bf16 K/V, fp32 arithmetic).
//
// Same work items, partial format and output as the tensor-core kernel
// ("Tangram: Unlocking Non-Uniform KV Cache for Efficient Multi-turn LLM
// Serving", Fig. 8(b) page addressing, Fig. 13 ahead-of-time split). Four
// warps per block. A token row of K (or V) is read with 16-byte vector loads:
// LPT = D * sizeof(T) / 16 lanes cover one row, so one warp step covers
// TPW = 32 / LPT tokens (lane group j of warp w takes tokens
// begin + w*TPW + j, then every kWarps*TPW further). Each lane group reduces
// its g dot products with shuffles inside the group and keeps its own online
// softmax state; the groups of a warp are merged by shuffles, the warps in
// shared memory at the end of each item, and split heads by the block that
// finishes their last piece. Page ids outside the pool read as zero rows and
// set KVX_DEV_BAD_PAGE.
#include <cuda_bf16.h>
#include <math.h>

#include "kvx_internal.h"
#include "ptx.cuh"
#include "split_merge.cuh"

namespace kvx {
namespace {

constexpr int kWarps = 4;

// Sixteen bytes of a row (one vector load) as EPL floats.
template <typename T>
struct Vec16;
template <>
struct Vec16<float> {
  static constexpr int kN = 4;
  __device__ __forceinline__ static void load(const float *src, float (&f)[4]) {
    const float4 v = __ldg(reinterpret_cast<const float4 *>(src));
    f[0] = v.x;
    f[1] = v.y;
    f[2] = v.z;
    f[3] = v.w;
  }
};
template <>
struct Vec16<__nv_bfloat16> {
  static constexpr int kN = 8;
  __device__ __forceinline__ static void load(const __nv_bfloat16 *src, float (&f)[8]) {
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(src));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
};

// Scale of a state with maximum m when the merged maximum is M (a state that
// has seen no token has m = -inf and contributes nothing).
__device__ __forceinline__ float rescale(float m, float M) {
  return m == -INFINITY ? 0.f : ex2(m - M);
}

template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32)
    attn_simt_kernel(const __grid_constant__ AttnParams p) {
  constexpr int EPL = Vec16<T>::kN;  // elements per lane per 16-byte load
  constexpr int LPT = D / EPL;       // lanes per token row
  constexpr int TPW = 32 / LPT;      // tokens per warp step
  constexpr int U = EPL == 4 ? 4 : 2;  // warp steps whose rows are in flight together
  static_assert(LPT >= 1 && LPT <= 32 && 32 % LPT == 0, "a row must tile the warp");
  constexpr int MW = 8 * D + 16;     // floats per warp record
  __shared__ float merge[2][kWarps][MW];
  __shared__ int last_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane / LPT, gl = lane % LPT;  // token of the step, lane within the row
  const int it0 = p.cta_off[blockIdx.x], it1 = p.cta_off[blockIdx.x + 1];
  const int g = p.g, P = p.P;
  uint64_t t_start = p.trace ? globaltimer_ns() : 0;
  pdl_launch_dependents();
  pdl_wait();  // global inputs may come from the previous kernel in the stream
  for (int it = it0; it < it1; ++it) {
    const Item item = p.items[it];
    const int b = item.bh / p.Hkv, h = item.bh - b * p.Hkv;
    const int gi = p.head_grp[h], row = p.head_row[h];
    const GroupDesc &gd = p.grp[gi];
    const int32_t *pt = gd.page_table + (size_t)b * gd.stride;
    const T *kp = (const T *)gd.k_pool;
    const T *vp = (const T *)gd.v_pool;
    if (warp == 0 && lane == 0) {
      const int L = __ldg(p.seq_len + b), bud = __ldg(p.head_budget + item.bh);
      if (min(L, bud) != __ldg(p.n_plan + item.bh)) atomicOr(p.status, KVX_DEV_BAD_BUDGET);
    }
    float qv[KVX_MAX_GQA][EPL], o[KVX_MAX_GQA][EPL], m[KVX_MAX_GQA], l[KVX_MAX_GQA];
    const T *qb = (const T *)p.q + ((size_t)b * p.Hq + (size_t)h * g) * D + gl * EPL;
#pragma unroll
    for (int j = 0; j < KVX_MAX_GQA; ++j) {
      m[j] = -INFINITY;
      l[j] = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) o[j][e] = qv[j][e] = 0.f;
      if (j < g) Vec16<T>::load(qb + (size_t)j * D, qv[j]);
    }
    // U warp steps per batch: their page ids, then all their K and V rows,
    // are loaded before any of them is used, so a short item costs one or two
    // memory round trips instead of two per warp step. Lane group grp still
    // takes tokens begin + warp*TPW + grp + k*kWarps*TPW in increasing k.
    for (int tb = item.begin + warp * TPW; tb < item.end; tb += U * kWarps * TPW) {
      int32_t page[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int t = tb + u * kWarps * TPW + grp;
        page[u] = t < item.end ? __ldg(pt + t / P) : 0;
      }
      float kv[U][EPL], vv[U][EPL];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int t = tb + u * kWarps * TPW + grp;
#pragma unroll
        for (int e = 0; e < EPL; ++e) kv[u][e] = vv[u][e] = 0.f;
        if (t < item.end) {
          if (page[u] < 0 || (int64_t)page[u] >= gd.num_pages) {
            if (gl == 0) atomicOr(p.status, KVX_DEV_BAD_PAGE);
          } else {
            const size_t rr = p.layout == KVX_LAYOUT_HEAD_MAJOR
                                  ? ((size_t)page[u] * gd.size + row) * P + (t & (P - 1))
                                  : ((size_t)page[u] * P + (t & (P - 1))) * gd.size + row;
            Vec16<T>::load(kp + rr * D + gl * EPL, kv[u]);
            Vec16<T>::load(vp + rr * D + gl * EPL, vv[u]);
          }
          // Coverage record (test hook): one count per token fed to the softmax.
          if (p.cover && gl == 0) atomicAdd(p.cover + (size_t)item.bh * p.cover_stride + t, 1);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const bool active = tb + u * kWarps * TPW + grp < item.end;
#pragma unroll
        for (int j = 0; j < KVX_MAX_GQA; ++j) {
          if (j >= g) break;
          float dot = 0.f;
#pragma unroll
          for (int e = 0; e < EPL; ++e) dot = fmaf(qv[j][e], kv[u][e], dot);
#pragma unroll
          for (int sh = LPT / 2; sh > 0; sh >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, sh);
          if (active) {
            const float x = dot * p.scale_log2;
            const float mn = fmaxf(m[j], x);
            const float al = ex2(m[j] - mn), pw = ex2(x - mn);
            l[j] = l[j] * al + pw;
#pragma unroll
            for (int e = 0; e < EPL; ++e) o[j][e] = fmaf(o[j][e], al, pw * vv[u][e]);
            m[j] = mn;
          }
        }
      }
    }
    // merge the lane groups of this warp (lanes gl of every group hold the
    // same dimensions)
#pragma unroll
    for (int sh = LPT; sh < 32; sh <<= 1) {
#pragma unroll
      for (int j = 0; j < KVX_MAX_GQA; ++j) {
        if (j >= g) break;
        const float mo = __shfl_xor_sync(0xffffffffu, m[j], sh);
        const float lo = __shfl_xor_sync(0xffffffffu, l[j], sh);
        const float M = fmaxf(m[j], mo);
        const float a = rescale(m[j], M), c = rescale(mo, M);
        l[j] = l[j] * a + lo * c;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
          const float oo = __shfl_xor_sync(0xffffffffu, o[j][e], sh);
          o[j][e] = o[j][e] * a + oo * c;
        }
        m[j] = M;
      }
    }
    float *buf = &merge[(it - it0) & 1][0][0];
    float *mw = buf + warp * MW;
    if (grp == 0) {
#pragma unroll
      for (int j = 0; j < KVX_MAX_GQA; ++j) {
        if (j >= g) break;
#pragma unroll
        for (int e = 0; e < EPL; ++e) mw[j * D + gl * EPL + e] = o[j][e];
        if (lane == 0) {
          mw[8 * D + j] = m[j];
          mw[8 * D + 8 + j] = l[j];
        }
      }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < g * D; idx += kWarps * 32) {
      const int qi = idx / D, d = idx - qi * D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, buf[w * MW + 8 * D + qi]);
      float Ls = 0.f, O = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float f = rescale(buf[w * MW + 8 * D + qi], M);
        Ls += f * buf[w * MW + 8 * D + 8 + qi];
        O += f * buf[w * MW + qi * D + d];
      }
      if (item.slot < 0) {
        p.out[((size_t)b * p.Hq + (size_t)h * g + qi) * D + d] = O / Ls;
      } else {
        p.part_o[((size_t)item.slot * g + qi) * D + d] = O;
        if (d == 0) p.part_ml[(size_t)item.slot * g + qi] = make_float2(M, Ls);
      }
    }
    if (item.slot >= 0) {
      // publish the piece: the ticket after the barrier releases the block's
      // partial writes and, in the block that counts last, acquires the
      // other pieces' partials for all threads through the second barrier
      __syncthreads();
      if (threadIdx.x == 0)
        last_flag = ticket_acq_rel(p.counters + item.split) == p.split[item.split].count - 1;
      __syncthreads();
      if (last_flag) {
        constexpr int NT = kWarps * 32, VM = (KVX_MAX_GQA * D / 4 + NT - 1) / NT;
        merge_split<D, NT, VM, 4>(p, p.split[item.split], threadIdx.x);
        if (threadIdx.x == 0) p.counters[item.split] = 0;
      }
    }
  }
  if (p.trace) {
    __syncthreads();
    if (threadIdx.x == 0) {
      int64_t tok = 0;
      for (int it = it0; it < it1; ++it) tok += p.items[it].end - p.items[it].begin;
      int64_t *tr = p.trace + 4 * (size_t)blockIdx.x;
      tr[0] = smid();
      tr[1] = (int64_t)t_start;
      tr[2] = (int64_t)globaltimer_ns();
      tr[3] = tok;
    }
  }
}

}  // namespace

cudaError_t launch_attn_simt(const AttnParams &p, int dtype, int num_ctas,
                             cudaStream_t st) {
  if (num_ctas <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_ctas);
  cfg.blockDim = dim3(kWarps * 32);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (dtype == KVX_F32)
    e = p.D == 128 ? cudaLaunchKernelEx(&cfg, attn_simt_kernel<float, 128>, p)
                   : cudaLaunchKernelEx(&cfg, attn_simt_kernel<float, 64>, p);
  else
    e = p.D == 128 ? cudaLaunchKernelEx(&cfg, attn_simt_kernel<__nv_bfloat16, 128>, p)
                   : cudaLaunchKernelEx(&cfg, attn_simt_kernel<__nv_bfloat16, 64>, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace kvx
