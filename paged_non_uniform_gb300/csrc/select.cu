// select.cu -- kept-set selection for sparse long-context decode, and the
// compaction of the kept K/V rows into head-group pages.
//
// "KVDrive" (Fig. 7, Fig. 16) decodes over the top-K critical KV entries of
// every head, with a recent window; "Tangram" (Fig. 8(b)) stores each head's
// kept tokens in its head group's pages. For sequence b and KV head h, with
// Q = the sum of h's g query vectors (the grouped query heads score a token
// by the sum of their dot products):
//     score_t = <k_t, Q>                     for t < L_b - recent,
//     kept    = the min(top, L_b - recent) largest scores (equal scores:
//               lower position first) and [max(0, L_b - recent), L_b),
//               in ascending position order.
//
// Kernels, in stream order:
//   score   streams every candidate key row once (HBM-bound), fp32 dot with Q;
//   topk    one block per head: 4-pass 8-bit radix select of the cut on
//           order-preserving keys, then an ordered compaction (block scans)
//           that writes the kept positions ascending;
//   pack    copies kept row i of each head into token i of its pages.
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>

#include "kvx_internal.h"
#include "ptx.cuh"

namespace kvx {
namespace {

constexpr int kScoreThreads = 256;
constexpr int kScoreTokensPerBlock = 2048;
constexpr int kTopkThreads = 1024;
constexpr int kPackThreads = 256;

// Order-preserving map of an fp32 score to uint32 (larger score, larger key);
// NaN maps to 0, below every number.
__device__ __forceinline__ uint32_t order_key(float f) {
  if (f != f) return 0u;
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct SelectParams {
  const __nv_bfloat16 *keys;  // [B][Hkv][Lmax][D]
  const __nv_bfloat16 *q;     // [B][Hq][D]
  const int32_t *seq_len;     // [B]
  float *scores;              // [B*Hkv][Lmax]
  int32_t *kept_idx;          // [B*Hkv][stride]
  int32_t *kept_count;        // [B*Hkv]
  uint32_t *status;
  int32_t B, Hq, Hkv, D, Lmax, top, recent, stride;
};

template <int D>
__global__ void __launch_bounds__(kScoreThreads) select_score_kernel(const SelectParams p) {
  constexpr int LPT = D / 8;          // lanes per token row (16 bytes each)
  constexpr int TPW = 32 / LPT;       // token rows per warp and step
  constexpr int U = 4;                // steps in flight per lane
  __shared__ float Q[D];
  const int bh = blockIdx.y;
  const int b = bh / p.Hkv, h = bh - b * p.Hkv;
  const int g = p.Hq / p.Hkv;
  const int L = p.seq_len[b];
  const int n = L - p.recent;
  const int t_begin = blockIdx.x * kScoreTokensPerBlock;
  if (t_begin >= n) return;
  for (int d = threadIdx.x; d < D; d += kScoreThreads) {
    float s = 0.f;
    for (int j = 0; j < g; ++j)
      s += __bfloat162float(p.q[((size_t)b * p.Hq + (size_t)h * g + j) * D + d]);
    Q[d] = s;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane / LPT, part = lane % LPT;
  float qv[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) qv[e] = Q[part * 8 + e];
  const uint4 *rows = reinterpret_cast<const uint4 *>(p.keys + (size_t)bh * p.Lmax * D);
  const int t_end = min(n, t_begin + kScoreTokensPerBlock);
  constexpr int WARPS = kScoreThreads / 32;
  for (int t0 = t_begin + warp * TPW * U; t0 < t_end; t0 += WARPS * TPW * U) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int t = t0 + u * TPW + sub;
      if (t < t_end) v[u] = __ldcs(rows + (size_t)t * LPT + part);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int t = t0 + u * TPW + sub;
      const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = unpack_bf16(w[e]);
        s = fmaf(f.x, qv[2 * e], s);
        s = fmaf(f.y, qv[2 * e + 1], s);
      }
#pragma unroll
      for (int sh = LPT / 2; sh > 0; sh >>= 1) s += __shfl_xor_sync(0xffffffffu, s, sh);
      if (part == 0 && t < t_end) p.scores[(size_t)bh * p.Lmax + t] = s;
    }
  }
}

// Exclusive scan over the block of one int per thread; returns the total.
__device__ __forceinline__ int block_scan(int v, int &excl, int *wsum) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int NW = kTopkThreads / 32;
  int x = v;
#pragma unroll
  for (int sh = 1; sh < 32; sh <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, sh);
    if (lane >= sh) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < NW ? wsum[lane] : 0;
#pragma unroll
    for (int sh = 1; sh < 32; sh <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, sh);
      if (lane >= sh) w += y;
    }
    if (lane < NW) wsum[lane] = w;
  }
  __syncthreads();
  excl = (warp ? wsum[warp - 1] : 0) + x - v;
  const int total = wsum[NW - 1];
  __syncthreads();
  return total;
}

__global__ void __launch_bounds__(kTopkThreads) select_topk_kernel(const SelectParams p) {
  __shared__ int hist[256];
  __shared__ int wsum[kTopkThreads / 32];
  __shared__ uint32_t s_prefix;
  __shared__ int s_k;
  const int bh = blockIdx.x;
  const int b = bh / p.Hkv;
  const int L = p.seq_len[b];
  const int n = max(0, L - p.recent);
  const int ksel = min(p.top, n);
  const float *sc = p.scores + (size_t)bh * p.Lmax;
  int32_t *out = p.kept_idx + (size_t)bh * p.stride;
  // --- threshold: the key of the ksel-th largest candidate (radix select)
  uint32_t prefix = 0, mask = 0;
  int k = ksel;
  if (ksel > 0 && ksel < n) {
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      for (int i = threadIdx.x; i < 256; i += kTopkThreads) hist[i] = 0;
      __syncthreads();
      for (int t = threadIdx.x; t < n; t += kTopkThreads) {
        const uint32_t u = order_key(__ldcg(sc + t));
        if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & 255u], 1);
      }
      __syncthreads();
      if (threadIdx.x < 32) {
        // lane l owns digits 255-8l .. 248-8l (descending); find the digit
        // where the count of keys from the top reaches k
        const int lane = threadIdx.x;
        int c[8], sum = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          c[e] = hist[255 - 8 * lane - e];
          sum += c[e];
        }
        int incl = sum;
#pragma unroll
        for (int sh = 1; sh < 32; sh <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, sh);
          if (lane >= sh) incl += y;
        }
        const int before = incl - sum;
        const bool mine = before < k && k <= incl;
        if (mine) {
          int acc = before;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            if (acc + c[e] >= k) {
              s_prefix = (uint32_t)(255 - 8 * lane - e);
              s_k = k - acc;
              break;
            }
            acc += c[e];
          }
        }
      }
      __syncthreads();
      prefix |= s_prefix << shift;
      mask |= 255u << shift;
      k = s_k;
      __syncthreads();
    }
  }
  // prefix = key of the cut; k = how many keys equal to it are kept
  const uint32_t cut = prefix;
  const bool take_all = ksel >= n;
  int written = 0, eq_seen = 0;
  for (int base = 0; base < n; base += kTopkThreads) {
    const int t = base + threadIdx.x;
    int gt = 0, eq = 0;
    if (t < n) {
      if (take_all) {
        gt = 1;
      } else if (ksel > 0) {
        const uint32_t u = order_key(__ldcg(sc + t));
        gt = u > cut;
        eq = u == cut;
      }
    }
    int eq_before;
    const int eq_total = block_scan(eq, eq_before, wsum);
    const int sel = gt || (eq && eq_seen + eq_before < k);
    int pos;
    const int sel_total = block_scan(sel, pos, wsum);
    if (sel) out[written + pos] = t;
    written += sel_total;
    eq_seen += eq_total;
  }
  // recent window, then padding
  for (int t = n + threadIdx.x; t < L; t += kTopkThreads) out[written + (t - n)] = t;
  const int cnt = written + (L - n);
  for (int i = cnt + threadIdx.x; i < p.stride; i += kTopkThreads) out[i] = -1;
  if (threadIdx.x == 0) p.kept_count[bh] = cnt;
}

struct PackParams {
  const uint4 *keys, *values;  // dense [B][Hkv][Lmax][D]
  const int32_t *kept_idx;     // [B*Hkv][stride]
  const int32_t *n;            // plan's kept counts [B*Hkv]
  GroupDesc grp[KVX_MAX_GROUPS];
  int8_t head_grp[KVX_MAX_KV_HEADS];
  int8_t head_row[KVX_MAX_KV_HEADS];
  uint32_t *status;
  int32_t B, Hkv, D, P, Lmax, stride, layout;
};

// One token row per LPT lanes: kept row i of head (b, h) -> token i of its pages.
__global__ void __launch_bounds__(kPackThreads) pack_kept_kernel(const __grid_constant__ PackParams p) {
  const int bh = blockIdx.y;
  const int b = bh / p.Hkv, h = bh - b * p.Hkv;
  const int n = p.n[bh];
  const int LPT = p.D / 8;  // 16-byte pieces per row
  const int rows_per_block = kPackThreads / LPT;
  const int i = blockIdx.x * rows_per_block + threadIdx.x / LPT;
  const int part = threadIdx.x % LPT;
  if (i >= n) return;
  const GroupDesc &gd = p.grp[p.head_grp[h]];
  const int r = p.head_row[h];
  const int t = p.kept_idx[(size_t)bh * p.stride + i];
  const int32_t page = gd.page_table[(size_t)b * gd.stride + i / p.P];
  if (t < 0 || t >= p.Lmax || page < 0 || (int64_t)page >= gd.num_pages) {
    if (part == 0) atomicOr(p.status, t < 0 || t >= p.Lmax ? KVX_DEV_BAD_BLOCK : KVX_DEV_BAD_PAGE);
    return;
  }
  const int slot = i & (p.P - 1);
  const size_t row = p.layout == KVX_LAYOUT_HEAD_MAJOR
                         ? ((size_t)page * gd.size + r) * p.P + slot
                         : ((size_t)page * p.P + slot) * gd.size + r;
  const size_t src = ((size_t)bh * p.Lmax + t) * LPT + part;
  const size_t dst = row * LPT + part;
  reinterpret_cast<uint4 *>(const_cast<void *>(gd.k_pool))[dst] = __ldcs(p.keys + src);
  reinterpret_cast<uint4 *>(const_cast<void *>(gd.v_pool))[dst] = __ldcs(p.values + src);
}

}  // namespace
}  // namespace kvx

using namespace kvx;

extern "C" int kvx_select_workspace_bytes(int32_t B, int32_t Hkv, int32_t Lmax, size_t *bytes) {
  if (!bytes || B < 1 || Hkv < 1 || Lmax < 1) return KVX_EINVAL;
  *bytes = KVX_WS_HEADER_BYTES + sizeof(float) * (size_t)B * Hkv * Lmax;
  return KVX_OK;
}

extern "C" int kvx_select_topk(const void *keys, const void *q, const int32_t *seq_len,
                               int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t Lmax,
                               int32_t top, int32_t recent, int32_t *kept_idx,
                               int32_t *kept_count, void *workspace, size_t workspace_bytes,
                               void *stream) {
  if (!keys || !q || !seq_len || !kept_idx || !kept_count || !workspace) return KVX_EINVAL;
  if (B < 1 || Hkv < 1 || Hq < 1 || Hq % Hkv || Lmax < 1 || top < 0 || recent < 0)
    return KVX_EINVAL;
  if (D != 64 && D != 128) return KVX_EUNSUPPORTED;
  if ((uintptr_t)keys % 16 || (uintptr_t)workspace % 256) return KVX_EINVAL;
  size_t need = 0;
  kvx_select_workspace_bytes(B, Hkv, Lmax, &need);
  if (workspace_bytes < need) return KVX_EINVAL;
  if ((int64_t)top + recent > (int64_t)1 << 30) return KVX_ERANGE;
  SelectParams p;
  p.keys = (const __nv_bfloat16 *)keys;
  p.q = (const __nv_bfloat16 *)q;
  p.seq_len = seq_len;
  p.scores = (float *)((char *)workspace + KVX_WS_HEADER_BYTES);
  p.kept_idx = kept_idx;
  p.kept_count = kept_count;
  p.status = (uint32_t *)workspace;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.D = D;
  p.Lmax = Lmax;
  p.top = top;
  p.recent = recent;
  p.stride = top + recent;
  cudaStream_t st = (cudaStream_t)stream;
  const dim3 sgrid((Lmax + kScoreTokensPerBlock - 1) / kScoreTokensPerBlock, B * Hkv);
  if (D == 128)
    select_score_kernel<128><<<sgrid, kScoreThreads, 0, st>>>(p);
  else
    select_score_kernel<64><<<sgrid, kScoreThreads, 0, st>>>(p);
  select_topk_kernel<<<B * Hkv, kTopkThreads, 0, st>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_cuda_error(e);
  return KVX_OK;
}

extern "C" int kvx_pack_kept(const kvx_plan *plan, const void *keys, const void *values,
                             int32_t Lmax, const int32_t *kept_idx, int32_t kept_stride,
                             void *const *k_pools, void *const *v_pools,
                             const int64_t *pool_pages, const int32_t *const *page_tables,
                             const int32_t *page_table_stride, void *workspace,
                             size_t workspace_bytes, void *stream) {
  if (!plan || !keys || !values || !kept_idx || !k_pools || !v_pools || !pool_pages ||
      !page_tables || !page_table_stride || !workspace)
    return KVX_EINVAL;
  if (!plan->d_buf) return KVX_ESTATE;
  const kvx_shape &s = plan->shape;
  if (s.dtype != KVX_BF16) return KVX_EUNSUPPORTED;
  if (Lmax < 1 || kept_stride < 1 || workspace_bytes < KVX_WS_HEADER_BYTES) return KVX_EINVAL;
  if ((uintptr_t)keys % 16 || (uintptr_t)values % 16) return KVX_EINVAL;
  PackParams p;
  std::memset(&p, 0, sizeof(p));
  int32_t maxn = 0;
  for (int32_t v : plan->n) maxn = std::max(maxn, v);
  if (maxn > kept_stride) return KVX_ERANGE;
  for (int gi = 0; gi < s.num_groups; ++gi) {
    if (!k_pools[gi] || !v_pools[gi] || !page_tables[gi] || pool_pages[gi] < 1) return KVX_EINVAL;
    if ((uintptr_t)k_pools[gi] % 16 || (uintptr_t)v_pools[gi] % 16) return KVX_EINVAL;
    int32_t mx = 0;
    for (int b = 0; b < s.B; ++b) mx = std::max(mx, plan->group_pages[(size_t)gi * s.B + b]);
    if (page_table_stride[gi] < std::max(mx, 1)) return KVX_ERANGE;
    p.grp[gi].page_table = page_tables[gi];
    p.grp[gi].k_pool = k_pools[gi];
    p.grp[gi].v_pool = v_pools[gi];
    p.grp[gi].num_pages = pool_pages[gi];
    p.grp[gi].stride = page_table_stride[gi];
    p.grp[gi].size = plan->group_size[gi];
  }
  for (int h = 0; h < s.Hkv; ++h) {
    p.head_grp[h] = (int8_t)plan->head_group[h];
    p.head_row[h] = (int8_t)plan->head_row[h];
  }
  p.keys = (const uint4 *)keys;
  p.values = (const uint4 *)values;
  p.kept_idx = kept_idx;
  p.n = plan->d_n;
  p.status = (uint32_t *)workspace;
  p.B = s.B;
  p.Hkv = s.Hkv;
  p.D = s.D;
  p.P = s.page_size;
  p.Lmax = Lmax;
  p.stride = kept_stride;
  p.layout = s.layout;
  const int rows_per_block = kPackThreads / (s.D / 8);
  const dim3 grid((maxn + rows_per_block - 1) / rows_per_block, s.B * s.Hkv);
  if (grid.x > 0)
    pack_kept_kernel<<<grid, kPackThreads, 0, (cudaStream_t)stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_cuda_error(e);
  return KVX_OK;
}
