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
//   score   streams every candidate key row once (HBM-bound), fp32 dot with Q,
//           and counts the first radix digit (top 11 key bits) per head;
//   bucket  many blocks per head: each reads a span of scores once, sets the
//           positions whose first radix digit is above the cut's in a
//           bitmask and appends those in the cut's bucket to a list;
//   topk    one block per head: the other two radix digits (11/11/10 bits
//           on order-preserving keys) over the bucket list in shared
//           memory, then bitmasks of the kept positions and an ordered
//           write, ascending;
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

// The float whose order-preserving key is k (inverse of order_key for keys
// of numbers).
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Length of sequence b, or 0 when it lies outside [0, Lmax] (the top-k
// kernel then reports KVX_DEV_BAD_LENGTH).
#define KVX_SELECT_LEN(p, b) \
  (((p).seq_len[b] >= 0 && (p).seq_len[b] <= (p).Lmax) ? (p).seq_len[b] : 0)

struct SelectParams {
  const __nv_bfloat16 *keys;  // [B][Hkv][Lmax][D]
  const __nv_bfloat16 *q;     // [B][Hq][D]
  const int32_t *seq_len;     // [B]
  float *scores;              // [B*Hkv][Lmax]
  int32_t *hist0;             // [B*Hkv][2048] counts of the top 11 key bits (zeroed per call)
  int32_t *kept_idx;          // [B*Hkv][stride]
  int32_t *kept_count;        // [B*Hkv]
  uint32_t *status;
  uint2 *blist;               // [B*Hkv][kBucketCap] (key, position) of the cut's first-digit bucket
  int32_t *bcnt;              // [B*Hkv] bucket sizes (zeroed per call with hist0)
  uint32_t *bgt;              // [B*Hkv][wstride] bitmask: first digit above the cut's
  int32_t B, Hq, Hkv, D, Lmax, top, recent, stride;
  int32_t ldsc;               // score row stride: Lmax rounded up to a multiple of 4
  int32_t wstride;            // bitmask row stride in words
};

template <int D>
__global__ void __launch_bounds__(kScoreThreads, 3) select_score_kernel(const SelectParams p) {
  constexpr int LPT = D / 8;          // lanes per token row (16 bytes each)
  constexpr int TPW = 32 / LPT;       // token rows per warp and step
  constexpr int U = 8;                // steps in flight per lane
  __shared__ float Q[D];
  __shared__ int hist[2048];
  __shared__ float s_sc[kScoreTokensPerBlock];
  pdl_launch_dependents();  // the bucket pass may launch; it waits for this grid
  const int bh = blockIdx.y;
  const int b = bh / p.Hkv, h = bh - b * p.Hkv;
  const int g = p.Hq / p.Hkv;
  const int L = KVX_SELECT_LEN(p, b);
  const int n = L - p.recent;
  const int t_begin = blockIdx.x * kScoreTokensPerBlock;
  if (t_begin >= n) return;
  for (int d = threadIdx.x; d < D; d += kScoreThreads) {
    float s = 0.f;
    for (int j = 0; j < g; ++j)
      s += __bfloat162float(p.q[((size_t)b * p.Hq + (size_t)h * g + j) * D + d]);
    Q[d] = s;
  }
  for (int i = threadIdx.x; i < 2048; i += kScoreThreads) hist[i] = 0;
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
      if (part == 0 && t < t_end) {
        p.scores[(size_t)bh * p.ldsc + t] = s;
        s_sc[t - t_begin] = s;
      }
    }
  }
  __syncthreads();
  // first radix digit of the selection (top 11 key bits), counted per block
  // with warp-aggregated shared-memory atomics, then added to the head's
  // global histogram
  const int cnt_here = t_end - t_begin;
  for (int i0 = warp * 32; i0 < cnt_here; i0 += kScoreThreads) {
    const int i = i0 + lane;
    const int bin = i < cnt_here ? (int)(order_key(s_sc[i]) >> 21) : -1;
    const unsigned grp = __match_any_sync(0xffffffffu, bin);
    if (bin >= 0 && (__ffs(grp) - 1) == lane) atomicAdd(&hist[bin], __popc(grp));
  }
  __syncthreads();
  int32_t *gh = p.hist0 + (size_t)bh * 2048;
  for (int i = threadIdx.x; i < 2048; i += kScoreThreads)
    if (hist[i]) atomicAdd(gh + i, hist[i]);
}

constexpr int kTopkWarps = kTopkThreads / 32;
static_assert(2048 % kTopkThreads == 0, "top-k: the first-digit histogram splits evenly");
constexpr int kBucketCap = 8192;       // (key, position) pairs kept per head
constexpr int kBucketThreads = 512;
static_assert(2048 % kBucketThreads == 0, "bucket: the first-digit histogram splits evenly");
constexpr int kBucketSpan = 32768;     // positions per bucket block
constexpr int kBucketUC = 4;           // float4 per thread in each of its sub-spans
constexpr int kBlockBucketCap = 4096;  // bucket entries one bucket block stages in shared memory
constexpr int kMaxSelectLmax = 1 << 18;

size_t select_wstride(int Lmax) { return (((size_t)Lmax + 31) / 32 + 3) & ~size_t(3); }

// Dynamic shared memory of the top-k kernel: the bucket list, then the
// above-cut and at-cut bitmasks of all candidate positions.
size_t topk_smem_bytes(int Lmax) {
  return (size_t)kBucketCap * sizeof(uint2) + 2 * select_wstride(Lmax) * sizeof(uint32_t);
}

// Finds, from a histogram of nb bins, the bin (counted from the top) that
// holds the k-th largest key and the rank of that key inside the bin. All NT
// threads of the block call it:
// thread t owns nb / NT consecutive bins from the top, a two-level scan gives
// each thread the count above its bins, and the thread whose bins hold the
// k-th key resolves it. wsum: NT / 32 ints of shared scratch.
template <int NT>
__device__ __forceinline__ void find_digit_block(const int *hist, int nb, int k,
                                                 uint32_t *s_digit, int *s_k, int *wsum) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = nb / NT;
  int sum = 0;
  for (int e = 0; e < per; ++e) sum += hist[nb - 1 - tid * per - e];
  int incl = sum;
#pragma unroll
  for (int sh = 1; sh < 32; sh <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, sh);
    if (lane >= sh) incl += y;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int v = lane < NT / 32 ? wsum[lane] : 0;
    int x = v;
#pragma unroll
    for (int sh = 1; sh < 32; sh <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, sh);
      if (lane >= sh) x += y;
    }
    if (lane < NT / 32) wsum[lane] = x - v;
  }
  __syncthreads();
  const int before = wsum[warp] + incl - sum;
  if (before < k && k <= before + sum) {
    int acc = before;
    for (int e = 0; e < per; ++e) {
      const int c = hist[nb - 1 - tid * per - e];
      if (acc + c >= k) {
        *s_digit = (uint32_t)(nb - 1 - tid * per - e);
        *s_k = k - acc;
        break;
      }
      acc += c;
    }
  }
  __syncthreads();
}

// Cut search shared by both kernels: the candidate count of a head and
// whether a cut has to be found (0 < ksel < n).
struct HeadSel {
  int L, n, ksel;
  bool search;
};
__device__ __forceinline__ HeadSel head_sel(const SelectParams &p, int bh) {
  HeadSel h;
  h.L = KVX_SELECT_LEN(p, bh / p.Hkv);
  h.n = max(0, h.L - p.recent);
  h.ksel = min(p.top, h.n);
  h.search = h.ksel > 0 && h.ksel < h.n;
  return h;
}

// Bucket pass, grid (position spans, heads). Every block finds the cut's
// first digit d0 from the score kernel's histogram, then reads its span of
// scores once (float4 per lane, the next sub-span loading while the current
// one is sorted): positions whose first digit is above d0 go
// into the above-cut bitmask (word j of a warp's 128 positions is collected
// from lanes 8j..8j+7), positions in the bucket d0 are appended to the head's
// (key, position) list: staged in shared memory (one shared atomic per warp)
// and copied out after one global atomic per block (many atomics on one
// global counter would serialise).
__global__ void __launch_bounds__(kBucketThreads, 2) select_bucket_kernel(const SelectParams p) {
  __shared__ int hist[2048];
  __shared__ uint2 sl[kBlockBucketCap];
  __shared__ uint32_t s_digit;
  __shared__ int s_k, s_cnt, s_base;
  __shared__ int wsum[kBucketThreads / 32];
  pdl_launch_dependents();
  pdl_wait();  // scores and histograms of the score pass
  const int bh = blockIdx.y;
  const HeadSel hs = head_sel(p, bh);
  const int t_begin = blockIdx.x * kBucketSpan;
  if (!hs.search || t_begin >= hs.n) return;
  const int tid = threadIdx.x, lane = tid & 31;
  const int n = hs.n, nwords = (n + 31) >> 5;
  const float4 *sc4 = reinterpret_cast<const float4 *>(p.scores + (size_t)bh * p.ldsc);
  uint32_t *gtw = p.bgt + (size_t)bh * p.wstride;
  uint2 *list = p.blist + (size_t)bh * kBucketCap;
  constexpr int SUB4 = kBucketThreads * kBucketUC;  // float4 per sub-span
  constexpr int NSUB = kBucketSpan / 4 / SUB4;
  const int i0 = t_begin / 4, n4 = (n + 3) >> 2;
  // the first sub-span's scores are loaded while the cut's first digit is
  // found; each later sub-span is loaded while the previous one is sorted
  float4 v[kBucketUC];
#pragma unroll
  for (int j = 0; j < kBucketUC; ++j) {
    const int i4 = i0 + j * kBucketThreads + tid;
    v[j] = i4 < n4 ? __ldcg(sc4 + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  {
    // the histogram's loads are all issued before the first store
    constexpr int CH = 2048 / kBucketThreads;
    int hv[CH];
#pragma unroll
    for (int j = 0; j < CH; ++j) hv[j] = __ldcg(p.hist0 + (size_t)bh * 2048 + tid + j * kBucketThreads);
#pragma unroll
    for (int j = 0; j < CH; ++j) hist[tid + j * kBucketThreads] = hv[j];
  }
  if (tid == 0) s_cnt = 0;
  __syncthreads();
  find_digit_block<kBucketThreads>(hist, 2048, hs.ksel, &s_digit, &s_k, wsum);
  const uint32_t d0 = s_digit;
  // Away from NaN, infinities and the two zeros (digits 0..3, 1023, 1024 and
  // 2044 up), the bucket d0 is the float interval [lo, hi) of its keys, so
  // two float compares classify a score; the key is computed only for the
  // few scores in the bucket. Elsewhere every score's key is compared.
  const bool fast = d0 >= 4 && d0 <= 2043 && d0 != 1023 && d0 != 1024;
  const float lo = key_float(d0 << 21), hi = key_float((d0 + 1) << 21);
#pragma unroll 1
  for (int c = 0; c < NSUB; ++c) {
    const int b4 = i0 + c * SUB4;
    if (4 * b4 >= n) break;  // block-uniform
    float4 nx[kBucketUC];
#pragma unroll
    for (int j = 0; j < kBucketUC; ++j) {
      const int i4 = b4 + SUB4 + j * kBucketThreads + tid;
      nx[j] = (c + 1 < NSUB && i4 < n4) ? __ldcg(sc4 + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int j = 0; j < kBucketUC; ++j) {
      const int t = 4 * (b4 + j * kBucketThreads + tid);
      if (t - 4 * lane >= n) break;  // warp-uniform: the warp's 128 positions start past n
      const float f[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
      uint32_t ng = 0, nb = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const bool in = t + e < n;
        bool above, inb;
        if (fast) {
          above = f[e] >= hi;
          inb = f[e] >= lo && !above;
        } else {
          const uint32_t dg = order_key(f[e]) >> 21;
          above = dg > d0;
          inb = dg == d0;
        }
        ng |= (uint32_t)(in && above) << e;
        nb |= (uint32_t)(in && inb) << e;
      }
      uint32_t wg = ng << (4 * (lane & 7));
#pragma unroll
      for (int sh = 1; sh < 8; sh <<= 1) wg |= __shfl_xor_sync(0xffffffffu, wg, sh);
      if ((lane & 7) == 0 && (t >> 5) < nwords) gtw[t >> 5] = wg;
      if (nb) {
        int off = atomicAdd(&s_cnt, __popc(nb));
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if ((nb >> e) & 1u) {
            if (off < kBlockBucketCap) sl[off] = make_uint2(order_key(f[e]), (uint32_t)(t + e));
            ++off;
          }
      }
    }
#pragma unroll
    for (int j = 0; j < kBucketUC; ++j) v[j] = nx[j];
  }
  __syncthreads();
  const int c = s_cnt;
  // a block whose bucket share does not fit marks the whole head as
  // overflowed (its count alone exceeds the list)
  if (tid == 0) s_base = atomicAdd(p.bcnt + bh, c > kBlockBucketCap ? kBucketCap + 1 : c);
  __syncthreads();
  if (c <= kBlockBucketCap)
    for (int i = tid; i < c && s_base + i < kBucketCap; i += kBucketThreads)
      list[s_base + i] = sl[i];
}

// One block per head. The cut (the key of the ksel-th largest candidate) is
// found by a radix select over 11, 11 and 10 bits, MSB first: the first digit
// from the score kernel's histogram, the other two over the bucket list that
// the bucket pass gathered (loaded into shared memory). List entries above
// the cut join the above-cut bitmask, entries equal to it the at-cut
// bitmask; each warp then writes the selected positions of its words in
// ascending order, keys equal to the cut lowest position first. If the bucket
// overflowed the list, the two digits and the bitmasks come from scans of
// the scores in global memory instead.
__global__ void __launch_bounds__(kTopkThreads) select_topk_kernel(const SelectParams p) {
  extern __shared__ __align__(16) uint8_t dsm[];
  uint2 *list = reinterpret_cast<uint2 *>(dsm);
  uint32_t *gtw = reinterpret_cast<uint32_t *>(list + kBucketCap);
  uint32_t *eqw = gtw + p.wstride;
  __shared__ int hist[2048];
  __shared__ int wcnt[2][kTopkWarps];
  __shared__ int wsum[kTopkWarps];
  __shared__ uint32_t s_digit;
  __shared__ int s_k;
  pdl_wait();  // bucket lists and bitmasks of the bucket pass
  const int bh = blockIdx.x;
  const HeadSel hs = head_sel(p, bh);
  const int L = hs.L, n = hs.n, ksel = hs.ksel;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0 && L != p.seq_len[bh / p.Hkv]) atomicOr(p.status, KVX_DEV_BAD_LENGTH);
  const int nwords = (n + 31) >> 5;
  const float *sc = p.scores + (size_t)bh * p.ldsc;
  int32_t *out = p.kept_idx + (size_t)bh * p.stride;
  const bool take_all = ksel >= n;
  // The first chunk of every input (bucket size, above-cut bitmask words,
  // bucket list, histogram) is loaded before any of it is stored, so that
  // the loads share one L2 round trip; list entries past the bucket's size
  // are read (inside the list's capacity) and dropped. Longer inputs finish
  // in plain loops.
  constexpr int CW = 4, CL = 4, CH = 2048 / kTopkThreads;
  const uint32_t *ggt = p.bgt + (size_t)bh * p.wstride;
  const uint2 *glist = p.blist + (size_t)bh * kBucketCap;
  const int32_t *ghist = p.hist0 + (size_t)bh * 2048;
  const int cnt_raw = hs.search ? __ldcg(p.bcnt + bh) : 0;
  uint32_t wv[CW];
  uint2 lv[CL];
  int hv[CH];
#pragma unroll
  for (int j = 0; j < CW; ++j) {
    const int w = tid + j * kTopkThreads;
    wv[j] = hs.search && w < nwords ? __ldcg(ggt + w) : 0u;
  }
#pragma unroll
  for (int j = 0; j < CL; ++j) {
    const int i = tid + j * kTopkThreads;
    lv[j] = hs.search && i < kBucketCap ? __ldcg(glist + i) : make_uint2(0u, 0u);
  }
#pragma unroll
  for (int j = 0; j < CH; ++j) hv[j] = hs.search ? __ldcg(ghist + tid + j * kTopkThreads) : 0;
  const int cnt = hs.search ? min(cnt_raw, kBucketCap + 1) : 0;
  const bool in_smem = cnt <= kBucketCap;
  // bitmasks: above-cut from the bucket pass (or all / none), at-cut empty
  auto word0 = [&](int w, uint32_t loaded) {
    const int rem = n - 32 * w;
    return hs.search ? (in_smem ? loaded : 0u)
                     : (take_all ? (rem >= 32 ? 0xffffffffu : (1u << rem) - 1u) : 0u);
  };
#pragma unroll
  for (int j = 0; j < CW; ++j) {
    const int w = tid + j * kTopkThreads;
    if (w < nwords) {
      gtw[w] = word0(w, wv[j]);
      eqw[w] = 0u;
    }
  }
  for (int w = tid + CW * kTopkThreads; w < nwords; w += kTopkThreads) {
    gtw[w] = word0(w, hs.search && in_smem ? __ldcg(ggt + w) : 0u);
    eqw[w] = 0u;
  }
  if (hs.search) {
    if (in_smem) {
#pragma unroll
      for (int j = 0; j < CL; ++j) {
        const int i = tid + j * kTopkThreads;
        if (i < cnt) list[i] = lv[j];
      }
      for (int i = tid + CL * kTopkThreads; i < cnt; i += kTopkThreads) list[i] = __ldcg(glist + i);
    }
#pragma unroll
    for (int j = 0; j < CH; ++j) hist[tid + j * kTopkThreads] = hv[j];
  }
  __syncthreads();
  uint32_t prefix = 0;
  int k = ksel;
  if (hs.search) {
    find_digit_block<kTopkThreads>(hist, 2048, k, &s_digit, &s_k, wsum);
    prefix = s_digit << 21;
    uint32_t mask = 0x7FFu << 21;
    k = s_k;
    __syncthreads();
    for (int pass = 1; pass < 3; ++pass) {
      const int bits = pass == 1 ? 11 : 10;
      const int shift = pass == 1 ? 10 : 0;
      const int nbins = 1 << bits;
      for (int i = tid; i < nbins; i += kTopkThreads) hist[i] = 0;
      __syncthreads();
      if (in_smem) {
        for (int i = tid; i < cnt; i += kTopkThreads) {
          const uint32_t uu = list[i].x;
          if ((uu & mask) == prefix) atomicAdd(&hist[(uu >> shift) & (uint32_t)(nbins - 1)], 1);
        }
      } else {
        for (int tt = tid; tt < n; tt += kTopkThreads) {
          const uint32_t uu = order_key(__ldcg(sc + tt));
          if ((uu & mask) == prefix) atomicAdd(&hist[(uu >> shift) & (uint32_t)(nbins - 1)], 1);
        }
      }
      __syncthreads();
      find_digit_block<kTopkThreads>(hist, nbins, k, &s_digit, &s_k, wsum);
      prefix |= s_digit << shift;
      mask |= (uint32_t)(nbins - 1) << shift;
      k = s_k;
      __syncthreads();
    }
    const uint32_t cut = prefix;
    if (in_smem) {
      for (int i = tid; i < cnt; i += kTopkThreads) {
        const uint2 e = list[i];
        if (e.x > cut) atomicOr(&gtw[e.y >> 5], 1u << (e.y & 31));
        else if (e.x == cut) atomicOr(&eqw[e.y >> 5], 1u << (e.y & 31));
      }
    } else {
      for (int w = warp; w < nwords; w += kTopkWarps) {
        const int tt = 32 * w + lane;
        const uint32_t uu = tt < n ? order_key(__ldcg(sc + tt)) : 0u;
        const unsigned bg = __ballot_sync(0xffffffffu, tt < n && uu > cut);
        const unsigned be = __ballot_sync(0xffffffffu, tt < n && uu == cut);
        if (lane == 0) {
          gtw[w] = bg;
          eqw[w] = be;
        }
      }
    }
    __syncthreads();
  }
  // k = how many keys equal to the cut are kept. Warp w owns words
  // [w*segw, (w+1)*segw).
  const int segw = (nwords + kTopkWarps - 1) / kTopkWarps;
  const int w_lo = min(nwords, warp * segw), w_hi = min(nwords, w_lo + segw);
  int cg = 0, ce = 0;
  for (int w = w_lo + lane; w < w_hi; w += 32) {
    cg += __popc(gtw[w]);
    ce += __popc(eqw[w]);
  }
#pragma unroll
  for (int sh = 16; sh > 0; sh >>= 1) {
    cg += __shfl_xor_sync(0xffffffffu, cg, sh);
    ce += __shfl_xor_sync(0xffffffffu, ce, sh);
  }
  if (lane == 0) {
    wcnt[0][warp] = cg;
    wcnt[1][warp] = ce;
  }
  __syncthreads();
  int selp = 0, eqp = 0, total = 0, eqtot = 0;
  for (int w = 0; w < kTopkWarps; ++w) {
    if (w < warp) {
      selp += wcnt[0][w] + max(0, min(wcnt[1][w], k - eqp));
      eqp += wcnt[1][w];
    }
    total += wcnt[0][w];
    eqtot += wcnt[1][w];
  }
  const int written = total + min(eqtot, k);
  // ascending write of the warp's words: one word per lane and step
  int wpos = selp, erank = eqp;
  for (int w0 = w_lo; w0 < w_hi; w0 += 32) {
    const int w = w0 + lane;
    const uint32_t g = w < w_hi ? gtw[w] : 0u;
    uint32_t e = w < w_hi ? eqw[w] : 0u;
    const int ne = __popc(e);
    int ie = ne;
#pragma unroll
    for (int sh = 1; sh < 32; sh <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, ie, sh);
      if (lane >= sh) ie += y;
    }
    // keep the first max(0, k - rank) equal keys of this word
    int take = min(ne, max(0, k - (erank + ie - ne)));
    uint32_t et = 0;
    while (take-- > 0) {
      const uint32_t low = e & (0u - e);
      et |= low;
      e ^= low;
    }
    uint32_t sel = g | et;
    const int ns = __popc(sel);
    int is = ns;
#pragma unroll
    for (int sh = 1; sh < 32; sh <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, is, sh);
      if (lane >= sh) is += y;
    }
    int o = wpos + is - ns;
    while (sel) {
      const int bit = __ffs(sel) - 1;
      if (o < p.stride) out[o] = w * 32 + bit;
      ++o;
      sel &= sel - 1;
    }
    wpos += __shfl_sync(0xffffffffu, is, 31);
    erank += __shfl_sync(0xffffffffu, ie, 31);
  }
  // recent window, then padding
  for (int t = n + tid; t < L; t += kTopkThreads)
    if (written + (t - n) < p.stride) out[written + (t - n)] = t;
  const int cntk = written + (L - n);
  for (int i = cntk + tid; i < p.stride; i += kTopkThreads) out[i] = -1;
  if (tid == 0) p.kept_count[bh] = cntk;
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

// Kept row i of head (b, h) -> token i of its pages. LPT lanes move one row
// (16 bytes each of K and V); a thread group handles kPackRows rows spaced
// rows_per_block apart, with every load issued before the stores.
constexpr int kPackRows = 4;
__global__ void __launch_bounds__(kPackThreads) pack_kept_kernel(const __grid_constant__ PackParams p) {
  const int bh = blockIdx.y;
  const int b = bh / p.Hkv, h = bh - b * p.Hkv;
  const int n = p.n[bh];
  const int LPT = p.D / 8;  // 16-byte pieces per row
  const int rows_per_block = kPackThreads / LPT;
  const int i0 = blockIdx.x * rows_per_block * kPackRows + threadIdx.x / LPT;
  const int part = threadIdx.x % LPT;
  if (i0 >= n) return;
  const GroupDesc &gd = p.grp[p.head_grp[h]];
  const int r = p.head_row[h];
  int t[kPackRows];
  int32_t page[kPackRows];
#pragma unroll
  for (int j = 0; j < kPackRows; ++j) {
    const int i = i0 + j * rows_per_block;
    t[j] = i < n ? p.kept_idx[(size_t)bh * p.stride + i] : -1;
    page[j] = i < n ? gd.page_table[(size_t)b * gd.stride + i / p.P] : -1;
  }
  uint4 kv[kPackRows][2];
  bool ok[kPackRows];
#pragma unroll
  for (int j = 0; j < kPackRows; ++j) {
    const int i = i0 + j * rows_per_block;
    ok[j] = i < n && t[j] >= 0 && t[j] < p.Lmax && page[j] >= 0 &&
            (int64_t)page[j] < gd.num_pages;
    if (i < n && !ok[j] && part == 0)
      atomicOr(p.status, t[j] < 0 || t[j] >= p.Lmax ? KVX_DEV_BAD_BLOCK : KVX_DEV_BAD_PAGE);
    if (ok[j]) {
      const size_t src = ((size_t)bh * p.Lmax + t[j]) * LPT + part;
      kv[j][0] = __ldcs(p.keys + src);
      kv[j][1] = __ldcs(p.values + src);
    }
  }
#pragma unroll
  for (int j = 0; j < kPackRows; ++j) {
    if (!ok[j]) continue;
    const int i = i0 + j * rows_per_block;
    const int slot = i & (p.P - 1);
    const size_t row = p.layout == KVX_LAYOUT_HEAD_MAJOR
                           ? ((size_t)page[j] * gd.size + r) * p.P + slot
                           : ((size_t)page[j] * p.P + slot) * gd.size + r;
    const size_t dst = row * LPT + part;
    reinterpret_cast<uint4 *>(const_cast<void *>(gd.k_pool))[dst] = kv[j][0];
    reinterpret_cast<uint4 *>(const_cast<void *>(gd.v_pool))[dst] = kv[j][1];
  }
}

}  // namespace
}  // namespace kvx

using namespace kvx;

// Workspace: header | hist0 int32 [BH][2048] | bcnt int32 [BH] | scores f32
// [BH][ldsc] | blist uint2 [BH][kBucketCap] | bgt uint32 [BH][wstride], each
// section 256-byte aligned; hist0 and bcnt are cleared by one memset per call.
struct SelectWs {
  size_t hist0, bcnt, scores, blist, bgt, total;
};
SelectWs select_ws_offsets(size_t BH, size_t ldsc, size_t wstride) {
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  SelectWs w;
  w.hist0 = KVX_WS_HEADER_BYTES;
  w.bcnt = w.hist0 + sizeof(int32_t) * 2048 * BH;
  w.scores = al(w.bcnt + sizeof(int32_t) * BH);
  w.blist = al(w.scores + sizeof(float) * BH * ldsc);
  w.bgt = al(w.blist + sizeof(uint2) * BH * kBucketCap);
  w.total = al(w.bgt + sizeof(uint32_t) * BH * wstride);
  return w;
}

extern "C" int kvx_select_workspace_bytes(int32_t B, int32_t Hkv, int32_t Lmax, size_t *bytes) {
  if (!bytes || B < 1 || Hkv < 1 || Lmax < 1) return KVX_EINVAL;
  const size_t BH = (size_t)B * Hkv, ldsc = ((size_t)Lmax + 3) & ~size_t(3);
  *bytes = select_ws_offsets(BH, ldsc, select_wstride(Lmax)).total;
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
  if (Lmax > kMaxSelectLmax) return KVX_EUNSUPPORTED;
  SelectParams p;
  p.keys = (const __nv_bfloat16 *)keys;
  p.q = (const __nv_bfloat16 *)q;
  p.seq_len = seq_len;
  const size_t BH = (size_t)B * Hkv;
  const SelectWs wl = select_ws_offsets(BH, ((size_t)Lmax + 3) & ~size_t(3), select_wstride(Lmax));
  char *ws = (char *)workspace;
  p.hist0 = (int32_t *)(ws + wl.hist0);
  p.bcnt = (int32_t *)(ws + wl.bcnt);
  p.scores = (float *)(ws + wl.scores);
  p.blist = (uint2 *)(ws + wl.blist);
  p.bgt = (uint32_t *)(ws + wl.bgt);
  p.wstride = (int32_t)select_wstride(Lmax);
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
  p.ldsc = (Lmax + 3) & ~3;
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e0 = cudaMemsetAsync(p.hist0, 0, wl.scores - wl.hist0, st);
  if (e0 != cudaSuccess) return set_cuda_error(e0);
  const dim3 sgrid((Lmax + kScoreTokensPerBlock - 1) / kScoreTokensPerBlock, B * Hkv);
  if (D == 128)
    select_score_kernel<128><<<sgrid, kScoreThreads, 0, st>>>(p);
  else
    select_score_kernel<64><<<sgrid, kScoreThreads, 0, st>>>(p);
  {
    static int configured[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !configured[dev]) {
      cudaError_t ea = cudaFuncSetAttribute(select_topk_kernel,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            (int)topk_smem_bytes(kMaxSelectLmax));
      if (ea != cudaSuccess) return set_cuda_error(ea);
      configured[dev] = 1;
    }
  }
  // The bucket and top-k passes are launched as programmatic dependents: each
  // starts while the grid before it drains and waits on the device for it.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3((Lmax + kBucketSpan - 1) / kBucketSpan, B * Hkv);
  cfg.blockDim = dim3(kBucketThreads);
  cudaError_t e = cudaLaunchKernelEx(&cfg, select_bucket_kernel, p);
  if (e != cudaSuccess) return set_cuda_error(e);
  cfg.gridDim = dim3(B * Hkv);
  cfg.blockDim = dim3(kTopkThreads);
  cfg.dynamicSmemBytes = topk_smem_bytes(Lmax);
  e = cudaLaunchKernelEx(&cfg, select_topk_kernel, p);
  if (e != cudaSuccess) return set_cuda_error(e);
  e = cudaGetLastError();
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
  const int rows_per_block = kPackThreads / (s.D / 8) * kPackRows;
  const dim3 grid((maxn + rows_per_block - 1) / rows_per_block, s.B * s.Hkv);
  if (grid.x > 0)
    pack_kept_kernel<<<grid, kPackThreads, 0, (cudaStream_t)stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_cuda_error(e);
  return KVX_OK;
}
