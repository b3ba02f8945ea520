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
//   topk    one block per head: radix select (11/11/10 bits) of the cut on
//           order-preserving keys -- first digit from the score kernel, the
//           rest over the cut's bucket, gathered into shared memory while the
//           scores stream through once -- then bitmasks of the kept
//           positions and an ordered write, ascending;
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
  int32_t B, Hq, Hkv, D, Lmax, top, recent, stride;
  int32_t ldsc;               // score row stride: Lmax rounded up to a multiple of 4
};

template <int D>
__global__ void __launch_bounds__(kScoreThreads) select_score_kernel(const SelectParams p) {
  constexpr int LPT = D / 8;          // lanes per token row (16 bytes each)
  constexpr int TPW = 32 / LPT;       // token rows per warp and step
  constexpr int U = 4;                // steps in flight per lane
  __shared__ float Q[D];
  __shared__ int hist[2048];
  __shared__ float s_sc[kScoreTokensPerBlock];
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

// Plain bulk copy global -> shared (addresses 16-byte aligned, bytes a
// multiple of 16), completing on `bar` with a transaction count of `bytes`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, "
      "[%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kBucketCap = 8192;           // keys of the cut's first-digit bucket
constexpr int kStageFloats = 4 * kTopkThreads;  // scores per streamed chunk (one float4 a thread)
constexpr int kStages = 4;
constexpr int kMaxSelectLmax = 1 << 18;
constexpr uint64_t kSelectWaitNs = 2000000000ull;

// Dynamic shared memory of the top-k kernel: the score chunk ring, the bucket
// list, then the above-cut and at-cut bitmasks of all candidate positions.
size_t topk_smem_bytes(int Lmax) {
  const size_t words = ((size_t)Lmax + 31) / 32;
  return (size_t)kStages * kStageFloats * sizeof(float) + (size_t)kBucketCap * sizeof(uint2) +
         2 * words * sizeof(uint32_t);
}

// Finds, from a histogram of nb bins, the bin (counted from the top) that
// holds the k-th largest key and the rank of that key inside the bin. Run by
// warp 0; lane l owns bins nb-1-l*per .. nb-per-l*per.
__device__ __forceinline__ void find_digit(const int *hist, int nb, int k, uint32_t *s_digit,
                                           int *s_k) {
  const int lane = threadIdx.x & 31, per = nb / 32;
  int sum = 0;
  for (int e = 0; e < per; ++e) sum += hist[nb - 1 - lane * per - e];
  int incl = sum;
#pragma unroll
  for (int sh = 1; sh < 32; sh <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, sh);
    if (lane >= sh) incl += y;
  }
  const int before = incl - sum;
  if (before < k && k <= incl) {
    int acc = before;
    for (int e = 0; e < per; ++e) {
      const int c = hist[nb - 1 - lane * per - e];
      if (acc + c >= k) {
        *s_digit = (uint32_t)(nb - 1 - lane * per - e);
        *s_k = k - acc;
        break;
      }
      acc += c;
    }
  }
}

// Issues the bulk copy of score chunk c (positions [c*kStageFloats, ...) of
// the n candidates, rounded up to whole float4s) into its ring slot.
__device__ __forceinline__ void issue_chunk(const float *sc, int n, int c, float *ring,
                                            uint64_t *bars) {
  const int t0 = c * kStageFloats;
  const int len = min(kStageFloats, n - t0);
  const uint32_t bytes = (uint32_t)((len + 3) & ~3) * 4u;
  const int slot = c % kStages;
  const uint32_t bar = smem_u32(&bars[slot]);
  mbar_arrive_expect_tx(bar, bytes);
  bulk_load(smem_u32(ring + (size_t)slot * kStageFloats), sc + t0, bytes, bar);
}

// One block per head. The cut (the key of the ksel-th largest candidate) is
// found by a radix select over 11, 11 and 10 bits, MSB first; the first
// digit's histogram comes from the score kernel.
//   stream  the head's scores pass once through a ring of shared-memory
//           chunks (bulk copies); each position whose first digit is above
//           the cut's goes into the above-cut bitmask, each one in the cut's
//           bucket into a (key, position) list;
//   cut     the other two digits are selected over the list;
//   mark    list entries above the cut join the above-cut bitmask, entries
//           equal to it the at-cut bitmask;
//   write   each warp writes the selected positions of its words in
//           ascending order, keys equal to the cut lowest position first.
// If the bucket overflows the list, the two digits and the bitmasks are
// computed by scans of the scores in global memory instead.
__global__ void __launch_bounds__(kTopkThreads) select_topk_kernel(const SelectParams p) {
  extern __shared__ __align__(128) uint8_t dsm[];
  float *ring = reinterpret_cast<float *>(dsm);
  uint2 *list = reinterpret_cast<uint2 *>(ring + kStages * kStageFloats);
  uint32_t *gtw = reinterpret_cast<uint32_t *>(list + kBucketCap);
  uint32_t *eqw = gtw + ((p.Lmax + 31) >> 5);
  __shared__ int hist[2048];
  __shared__ int wcnt[2][kTopkWarps];
  __shared__ __align__(8) uint64_t bars[kStages];
  __shared__ uint32_t s_digit;
  __shared__ int s_k, s_cnt, s_abort;
  const int bh = blockIdx.x;
  const int b = bh / p.Hkv;
  const int L = KVX_SELECT_LEN(p, b);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0 && L != p.seq_len[b]) atomicOr(p.status, KVX_DEV_BAD_LENGTH);
  const int n = max(0, L - p.recent);
  const int ksel = min(p.top, n);
  const int nwords = (n + 31) >> 5;
  const float *sc = p.scores + (size_t)bh * p.ldsc;
  int32_t *out = p.kept_idx + (size_t)bh * p.stride;
  const bool take_all = ksel >= n, none = ksel == 0;
  const bool search = !take_all && !none;
  const int nch = (n + kStageFloats - 1) / kStageFloats;
  if (tid == 0) {
    s_cnt = 0;
    s_abort = 0;
    for (int i = 0; i < kStages; ++i) mbar_init(smem_u32(&bars[i]), 1);
    fence_barrier_init();
  }
  // above-cut words start as "all candidates" or "none"; at-cut words empty
  for (int w = tid; w < nwords; w += kTopkThreads) {
    const int rem = n - 32 * w;
    gtw[w] = take_all ? (rem >= 32 ? 0xffffffffu : (1u << rem) - 1u) : 0u;
    eqw[w] = 0u;
  }
  if (search)
    for (int i = tid; i < 2048; i += kTopkThreads) hist[i] = p.hist0[(size_t)bh * 2048 + i];
  __syncthreads();
  uint32_t prefix = 0;
  int k = ksel;
  if (search) {
    if (tid == 0)
      for (int c = 0; c < min(kStages, nch); ++c) issue_chunk(sc, n, c, ring, bars);
    if (warp == 0) find_digit(hist, 2048, k, &s_digit, &s_k);
    __syncthreads();
    const uint32_t d0 = s_digit;
    prefix = d0 << 21;
    uint32_t mask = 0x7FFu << 21;
    k = s_k;
    // stream: one float4 of each chunk per thread
    int c_stop = nch;
    for (int c = 0; c < nch; ++c) {
      const int slot = c % kStages;
      if (!mbar_wait(smem_u32(&bars[slot]), (uint32_t)(c / kStages) & 1u, kSelectWaitNs))
        s_abort = 1;
      const int t = c * kStageFloats + 4 * tid;
      const float4 v = reinterpret_cast<const float4 *>(ring + (size_t)slot * kStageFloats)[tid];
      const float f[4] = {v.x, v.y, v.z, v.w};
      uint32_t ng = 0, nb = 0;
      uint32_t u[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        u[e] = order_key(f[e]);
        const bool in = t + e < n;
        ng |= (uint32_t)(in && (u[e] >> 21) > d0) << e;
        nb |= (uint32_t)(in && (u[e] >> 21) == d0) << e;
      }
      // above-cut bits: lanes 8j..8j+7 hold word j of the warp's 128 positions
      uint32_t wg = ng << (4 * (lane & 7));
#pragma unroll
      for (int sh = 1; sh < 8; sh <<= 1) wg |= __shfl_xor_sync(0xffffffffu, wg, sh);
      const int w = (t >> 5);
      if ((lane & 7) == 0 && w < nwords) gtw[w] = wg;
      // bucket entries: one shared atomic per warp
      if (__any_sync(0xffffffffu, nb != 0)) {
        const int cntl = __popc(nb);
        int incl = cntl;
#pragma unroll
        for (int sh = 1; sh < 32; sh <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, sh);
          if (lane >= sh) incl += y;
        }
        int base = 0;
        if (lane == 31) base = atomicAdd(&s_cnt, incl);
        int off = __shfl_sync(0xffffffffu, base, 31) + incl - cntl;
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if ((nb >> e) & 1u) {
            if (off < kBucketCap) list[off] = make_uint2(u[e], (uint32_t)(t + e));
            ++off;
          }
      }
      __syncthreads();
      if (s_abort) {
        c_stop = c;
        break;
      }
      if (tid == 0 && c + kStages < nch) issue_chunk(sc, n, c + kStages, ring, bars);
    }
    if (s_abort) {
      // let copies still in flight land before the block exits: chunks up
      // to c_stop + kStages - 1 were issued
      if (tid == 0) {
        const int last = min(nch, c_stop + kStages) - 1;
        for (int c = max(c_stop, last - kStages + 1); c <= last; ++c)
          mbar_wait(smem_u32(&bars[c % kStages]), (uint32_t)(c / kStages) & 1u, kSelectWaitNs);
        atomicOr(p.status, KVX_DEV_TIMEOUT);
        p.kept_count[bh] = 0;
      }
      for (int i = tid; i < p.stride; i += kTopkThreads) out[i] = -1;
      return;
    }
    const int cnt = s_cnt;
    const bool in_smem = cnt <= kBucketCap;
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
      if (warp == 0) find_digit(hist, nbins, k, &s_digit, &s_k);
      __syncthreads();
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
  const size_t ldsc = ((size_t)Lmax + 3) & ~size_t(3);
  *bytes = KVX_WS_HEADER_BYTES + sizeof(int32_t) * 2048 * (size_t)B * Hkv +
           sizeof(float) * (size_t)B * Hkv * ldsc;
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
  p.hist0 = (int32_t *)((char *)workspace + KVX_WS_HEADER_BYTES);
  p.scores = (float *)((char *)workspace + KVX_WS_HEADER_BYTES +
                       sizeof(int32_t) * 2048 * (size_t)B * Hkv);
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
  cudaError_t e0 = cudaMemsetAsync(p.hist0, 0, sizeof(int32_t) * 2048 * (size_t)B * Hkv, st);
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
  select_topk_kernel<<<B * Hkv, kTopkThreads, topk_smem_bytes(Lmax), st>>>(p);
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
