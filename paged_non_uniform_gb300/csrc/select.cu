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
//   cut     one thread-block cluster per head (this GPU only): every block
//           reads its span of the head's scores once, sets the positions
//           whose first digit is above the cut's in a bitmask and keeps
//           those in the cut's bucket in its shared memory; the leader block
//           finds the other two radix digits (11/11/10 bits on
//           order-preserving keys) over the blocks' buckets through
//           distributed shared memory; every block then marks its positions
//           against the cut and writes its kept positions, ascending, at an
//           offset counted over the cluster;
//   pack    copies kept row i of each head into token i of its pages.
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>

#include "kvx_internal.h"
#include "ptx.cuh"

namespace kvx {
namespace {

constexpr int kScoreThreads = 256;
constexpr int kScoreTokensPerBlock = 1024;  // a multiple of 8: groups stay in one block
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
  float *scores;              // [B*Hkv][ldsc]
  int32_t *hist0;             // [B*Hkv][2048] counts of the top 11 key bits (zeroed per call)
  uint16_t *gmax;             // [B*Hkv][ldg] top 11 key bits of the largest score of 8 positions
  int32_t *kept_idx;          // [B*Hkv][stride]
  int32_t *kept_count;        // [B*Hkv]
  uint32_t *status;
  int32_t B, Hq, Hkv, D, Lmax, top, recent, stride;
  int32_t ldsc;               // score row stride: Lmax rounded up to a multiple of 8
  int32_t ldg;                // group row stride: Lmax / 8 rounded up to a multiple of 8
};

// Clears the first-digit histograms. Launched as a programmatic dependent of
// whatever precedes the call: it waits for that work to complete (the cut pass
// of an earlier call may still read the histograms and scores) before it
// writes or lets the score pass start, which then runs as its dependent.
constexpr int kZeroThreads = 256;
__global__ void __launch_bounds__(kZeroThreads) select_zero_kernel(int4 *h, int n4) {
  pdl_wait();
  pdl_launch_dependents();
  const int i = blockIdx.x * kZeroThreads + threadIdx.x;
  if (i < n4) h[i] = make_int4(0, 0, 0, 0);
}

// Score pass: block (x, bh) takes candidates [x * kScoreTokensPerBlock, ...)
// of head bh. It issues the loads of each warp's first step of key rows, sums
// the g query vectors meanwhile, then streams the rest (LPT lanes per row, U
// rows in flight per lane) and writes the fp32 scores. After a step's scores,
// once the next step's loads are issued, a warp counts their first radix
// digit (top 11 key bits) in shared memory and writes, for each group of 8
// positions, the first digit of the group's largest score, so that the cut
// pass can skip groups below its bucket without reading their scores. At the
// end the block adds its counts to the head's histogram.
template <int D>
__global__ void __launch_bounds__(kScoreThreads, 3) select_score_kernel(const SelectParams p) {
  constexpr int LPT = D / 8;          // lanes per token row (16 bytes each)
  constexpr int TPW = 32 / LPT;       // token rows per warp and step
  constexpr int U = 8;                // steps in flight per lane
  static_assert((U * TPW) % 8 == 0, "score: a warp step covers whole groups of 8 positions");
  __shared__ float Q[D];
  __shared__ int hist[2048];
  pdl_launch_dependents();  // the cut pass may launch; it waits for this grid
  const int bh = blockIdx.y;
  const int b = bh / p.Hkv, h = bh - b * p.Hkv;
  const int g = p.Hq / p.Hkv;
  const int L = KVX_SELECT_LEN(p, b);
  const int n = L - p.recent;
  const int t_begin = blockIdx.x * kScoreTokensPerBlock;
  if (t_begin >= n) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane / LPT, part = lane % LPT;
  const uint4 *rows = reinterpret_cast<const uint4 *>(p.keys + (size_t)bh * p.Lmax * D);
  const int t_end = min(n, t_begin + kScoreTokensPerBlock);
  constexpr int WARPS = kScoreThreads / 32;
  constexpr int STEP = WARPS * TPW * U;
  // the rows of this warp's first step: their loads are in flight while Q is
  // summed and the counts are cleared
  auto issue = [&](uint4 (&v)[U], int t0) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int t = t0 + u * TPW + sub;
      if (t < t_end) v[u] = __ldcs(rows + (size_t)t * LPT + part);
    }
  };
  uint4 v[U];
  const int t_first = t_begin + warp * TPW * U;
  issue(v, t_first);
  for (int d = threadIdx.x; d < D; d += kScoreThreads) {
    float s = 0.f;
    for (int j = 0; j < g; ++j)
      s += __bfloat162float(p.q[((size_t)b * p.Hq + (size_t)h * g + j) * D + d]);
    Q[d] = s;
  }
  for (int i = threadIdx.x; i < 2048; i += kScoreThreads) hist[i] = 0;
  __syncthreads();
  float qv[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) qv[e] = Q[part * 8 + e];
  uint16_t *gm = p.gmax + (size_t)bh * p.ldg;
  for (int t0 = t_first; t0 < t_end; t0 += STEP) {
    float sv[U];
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
      sv[u] = s;
      if (part == 0 && t < t_end) p.scores[(size_t)bh * p.ldsc + t] = s;
    }
    if (t0 + STEP < t_end) issue(v, t0 + STEP);
    // while those loads are in flight: the step's first digits, and the
    // largest digit of its groups of 8 positions
    constexpr int NG = U * TPW / 8;  // groups of 8 positions in a warp step
    int gmx[NG];
#pragma unroll
    for (int q = 0; q < NG; ++q) gmx[q] = -1;
    if (part == 0) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int t = t0 + u * TPW + sub;
        if (t < t_end) {
          const int bin = (int)(order_key(sv[u]) >> 21);
          atomicAdd(&hist[bin], 1);
          gmx[(u * TPW) / 8] = max(gmx[(u * TPW) / 8], bin);
        }
      }
    }
#pragma unroll
    for (int q = 0; q < NG; ++q) {
#pragma unroll
      for (int sh = LPT; sh < 32; sh <<= 1) gmx[q] = max(gmx[q], __shfl_xor_sync(0xffffffffu, gmx[q], sh));
      if (lane == 0 && t0 + 8 * q < t_end) gm[(t0 + 8 * q) >> 3] = (uint16_t)gmx[q];
    }
  }
  __syncthreads();
  pdl_wait();  // the histograms have been zeroed
  int32_t *gh = p.hist0 + (size_t)bh * 2048;
  for (int i = threadIdx.x; i < 2048; i += kScoreThreads)
    if (hist[i]) atomicAdd(gh + i, hist[i]);
}

constexpr int kMaxSelectLmax = 1 << 18;

// Finds, with one warp, the bin (counted from the top) of a histogram of NB
// bins that holds the k-th largest key, and the rank of that key inside the
// bin (1 = the bin's largest). Lane i owns the NB / 32 bins below the top
// i * NB / 32; a warp scan of the lanes' sums finds the lane that reaches k,
// and a second scan over that lane's bins, spread over the warp, finds the
// bin. Every lane returns the same result; with 1 <= k <= the histogram's
// total. Bins are read as int4 (hist 16-byte aligned).
template <int NB>
__device__ __forceinline__ void find_digit_warp(const int *hist, int k, uint32_t &digit, int &rank) {
  constexpr int PER = NB / 32;   // bins per lane
  constexpr int P2 = PER / 32;   // bins per lane in the second scan
  static_assert(PER % 4 == 0 && P2 >= 1 && PER % 32 == 0, "histogram size");
  const int lane = threadIdx.x & 31;
  const int4 *h4 = reinterpret_cast<const int4 *>(hist + NB - PER * (lane + 1));
  int sum = 0;
#pragma unroll
  for (int q = 0; q < PER / 4; ++q) {
    const int4 h = h4[(q + lane) % (PER / 4)];  // rotated: eight lanes hit eight bank groups
    sum += h.x + h.y + h.z + h.w;
  }
  int incl = sum;
#pragma unroll
  for (int sh = 1; sh < 32; sh <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, sh);
    if (lane >= sh) incl += y;
  }
  const unsigned hit = __ballot_sync(0xffffffffu, incl >= k);
  const int L = hit ? __ffs(hit) - 1 : 31;
  const int kk = k - __shfl_sync(0xffffffffu, incl - sum, L);
  const int top = NB - 1 - PER * L;  // the highest bin of lane L
  int c[P2], s2 = 0;
#pragma unroll
  for (int e = 0; e < P2; ++e) {
    c[e] = hist[top - lane * P2 - e];
    s2 += c[e];
  }
  int incl2 = s2;
#pragma unroll
  for (int sh = 1; sh < 32; sh <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl2, sh);
    if (lane >= sh) incl2 += y;
  }
  const unsigned hit2 = __ballot_sync(0xffffffffu, incl2 >= kk);
  const int J = hit2 ? __ffs(hit2) - 1 : 31;
  int dg = top - lane * P2, rk = kk - (incl2 - s2);
#pragma unroll
  for (int e = 0; e + 1 < P2; ++e) {
    if (rk <= c[e]) break;
    rk -= c[e];
    --dg;
  }
  digit = (uint32_t)__shfl_sync(0xffffffffu, dg, J);
  rank = __shfl_sync(0xffffffffu, rk, J);
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

// ---- cut and ordered write: one cluster of kCutCluster blocks per head -----
constexpr int kCutCluster = 4;                 // blocks per head
constexpr int kCutThreads = 512;
constexpr int kCutWarps = kCutThreads / 32;
constexpr int kCutLocalCap = 2048;             // bucket entries a block keeps
constexpr int kCutMaxWords = (kMaxSelectLmax / 32 + kCutCluster - 1) / kCutCluster;
constexpr int kCutPassC = 4;                   // chunks of 32 groups per warp and pass
constexpr int kCutWarpCap = 128;               // bucket entries a warp keeps
constexpr int kCutRB = 8;                      // rounds (of 4 groups) whose scores load together
static_assert(kCutWarps * kCutWarpCap == kCutLocalCap, "cut: the warps' lists fill the block's");
constexpr int kCutCand = 32;                   // final-digit candidates one warp resolves
static_assert(2048 == 4 * kCutThreads, "cut: one int4 of the first-digit histogram per thread");

// Shared memory of a cut block; the same layout in every block, so that a
// field's address maps to the same field of another block of the cluster.
struct CutSmem {
  int hist[2048];
  uint2 list[kCutWarps][kCutWarpCap];          // (key, position) of the block's bucket, per warp
  int slot[kCutWarps][kCutPassC * 32];         // a warp's active groups of a pass
  int wcount[kCutWarps];                       // entries of each warp (may pass the cap)
  uint32_t keys[kCutCluster][kCutLocalCap];    // leader: every block's bucket keys
  uint32_t gtw[kCutMaxWords];                  // the block's words: positions above the cut
  uint32_t eqw[kCutMaxWords];                  // positions whose key equals the cut
  uint32_t ckey[kCutCand];                     // leader: keys sharing the cut's top 22 bits
  int creg[kCutCand];                          //   and the block each came from
  int wcnt[2][kCutWarps];
  int rcnt[kCutCluster];                       // leader: every block's bucket size
  int rgt[kCutCluster];                        // leader: every block's count above the bucket
  int rG[kCutCluster], rE[kCutCluster];        // leader: above / equal to the cut, per block
  int ncand;
  int lcount;                                  // this block's bucket size (may pass the cap)
  int cgt;                                     // this block's positions above the bucket
  uint32_t s_digit;
  int s_k;
  uint32_t s_cut;
  int s_keq;
  // from the leader, for this block
  uint32_t cut;
  int keq;                                     // keys equal to the cut that this block keeps
  int base;                                    // kept positions in the blocks before this one
  int mode;                                    // 0 none, 1 all, 2 from the buckets, 3 from scans
  int written;                                 // leader: kept candidates of the head
};
constexpr size_t kCutSmemBytes = sizeof(CutSmem);

// Leader helper: adds, for every block r, the keys of block r above and equal
// to the cut (from the blocks' bucket keys, or, from_scores, from the scores
// in global memory over block r's positions) to rG[r] and rE[r].
__device__ __forceinline__ void count_against_cut(CutSmem &S, const float *sc, int n, int nwords,
                                                  int per, uint32_t cut, bool from_scores) {
  const int tid = threadIdx.x, lane = tid & 31;
#pragma unroll
  for (int r = 0; r < kCutCluster; ++r) {
    int gt = 0, eq = 0;
    if (!from_scores) {
      for (int i = tid; i < S.rcnt[r]; i += kCutThreads) {
        const uint32_t uu = S.keys[r][i];
        gt += uu > cut;
        eq += uu == cut;
      }
    } else {
      const int a = 32 * min(nwords, r * per), e = min(n, 32 * min(nwords, r * per + per));
      for (int tt = a + tid; tt < e; tt += kCutThreads) {
        const uint32_t uu = order_key(__ldcg(sc + tt));
        gt += uu > cut;
        eq += uu == cut;
      }
    }
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) {
      gt += __shfl_xor_sync(0xffffffffu, gt, sh);
      eq += __shfl_xor_sync(0xffffffffu, eq, sh);
    }
    if (lane == 0 && (gt | eq)) {
      atomicAdd(&S.rG[r], gt);
      atomicAdd(&S.rE[r], eq);
    }
  }
}

// Cluster (rank r of kCutCluster) per head bh. Rank r owns the head's
// candidate words [w0, w1) (32 positions each). The cut is the key of the
// ksel-th largest candidate, found by a radix select over 11, 11 and 10 bits,
// MSB first: every block takes the first digit from the score kernel's
// histogram, marks its positions above that digit's bucket and keeps the
// bucket's entries; the blocks send their bucket keys to the leader (rank 0),
// which finds the other two digits in its own shared memory (or by scans of
// the scores in global memory when a bucket does not fit), counts each block's
// positions above and equal to the cut, and sends every block its offset.
// Positions above the cut are kept; of the positions equal to it, the lowest.
// Each block then writes its kept positions in ascending order from its
// offset; rank 0 also writes the recent window, the padding and the count.
// Shared memory of another block is touched only between the first and the
// last cluster barrier, so that no block leaves while it may be accessed.
__global__ void __launch_bounds__(kCutThreads, 2) select_cut_kernel(const SelectParams p) {
  extern __shared__ __align__(16) unsigned char cut_smem[];
  CutSmem &S = *reinterpret_cast<CutSmem *>(cut_smem);
  pdl_launch_dependents();
  cluster_arrive_relaxed();  // this block has started
  const int rank = (int)cluster_ctarank();
  const int bh = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const HeadSel hs = head_sel(p, bh);
  const int L = hs.L, n = hs.n, ksel = hs.ksel;
  const int nwords = (n + 31) >> 5;
  const int per = (nwords + kCutCluster - 1) / kCutCluster;
  const int w0 = min(nwords, rank * per), w1 = min(nwords, w0 + per), nw = w1 - w0;
  const float *sc = p.scores + (size_t)bh * p.ldsc;
  for (int i = tid; i < nw; i += kCutThreads) {
    S.gtw[i] = 0u;
    S.eqw[i] = 0u;
  }
  if (tid == 0) {
    S.lcount = 0;
    S.cgt = 0;
  }
  pdl_wait();  // scores and histogram of the score pass
  // ---- first digit, and this block's span against it
  if (hs.search) {
    // Groups of 8 positions; the block's groups that hold candidates are
    // [gb, gend). Warp w takes chunks of 32 consecutive groups, w, w + 16, ...,
    // kCutPassC per pass. From the first digit of each group's largest score
    // it lists the groups that reach the bucket in its slots, then reads and
    // classifies them four at a time, eight lanes (one position each) per
    // group: one ballot gives the four groups' positions above the bucket,
    // another those in it.
    const uint16_t *gm = p.gmax + (size_t)bh * p.ldg;
    const int glast = (n + 7) >> 3;
    const int gb = 4 * w0, gend = min(4 * w1, glast);
    const int nch = (max(0, gend - gb) + 31) >> 5;
    auto load_max = [&](uint32_t (&md)[kCutPassC], int c0) {
#pragma unroll
      for (int i = 0; i < kCutPassC; ++i) {
        const int c = c0 + warp + kCutWarps * i;
        const int g = gb + 32 * c + lane;
        md[i] = c < nch && g < gend ? (uint32_t)__ldcg(gm + g) : 0xFFFFFFFFu;
      }
    };
    const int4 h4 = __ldcg(reinterpret_cast<const int4 *>(p.hist0 + (size_t)bh * 2048) + tid);
    uint32_t md[kCutPassC];
    load_max(md, 0);  // in flight while the first digit is found
    reinterpret_cast<int4 *>(S.hist)[tid] = h4;
    __syncthreads();
    if (warp == 0) {
      uint32_t dg;
      int rk;
      find_digit_warp<2048>(S.hist, ksel, dg, rk);
      if (lane == 0) {
        S.s_digit = dg;
        S.s_k = rk;
      }
    }
    __syncthreads();
    const uint32_t d0 = S.s_digit;
    // Away from NaN, infinities and the two zeros (digits 0..3, 1023, 1024
    // and 2044 up), the bucket d0 is the float interval [lo, hi) of its keys,
    // so two float compares classify a score. Elsewhere its key is compared.
    const bool fast = d0 >= 4 && d0 <= 2043 && d0 != 1023 && d0 != 1024;
    const float lo = key_float(d0 << 21), hi = key_float((d0 + 1) << 21);
    const uint32_t lt_mask = (1u << lane) - 1u;
    const int tq = lane >> 3, e = lane & 7;  // group of the round, position in it
    int *slot = S.slot[warp];
    uint2 *wl = S.list[warp];
    int wcnt = 0, cg = 0;  // the warp's bucket entries and positions above (warp-uniform)
    for (int c0 = 0; c0 < nch; c0 += kCutWarps * kCutPassC) {
      if (c0 > 0) load_max(md, c0);
      int na = 0;
#pragma unroll
      for (int i = 0; i < kCutPassC; ++i) {
        const bool act = md[i] <= 2047u && md[i] >= d0;
        const unsigned A = __ballot_sync(0xffffffffu, act);
        if (act) slot[na + __popc(A & lt_mask)] = 32 * (c0 + warp + kCutWarps * i) + lane;
        na += __popc(A);
      }
      __syncwarp();
      for (int r0 = 0; r0 < na; r0 += 4 * kCutRB) {
        float f[kCutRB];
        int grp[kCutRB];
#pragma unroll
        for (int q = 0; q < kCutRB; ++q) {
          const int k = r0 + 4 * q + tq;
          grp[q] = k < na ? slot[k] : -1;
          f[q] = grp[q] >= 0 ? __ldcg(sc + 8 * (gb + grp[q]) + e) : 0.f;
        }
#pragma unroll
        for (int q = 0; q < kCutRB; ++q) {
          if (r0 + 4 * q >= na) break;  // warp-uniform
          const int pos = 8 * (gb + grp[q]) + e;
          const bool in = grp[q] >= 0 && pos < n;
          bool above, inb;
          if (fast) {
            above = f[q] >= hi;
            inb = f[q] >= lo && !above;
          } else {
            const uint32_t dg = order_key(f[q]) >> 21;
            above = dg > d0;
            inb = dg == d0;
          }
          const unsigned ab = __ballot_sync(0xffffffffu, in && above);
          const unsigned bb = __ballot_sync(0xffffffffu, in && inb);
          if (e == 0 && grp[q] >= 0) {
            const uint32_t byte = (ab >> (8 * tq)) & 0xFFu;
            if (byte) atomicOr(&S.gtw[grp[q] >> 2], byte << (8 * (grp[q] & 3)));
          }
          cg += __popc(ab);
          if (bb) {  // warp-uniform
            if (in && inb) {
              const int o = wcnt + __popc(bb & lt_mask);
              if (o < kCutWarpCap) wl[o] = make_uint2(order_key(f[q]), (uint32_t)pos);
            }
            wcnt += __popc(bb);
          }
        }
      }
      __syncwarp();  // the slots are rewritten by the next pass
    }
    if (lane == 0) {
      S.wcount[warp] = wcnt;
      if (cg) atomicAdd(&S.cgt, cg);
    }
  }
  __syncthreads();
  cluster_wait();  // every block of the cluster has started: its shared memory is there
  // ---- every block sends its bucket keys and counts to the leader: warp w's
  // entries after those of the warps before it; a block whose bucket does not
  // fit reports more than the cap and sends none
  if (hs.search) {
    int pre = 0, total = 0;
    bool ovf = false;
#pragma unroll
    for (int w = 0; w < kCutWarps; ++w) {
      const int c = S.wcount[w];
      pre += w < warp ? c : 0;
      total += c;
      ovf = ovf || c > kCutWarpCap;
    }
    if (ovf) total = kCutLocalCap + 1;
    if (total <= kCutLocalCap) {
      const uint32_t dst = mapa_shared(smem_u32(&S.keys[rank][pre]), 0u);
      for (int i = lane; i < S.wcount[warp]; i += 32)
        st_cluster_u32(dst + 4u * (uint32_t)i, S.list[warp][i].x);
    }
    if (tid == 0) {
      S.lcount = total;
      st_cluster_u32(mapa_shared(smem_u32(&S.rcnt[rank]), 0u), (uint32_t)total);
      st_cluster_u32(mapa_shared(smem_u32(&S.rgt[rank]), 0u), (uint32_t)S.cgt);
    }
  }
  cluster_arrive();
  cluster_wait();  // the leader holds every block's keys and counts
  // ---- the leader finds the cut and every block's offset
  if (rank == 0) {
    if (tid < kCutCluster) {
      S.rG[tid] = 0;
      S.rE[tid] = 0;
    }
    if (tid == 0) S.ncand = 0;
    int mode = 0;
    if (!hs.search) {
      mode = ksel >= n && n > 0 ? 1 : 0;
      if (tid == 0) {
        S.s_cut = 0u;
        S.s_keq = 0;
      }
    } else {
      bool overflow = false;
#pragma unroll
      for (int r = 0; r < kCutCluster; ++r) overflow = overflow || S.rcnt[r] > kCutLocalCap;
      mode = overflow ? 3 : 2;
      const uint32_t d0 = S.s_digit;
      const int k0 = S.s_k;
      // second digit (key bits 20..10) over the bucket keys, or over a scan
      for (int i = tid; i < 2048; i += kCutThreads) S.hist[i] = 0;
      __syncthreads();
      if (!overflow) {
#pragma unroll
        for (int r = 0; r < kCutCluster; ++r)
          for (int i = tid; i < S.rcnt[r]; i += kCutThreads)
            atomicAdd(&S.hist[(S.keys[r][i] >> 10) & 2047u], 1);
      } else {
        for (int tt = tid; tt < n; tt += kCutThreads) {
          const uint32_t uu = order_key(__ldcg(sc + tt));
          if ((uu >> 21) == d0) atomicAdd(&S.hist[(uu >> 10) & 2047u], 1);
        }
      }
      __syncthreads();
      if (warp == 0) {
        uint32_t dg;
        int rk;
        find_digit_warp<2048>(S.hist, k0, dg, rk);
        if (lane == 0) {
          S.s_digit = dg;
          S.s_k = rk;
        }
      }
      __syncthreads();
      const uint32_t p22 = (d0 << 11) | S.s_digit;  // the cut's top 22 bits
      const int k1 = S.s_k;
      bool resolved = false;
      if (!overflow) {
        // keys above the top 22 bits, per block; the keys sharing them
        // collected for one warp
#pragma unroll
        for (int r = 0; r < kCutCluster; ++r) {
          int gt = 0;
          for (int i = tid; i < S.rcnt[r]; i += kCutThreads) {
            const uint32_t uu = S.keys[r][i];
            gt += (uu >> 10) > p22;
            if ((uu >> 10) == p22) {
              const int o = atomicAdd(&S.ncand, 1);
              if (o < kCutCand) {
                S.ckey[o] = uu;
                S.creg[o] = r;
              }
            }
          }
#pragma unroll
          for (int sh = 16; sh > 0; sh >>= 1) gt += __shfl_xor_sync(0xffffffffu, gt, sh);
          if (lane == 0 && gt) atomicAdd(&S.rG[r], gt);
        }
        __syncthreads();
        resolved = S.ncand <= kCutCand;
        if (resolved && warp == 0) {
          // the k1-th largest of the m candidates: a lane's key is the cut
          // when fewer than k1 keys are above it and at least k1 are not below
          const int m = S.ncand;
          const bool own = lane < m;
          const uint32_t key = own ? S.ckey[lane] : 0u;
          const int reg = own ? S.creg[lane] : -1;
          int above = 0, notbelow = 0;
          for (int j = 0; j < m; ++j) {
            const uint32_t kj = __shfl_sync(0xffffffffu, key, j);
            above += kj > key;
            notbelow += kj >= key;
          }
          const unsigned hit = __ballot_sync(0xffffffffu, own && above < k1 && k1 <= notbelow);
          const int src = hit ? __ffs(hit) - 1 : 0;
          const uint32_t cut = __shfl_sync(0xffffffffu, key, src);
          const int keq = k1 - __shfl_sync(0xffffffffu, above, src);
#pragma unroll
          for (int r = 0; r < kCutCluster; ++r) {
            const int gtx = __popc(__ballot_sync(0xffffffffu, own && reg == r && key > cut));
            const int eqx = __popc(__ballot_sync(0xffffffffu, own && reg == r && key == cut));
            if (lane == r) {
              S.rG[r] += gtx;
              S.rE[r] = eqx;
            }
          }
          if (lane == 0) {
            S.s_cut = cut;
            S.s_keq = keq;
          }
        }
      }
      if (!resolved) {
        // third digit (key bits 9..0) by a histogram, then every block's
        // counts against the cut
        for (int i = tid; i < 1024; i += kCutThreads) S.hist[i] = 0;
        if (tid < kCutCluster) S.rG[tid] = 0;
        __syncthreads();
        if (!overflow) {
#pragma unroll
          for (int r = 0; r < kCutCluster; ++r)
            for (int i = tid; i < S.rcnt[r]; i += kCutThreads) {
              const uint32_t uu = S.keys[r][i];
              if ((uu >> 10) == p22) atomicAdd(&S.hist[uu & 1023u], 1);
            }
        } else {
          for (int tt = tid; tt < n; tt += kCutThreads) {
            const uint32_t uu = order_key(__ldcg(sc + tt));
            if ((uu >> 10) == p22) atomicAdd(&S.hist[uu & 1023u], 1);
          }
        }
        __syncthreads();
        if (warp == 0) {
          uint32_t dg;
          int rk;
          find_digit_warp<1024>(S.hist, k1, dg, rk);
          if (lane == 0) {
            S.s_cut = (p22 << 10) | dg;
            S.s_keq = rk;
          }
        }
        __syncthreads();
        count_against_cut(S, sc, n, nwords, per, S.s_cut, overflow);
      }
    }
    __syncthreads();
    if (tid == 0) {
      const uint32_t cut = S.s_cut;
      const int keq = S.s_keq;
      int base = 0, eqseen = 0;
      for (int r = 0; r < kCutCluster; ++r) {
        int G = 0, E = 0;
        const int a = 32 * min(nwords, r * per), e = min(n, 32 * min(nwords, r * per + per));
        if (mode == 1) G = max(0, e - a);
        if (mode == 2) G = S.rgt[r] + S.rG[r], E = S.rE[r];
        if (mode == 3) G = S.rG[r], E = S.rE[r];
        const int kr = max(0, min(E, keq - eqseen));
        const uint32_t rr = (uint32_t)r;
        st_cluster_u32(mapa_shared(smem_u32(&S.cut), rr), cut);
        st_cluster_u32(mapa_shared(smem_u32(&S.keq), rr), (uint32_t)kr);
        st_cluster_u32(mapa_shared(smem_u32(&S.base), rr), (uint32_t)base);
        st_cluster_u32(mapa_shared(smem_u32(&S.mode), rr), (uint32_t)mode);
        base += G + kr;
        eqseen += E;
      }
      S.written = base;
    }
  }
  cluster_arrive();
  cluster_wait();  // every block holds its cut, count of equal keys and offset
  // ---- every block marks its positions against the cut and writes them
  const uint32_t cut = S.cut;
  const int keq = S.keq, mode = S.mode;
  if (mode == 1) {
    for (int i = tid; i < nw; i += kCutThreads) {
      const int rem = n - 32 * (w0 + i);
      S.gtw[i] = rem >= 32 ? 0xffffffffu : (1u << rem) - 1u;
    }
  } else if (mode == 2) {
    // mode 2: every warp's list fits (the leader saw no block over the cap)
    for (int i = lane; i < S.wcount[warp]; i += 32) {
      const uint2 e = S.list[warp][i];
      const int w = (int)(e.y >> 5) - w0;
      if (e.x > cut) atomicOr(&S.gtw[w], 1u << (e.y & 31));
      else if (e.x == cut) atomicOr(&S.eqw[w], 1u << (e.y & 31));
    }
  } else if (mode == 3) {
    for (int w = w0 + warp; w < w1; w += kCutWarps) {
      const int tt = 32 * w + lane;
      const uint32_t uu = tt < n ? order_key(__ldcg(sc + tt)) : 0u;
      const unsigned bg = __ballot_sync(0xffffffffu, tt < n && uu > cut);
      const unsigned be = __ballot_sync(0xffffffffu, tt < n && uu == cut);
      if (lane == 0) {
        S.gtw[w - w0] = bg;
        S.eqw[w - w0] = be;
      }
    }
  }
  __syncthreads();
  // warp w of the block owns local words [w*segw, (w+1)*segw)
  const int segw = (nw + kCutWarps - 1) / kCutWarps;
  const int v_lo = min(nw, warp * segw), v_hi = min(nw, v_lo + segw);
  {
    int cg = 0, ce = 0;
    for (int v = v_lo + lane; v < v_hi; v += 32) {
      cg += __popc(S.gtw[v]);
      ce += __popc(S.eqw[v]);
    }
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) {
      cg += __shfl_xor_sync(0xffffffffu, cg, sh);
      ce += __shfl_xor_sync(0xffffffffu, ce, sh);
    }
    if (lane == 0) {
      S.wcnt[0][warp] = cg;
      S.wcnt[1][warp] = ce;
    }
  }
  __syncthreads();
  // kept positions before this warp; the block keeps its keq lowest
  // positions equal to the cut
  int selp = S.base, eqp = 0;
  for (int w = 0; w < warp; ++w) {
    selp += S.wcnt[0][w] + max(0, min(S.wcnt[1][w], keq - eqp));
    eqp += S.wcnt[1][w];
  }
  int32_t *out = p.kept_idx + (size_t)bh * p.stride;
  // ascending write of the warp's words: one word per lane and step
  int wpos = selp, erank = eqp;
  for (int v0 = v_lo; v0 < v_hi; v0 += 32) {
    const int v = v0 + lane;
    const uint32_t gw = v < v_hi ? S.gtw[v] : 0u;
    uint32_t e = v < v_hi ? S.eqw[v] : 0u;
    const int ne = __popc(e);
    int ie = ne;
#pragma unroll
    for (int sh = 1; sh < 32; sh <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, ie, sh);
      if (lane >= sh) ie += y;
    }
    // keep the first max(0, keq - rank) equal keys of this word
    int take = min(ne, max(0, keq - (erank + ie - ne)));
    uint32_t et = 0;
    while (take-- > 0) {
      const uint32_t low = e & (0u - e);
      et |= low;
      e ^= low;
    }
    uint32_t sel = gw | et;
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
      if (o < p.stride) out[o] = (w0 + v) * 32 + bit;
      ++o;
      sel &= sel - 1;
    }
    wpos += __shfl_sync(0xffffffffu, is, 31);
    erank += __shfl_sync(0xffffffffu, ie, 31);
  }
  if (rank == 0) {
    if (tid == 0 && L != p.seq_len[bh / p.Hkv]) atomicOr(p.status, KVX_DEV_BAD_LENGTH);
    // recent window, then padding
    const int written = S.written;
    for (int t = n + tid; t < L; t += kCutThreads)
      if (written + (t - n) < p.stride) out[written + (t - n)] = t;
    const int cntk = written + (L - n);
    for (int i = cntk + tid; i < p.stride; i += kCutThreads) out[i] = -1;
    if (tid == 0) p.kept_count[bh] = cntk;
  }
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
constexpr int kPackRows = 2;
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

// Workspace: header | hist0 int32 [BH][2048] | gmax u16 [BH][ldg] | scores f32 [BH][ldsc], each
// section 256-byte aligned; hist0 is cleared by a kernel at the start of each call.
struct SelectWs {
  size_t hist0, gmax, scores, total;
  size_t ldsc, ldg;
};
SelectWs select_ws_offsets(size_t BH, size_t Lmax) {
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  SelectWs w;
  w.ldsc = (Lmax + 7) & ~size_t(7);
  w.ldg = ((Lmax + 7) / 8 + 7) & ~size_t(7);
  w.hist0 = KVX_WS_HEADER_BYTES;
  w.gmax = al(w.hist0 + sizeof(int32_t) * 2048 * BH);
  w.scores = al(w.gmax + sizeof(uint16_t) * BH * w.ldg);
  w.total = al(w.scores + sizeof(float) * BH * w.ldsc);
  return w;
}

extern "C" int kvx_select_workspace_bytes(int32_t B, int32_t Hkv, int32_t Lmax, size_t *bytes) {
  if (!bytes || B < 1 || Hkv < 1 || Lmax < 1) return KVX_EINVAL;
  *bytes = select_ws_offsets((size_t)B * Hkv, (size_t)Lmax).total;
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
  const SelectWs wl = select_ws_offsets(BH, (size_t)Lmax);
  char *ws = (char *)workspace;
  p.hist0 = (int32_t *)(ws + wl.hist0);
  p.gmax = (uint16_t *)(ws + wl.gmax);
  p.scores = (float *)(ws + wl.scores);
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
  p.ldsc = (int32_t)wl.ldsc;
  p.ldg = (int32_t)wl.ldg;
  cudaStream_t st = (cudaStream_t)stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kCutCluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // zero the first-digit histograms; the score pass starts as its
  // programmatic dependent and waits for it only before adding its counts
  const int hist4 = (int)(BH * 2048 / 4);
  cfg.gridDim = dim3((hist4 + kZeroThreads - 1) / kZeroThreads);
  cfg.blockDim = dim3(kZeroThreads);
  {
    const cudaError_t ez = cudaLaunchKernelEx(&cfg, select_zero_kernel,
                                              reinterpret_cast<int4 *>(p.hist0), hist4);
    if (ez != cudaSuccess) return set_cuda_error(ez);
  }
  cfg.gridDim = dim3((Lmax + kScoreTokensPerBlock - 1) / kScoreTokensPerBlock, B * Hkv);
  cfg.blockDim = dim3(kScoreThreads);
  cudaError_t e = D == 128 ? cudaLaunchKernelEx(&cfg, select_score_kernel<128>, p)
                           : cudaLaunchKernelEx(&cfg, select_score_kernel<64>, p);
  if (e != cudaSuccess) return set_cuda_error(e);
  // The cut kernel runs one cluster of kCutCluster blocks per head, as a
  // programmatic dependent of the score pass: it starts while that grid
  // drains and waits on the device for it.
  e = cudaFuncSetAttribute(select_cut_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kCutSmemBytes);
  if (e != cudaSuccess) return set_cuda_error(e);
  cfg.numAttrs = 2;
  cfg.gridDim = dim3(kCutCluster, B * Hkv);
  cfg.blockDim = dim3(kCutThreads);
  cfg.dynamicSmemBytes = kCutSmemBytes;
  e = cudaLaunchKernelEx(&cfg, select_cut_kernel, p);
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
