// attn_mma.cu -- split decode attention over head-group pages, bf16 K/V,
// tensor-core (warp MMA) path for sm_103a.
//
// Computes, for every work item {head (b,h), kept tokens [begin,end)} of the
// ahead-of-time plan ("Tangram: Unlocking Non-Uniform KV Cache for Efficient
// Multi-turn LLM Serving", AOT Load Balancing, Fig. 13), the softmax
// attention of the g query heads of KV head h over those tokens, either as
// the final output (item covers the head) or as a log-sum-exp partial
// (max, sum, un-normalised output) merged in the same launch (below).
//
// Data path, per thread block (two per SM, persistent over their items):
//  * one producer warp walks the items' pages through the head group's page
//    table (Fig. 8(b)) and issues one bulk-tensor load per page slot of K and
//    of V (a 5-D tensor map {64 elements, slot, half, head, page} covers both
//    page layouts; the box lands as [half][token row][128 B], 128-byte
//    swizzled) into a ring of 32-token stages, completing on mbarriers;
//  * kCons consumer warps take the stages round-robin (ring slot s always
//    belongs to warp s % kCons, so each warp sees its slots' mbarrier phases
//    in order). Each warp owns kStages / kCons slots, so one of its slots is
//    loading while it computes on another. Per stage a warp
//    computes S^T = K Q^T on m16n8k16 bf16 MMAs (16 tokens x 8 query columns;
//    GQA query heads of one KV head are the columns), runs the online softmax
//    on the accumulator fragments (column max by three shuffles), transposes
//    P into the B operand with movmatrix, and accumulates O^T += V^T P^T with
//    V^T fragments read by ldmatrix.trans. P is split into a bf16 high part
//    and a bf16 residual, so the product keeps ~16 bits of P;
//  * at the end of an item the consumer warps merge their (m, l, O) in shared
//    memory and write the output or, for a head cut into pieces, the piece's
//    partial; the block that completes a head's last piece then merges all its
//    partials (split_merge.cuh).
// No spin-wait is unbounded: every mbarrier wait gives up after p.wait_ns
// (2 s unless a test shortens it) and sets KVX_DEV_TIMEOUT. Pages outside the
// pool are loaded as zeros (the box is placed past the tensor's end) and set
// KVX_DEV_BAD_PAGE.
#include <math.h>

#include "kvx_internal.h"
#include "ptx.cuh"
#include "split_merge.cuh"

namespace kvx {
namespace {

// Tuning knobs (compile-time).
#ifndef KVX_ATTN_CONS
#define KVX_ATTN_CONS 3          // consumer warps per block
#endif
#ifndef KVX_ATTN_STAGES
#define KVX_ATTN_STAGES 6        // ring depth, in 32-token stages (2 slots per consumer)
#endif
#ifndef KVX_ATTN_CTAS_PER_SM
#define KVX_ATTN_CTAS_PER_SM 2   // resident blocks per SM
#endif
#ifndef KVX_ATTN_MERGE_BUFS
#define KVX_ATTN_MERGE_BUFS 1    // cross-warp merge records (2: alternate between items)
#endif
#ifndef KVX_TMA_LANES
#define KVX_TMA_LANES 1          // issue a stage's boxes from separate lanes
#endif
constexpr int kCons = KVX_ATTN_CONS;
constexpr int kStages = KVX_ATTN_STAGES;
constexpr int kMergeBufs = KVX_ATTN_MERGE_BUFS;
static_assert(kMergeBufs == 1 || kMergeBufs == 2, "one or two merge buffers");
// Stage gs goes to consumer warp gs % kCons and ring slot gs % kStages. With
// kStages a multiple of kCons every slot belongs to one warp, which waits on
// that slot's phases strictly in order. Otherwise a warp could wait for phase
// k of a slot while another warp's phase k-1 is still loading; a parity wait
// cannot tell those phases apart and would pass early.
static_assert(kStages % kCons == 0, "each ring slot must belong to one consumer warp");
static_assert(kCons <= 3, "the cross-warp merge keeps one weight per warp in a row's 4 padding floats");

template <int D>
struct Cfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kTile = kHalves * kStageTokens * 128;  // K (or V) bytes/stage
  static constexpr int kStage = 2 * kTile;
  static constexpr int kMS = D + 4;                   // merge row stride (floats)
  static constexpr int kMW = 8 * kMS + 16;            // floats per warp record
  static constexpr int kSmem =
      1024 + kStages * kStage + kMergeBufs * kCons * kMW * 4 + 2 * kStages * 8 + 16;
  // a launch in clusters also keeps its inbox barrier (cluster merge), after
  // the rest
  static constexpr int kSmemCluster = kSmem + 16;
};

// Load warp of kept-row attention (kvx_decode_attn_kept). Token i of head bh
// is row kept[bh * kept_stride + i] of the dense caches. Lane j copies row
// kept[t0 + j] of K and V into row j of the stage, into the same swizzled
// [half][row][128 B] tiles that one 32-row bulk-tensor box lands in (16-byte
// chunk c of row j goes to chunk c ^ (j & 7)), as 16-byte asynchronous
// copies; every lane's copies arrive on the stage's barrier as they land, and
// lane 0's plain arrival, made after all lanes have registered theirs, is the
// one the barrier was initialised to expect. The next stage's kept entries
// load while the warp waits for the stage's slot. An index outside
// [0, Lmax) loads a zero row and sets KVX_DEV_BAD_BLOCK.
template <int D>
__device__ __forceinline__ void produce_kept(const AttnParams &p, int it0, int it1,
                                             const Item &item0, uint32_t stage0,
                                             uint32_t full0, uint32_t empty0,
                                             volatile int *abort_flag, uint64_t pol, int lane,
                                             int &gs, bool &dead) {
  using C = Cfg<D>;
  for (int it = it0; it < it1 && !dead; ++it) {
    const Item item = it == it0 ? item0 : p.items[it];
    const int32_t *kl = p.kept + (size_t)item.bh * p.kept_stride;
    const size_t head_row0 = (size_t)item.bh * p.Lmax;
    int pos = item.begin + lane < item.end ? __ldg(kl + item.begin + lane) : 0;
    for (int t0 = item.begin; t0 < item.end; t0 += kStageTokens, ++gs) {
      const int slot = gs % kStages;
      const int valid = min(kStageTokens, item.end - t0);
      const int tn = t0 + kStageTokens + lane;
      const int pos_next = tn < item.end ? __ldg(kl + tn) : 0;
      if (gs >= kStages) {
        bool ok = true;
        if (lane == 0)
          ok = !*abort_flag && mbar_wait(empty0 + 8 * slot, ((gs / kStages) - 1) & 1, p.wait_ns);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) {
          if (lane == 0) {
            atomicOr(p.status, KVX_DEV_TIMEOUT);
            *abort_flag = 1;
          }
          dead = true;
          break;
        }
      }
      // Failure-detection test only: the chosen block arms nothing for its
      // first stage, so that stage's wait runs out.
      if (gs == 0 && (int)blockIdx.x == p.stall_block) {
        pos = pos_next;
        continue;
      }
      const uint32_t full = full0 + 8 * slot;
      if (lane < valid) {
        const bool in = pos >= 0 && pos < p.Lmax;
        if (!in) atomicOr(p.status, KVX_DEV_BAD_BLOCK);
        const size_t off = (head_row0 + (size_t)(in ? pos : 0)) * (size_t)(D * 2);
        const char *ks = (const char *)p.kdense + off;
        const char *vs = (const char *)p.vdense + off;
        const uint32_t nbytes = in ? 16u : 0u;
        const uint32_t kd = stage0 + slot * C::kStage + (uint32_t)lane * 128u;
#pragma unroll
        for (int hf = 0; hf < C::kHalves; ++hf)
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint32_t so =
                (uint32_t)hf * (kStageTokens * 128) + ((uint32_t)(c ^ (lane & 7)) << 4);
            cp_async_16(kd + so, ks + hf * 128 + c * 16, nbytes, pol);
            cp_async_16(kd + C::kTile + so, vs + hf * 128 + c * 16, nbytes, pol);
          }
      }
      cp_async_mbar_arrive(full);
      __syncwarp();
      if (lane == 0) mbar_arrive(full);
      pos = pos_next;
    }
  }
}

// Merge of a head whose pieces ran on blocks of one thread-block cluster
// (distributed shared memory, this GPU only). Every piece's block has left
// its merged (m, l, o) in its own ring, which is idle once its last item is
// done: o [g][D] floats from offset 0, then (m, l) [g] float2 (obox, the same
// offset in every block). The block of piece 0, once all others have arrived
// on its inbox barrier, reads the pieces through the cluster's shared window
// and folds them in piece order, as merge_split does for workspace partials.
template <int D, int NT, int V>
__device__ __forceinline__ void merge_cluster(const AttnParams &p, const SplitHead &sh, int tid,
                                              uint32_t obox) {
  const int g = p.g, cnt = sh.count, n4 = g * D / 4;
  const int b = sh.bh / p.Hkv, h = sh.bh - b * p.Hkv;
  float4 *out = reinterpret_cast<float4 *>(p.out + ((size_t)b * p.Hq + (size_t)h * g) * D);
  const uint32_t ml_off = (uint32_t)(g * D * 4);
#pragma unroll
  for (int k = 0; k < V; ++k) {
    const int q4 = tid + k * NT;
    if (q4 >= n4) continue;
    const int qi = (4 * q4) / D;
    float M = -INFINITY, L = 0.f;
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j0 = 0; j0 < cnt; j0 += 4) {  // four pieces per round trip
      float2 mv[4];
      float4 ov[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (j0 + j < cnt) {
          const uint32_t base = mapa_shared(obox, (sh.ranks >> (4 * (j0 + j))) & 15u);
          mv[j] = ld_cluster_f2(base + ml_off + 8u * qi);
          ov[j] = ld_cluster_f4(base + 16u * q4);
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (j0 + j < cnt) {
          const float mn = fmaxf(M, mv[j].x);
          const float a = ex2(M - mn), f = ex2(mv[j].x - mn);
          L = L * a + f * mv[j].y;
          O.x = O.x * a + f * ov[j].x;
          O.y = O.y * a + f * ov[j].y;
          O.z = O.z * a + f * ov[j].z;
          O.w = O.w * a + f * ov[j].w;
          M = mn;
        }
      }
    }
    const float r = 1.f / L;
    out[q4] = make_float4(O.x * r, O.y * r, O.z * r, O.w * r);
  }
}

// Shared-memory layout of a stage's K (or V) tile: the stage's 32 tokens
// come in boxes of `box_h` tokens (one bulk-tensor load each, box_h = min(P,
// 32)); box b holds [half][box_h rows][128 B] with the row's 16-byte chunks
// XOR-swizzled by the token's low 3 bits (128-byte swizzle). Every box and
// half starts on a 1024-byte boundary, so the swizzle key of a row is tok & 7.
// Row part of the offset of token `tok`:
__device__ __forceinline__ uint32_t row_off(int tok, int lb, int halves) {
  return (uint32_t)(((tok >> lb) << (lb + 7)) * halves + ((tok & ((1 << lb) - 1)) << 7));
}

// Per-lane ldmatrix addressing of one stage, fixed for the whole kernel.
struct LaneAddr {
  uint32_t krow[2], vrow[2];  // row offsets for the two 16-token m-tiles
  uint32_t half;              // bytes between the two 64-element halves
  int ksel, vsel, key;        // chunk parity of this lane's matrix, swizzle key
};

template <int D>
__device__ __forceinline__ LaneAddr lane_addr(int lane, int lb) {
  constexpr int H = D / 64;
  const int mi = lane >> 3, lr = lane & 7;
  LaneAddr a;
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
    a.krow[mt] = row_off(mt * 16 + (mi & 1) * 8 + lr, lb, H);
    a.vrow[mt] = row_off(mt * 16 + (mi >> 1) * 8 + lr, lb, H);
  }
  a.half = 1u << (lb + 7);
  a.ksel = mi >> 1;
  a.vsel = mi & 1;
  a.key = lr;
  return a;
}

// Offset of 16-byte chunk pair index `j` (dims 16j .. 16j+15), chunk `sel`.
__device__ __forceinline__ uint32_t chunk_off(const LaneAddr &a, int j, int sel) {
  return (uint32_t)(j >> 2) * a.half + ((uint32_t)(((2 * j) & 7) + sel) ^ (uint32_t)a.key) * 16u;
}

template <int D>
__device__ __forceinline__ void consume_stage(
    uint32_t kbase, uint32_t vbase, const LaneAddr &la, int valid,
    const uint32_t (&qf)[D / 16][2], float (&o)[D / 16][4], float &m0, float &m1,
    float &l0, float &l1, float sl2, int lane) {
  constexpr int NK = D / 16;
  const int r = lane >> 2, c = lane & 3;
  float s[2][4];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
    s[mt][0] = s[mt][1] = s[mt][2] = s[mt][3] = 0.f;
#pragma unroll
    for (int j = 0; j < NK; ++j) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(kbase + la.krow[mt] + chunk_off(la, j, la.ksel), a0, a1, a2, a3);
      mma_bf16(s[mt], a0, a1, a2, a3, qf[j][0], qf[j][1]);
    }
  }
  // s[mt][e]: token mt*16 + r (+8 for e >= 2), query column 2c + (e & 1).
  float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float x = s[mt][e] * sl2;
      const int tok = mt * 16 + r + ((e >> 1) << 3);
      x = tok < valid ? x : -INFINITY;
      s[mt][e] = x;
      if (e & 1)
        mx1 = fmaxf(mx1, x);
      else
        mx0 = fmaxf(mx0, x);
    }
#pragma unroll
  for (int sh = 4; sh < 32; sh <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, sh));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, sh));
  }
  const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
  const float al0 = ex2(m0 - mn0), al1 = ex2(m1 - mn1);
  m0 = mn0;
  m1 = mn1;
  float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float pv = ex2(s[mt][e] - ((e & 1) ? mn1 : mn0));
      s[mt][e] = pv;
      if (e & 1)
        ps1 += pv;
      else
        ps0 += pv;
    }
  l0 = l0 * al0 + ps0;
  l1 = l1 * al1 + ps1;
#pragma unroll
  for (int dm = 0; dm < NK; ++dm) {
    o[dm][0] *= al0;
    o[dm][1] *= al1;
    o[dm][2] *= al0;
    o[dm][3] *= al1;
  }
  // P^T as the B operand (k = tokens, n = query columns), high and residual.
  uint32_t bh[2][2], bl[2][2];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
    const uint32_t h01 = pack_bf16(s[mt][0], s[mt][1]);
    const uint32_t h23 = pack_bf16(s[mt][2], s[mt][3]);
    const float2 f01 = unpack_bf16(h01), f23 = unpack_bf16(h23);
    const uint32_t r01 = pack_bf16(s[mt][0] - f01.x, s[mt][1] - f01.y);
    const uint32_t r23 = pack_bf16(s[mt][2] - f23.x, s[mt][3] - f23.y);
    bh[mt][0] = movmatrix_t(h01);
    bh[mt][1] = movmatrix_t(h23);
    bl[mt][0] = movmatrix_t(r01);
    bl[mt][1] = movmatrix_t(r23);
  }
  const bool tail = valid < kStageTokens;
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
    // tokens held by this lane in the V^T fragment (for tail masking)
    const int t0 = mt * 16 + 2 * c;
    const uint32_t k01 = (t0 < valid ? 0x0000ffffu : 0u) | (t0 + 1 < valid ? 0xffff0000u : 0u);
    const uint32_t k89 = (t0 + 8 < valid ? 0x0000ffffu : 0u) | (t0 + 9 < valid ? 0xffff0000u : 0u);
#pragma unroll
    for (int dm = 0; dm < NK; ++dm) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4_t(vbase + la.vrow[mt] + chunk_off(la, dm, la.vsel), a0, a1, a2, a3);
      if (tail) {  // rows past the valid tokens may hold stale or padding data
        a0 &= k01;
        a1 &= k01;
        a2 &= k89;
        a3 &= k89;
      }
      mma_bf16(o[dm], a0, a1, a2, a3, bh[mt][0], bh[mt][1]);
      mma_bf16(o[dm], a0, a1, a2, a3, bl[mt][0], bl[mt][1]);
    }
  }
}

// VM: float4 groups of a head's g x D outputs that each consumer thread owns
// in the split merge (one kernel per VM keeps a single merge inlined).
// kCluster: the launch runs in thread-block clusters and merges cluster heads
// through distributed shared memory (a separate instance, so that launches
// without clusters carry none of that code).
template <int D, int VM, bool kCluster, bool kKept>
__global__ void __launch_bounds__((kCons + 1) * 32, KVX_ATTN_CTAS_PER_SM)
    attn_mma_kernel(const __grid_constant__ AttnParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment by pointer arithmetic on the shared array, so that
  // every pointer derived from it stays in the shared state space
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  float *merge = (float *)(smem + kStages * C::kStage);
  uint64_t *bars = (uint64_t *)(merge + kMergeBufs * kCons * C::kMW);
  volatile int *abort_flag = (volatile int *)(bars + 2 * kStages);
  volatile int *last_flag = abort_flag + 1;
  // cluster merge: the head's other pieces have arrived (cluster instance only)
  const uint32_t inbox = smem_u32(bars + 2 * kStages) + 16;
  const uint32_t stage0 = smem_u32(smem);
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kStages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int it0 = p.cta_off[blockIdx.x], it1 = p.cta_off[blockIdx.x + 1];
  const int P = p.P, g = p.g;
  uint64_t t_start = 0;
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    if (p.trace) t_start = globaltimer_ns();
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    // A block that merges a cluster head (it runs the head's piece 0 as its
    // last item) waits on its inbox for the head's other pieces.
    if (kCluster) {
      uint32_t expect = 1;
      if (it0 < it1) {
        const Item last = p.items[it1 - 1];
        if (last.mode == kMergeCluster && last.piece == 0)
          expect = (uint32_t)max(1, p.split[last.split].count - 1);
      }
      mbar_init(inbox, expect);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (!kKept && warp == kCons && lane < p.num_groups) {
    prefetch_tensormap(&p.tmK[lane]);
    prefetch_tensormap(&p.tmV[lane]);
  }
  __syncthreads();
  // Cluster barrier, phase 0: no block touches another's shared memory before
  // that block has initialised its barriers (every thread waits for this
  // phase before its first remote access, at the latest before the final
  // phase).
  bool phase0_done = !kCluster;
  if (kCluster) cluster_arrive();
  // Everything above touches only this block's shared memory and the kernel
  // parameters; global inputs may come from the previous kernel in the stream.
  if (!kKept && warp == kCons - 1 && p.pf_tokens > 0) {
    // While that kernel finishes, warm L2 with the first pf_tokens tokens of
    // this block's items (done by the consumer warp whose first stage comes
    // last, so that the producer's first loads are not held up). A prefetch changes no data, so a page-table entry
    // that the previous kernel is still rewriting costs at most a wasted
    // prefetch; the entries are read through L2 only (ld.global.cg), leaving
    // no copy in L1 for the loads after the wait.
    const int box_h = P < kStageTokens ? P : kStageTokens;
    int left = p.pf_tokens;
    for (int it = it0; it < it1 && left > 0; ++it) {
      const Item item = p.items[it];
      const int b = item.bh / p.Hkv, h = item.bh - b * p.Hkv;
      const int gi = p.head_grp[h], row = p.head_row[h];
      const GroupDesc &gd = p.grp[gi];
      const int32_t *pt = gd.page_table + (size_t)b * gd.stride;
      const int end = min(item.end, item.begin + left);
      const int nbox = (end - item.begin + box_h - 1) / box_h;
      for (int j = lane; j < nbox; j += 32) {
        const int tb = item.begin + j * box_h;
        const int32_t page = __ldcg(pt + tb / P);
        if (page >= 0 && (int64_t)page < gd.num_pages) {
          tma_prefetch_5d(&p.tmK[gi], 0, tb & (P - 1), 0, row, page);
          tma_prefetch_5d(&p.tmV[gi], 0, tb & (P - 1), 0, row, page);
        }
      }
      left -= end - item.begin;
    }
  }
  // The plan was uploaded (synchronously) before any call: its first item can
  // be read before the wait too.
  Item item0{};
  if (it0 < it1) item0 = p.items[it0];
  if (!(p.early_kv && warp == kCons)) pdl_wait();  // an early producer waits later

  if (warp == kCons) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = policy_evict_first();
    const int box_h = P < kStageTokens ? P : kStageTokens;
    const uint32_t box_bytes = (uint32_t)box_h * 128u * C::kHalves;
    int gs = 0;
    bool dead = false;
    bool waited = !p.early_kv;
    if constexpr (kKept)  // kept rows of a dense cache (the host turns early loads off)
      produce_kept<D>(p, it0, it1, item0, stage0, full0, empty0, abort_flag, pol, lane, gs, dead);
    for (int it = it0; it < it1 && !dead && !kKept; ++it) {
      const Item item = it == it0 ? item0 : p.items[it];
      const int b = item.bh / p.Hkv, h = item.bh - b * p.Hkv;
      const int gi = p.head_grp[h], row = p.head_row[h];
      const GroupDesc &gd = p.grp[gi];
      const int32_t *pt = gd.page_table + (size_t)b * gd.stride;
      const void *tmk = &p.tmK[gi];
      const void *tmv = &p.tmV[gi];
      const int maxpg = (item.end - 1) / P;
      const int last_pg = (__ldg(p.n_plan + item.bh) - 1) / P;  // the head's newest page
      int win = -1;
      int32_t my_page = 0;
      for (int t0 = item.begin; t0 < item.end; t0 += kStageTokens, ++gs) {
        const int slot = gs % kStages;
        const int valid = min(kStageTokens, item.end - t0);
        const int nbox = (valid + box_h - 1) / box_h;
        const int pg_last = (t0 + valid - 1) / P;
        // Early loads (kvx_plan_set_early_kv): before the preceding kernel has
        // completed, only stages clear of the head's newest page load, and
        // only into the empty ring; the page-table window is read again after
        // the wait.
        if (!waited && (gs >= kStages || pg_last >= last_pg)) {
          pdl_wait();
          waited = true;
          win = -1;
        }
        if (win < 0 || pg_last >= win + 32) {
          win = t0 / P;
          const int idx = win + lane;
          // through L2 only: an early read must leave no stale copy in L1
          my_page = idx <= maxpg ? __ldcg(pt + idx) : 0;
        }
        if (gs >= kStages) {
          bool ok = true;
          if (lane == 0)
            ok = !*abort_flag &&
                 mbar_wait(empty0 + 8 * slot, ((gs / kStages) - 1) & 1, p.wait_ns);
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
          if (!ok) {
            if (lane == 0) {
              atomicOr(p.status, KVX_DEV_TIMEOUT);
              *abort_flag = 1;
            }
            dead = true;
            break;
          }
        }
        const uint32_t full = full0 + 8 * slot;
        if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)nbox * box_bytes * 2u);
        __syncwarp();
        const uint32_t kdst = stage0 + slot * C::kStage;
#if KVX_TMA_LANES
        {
          const int i = lane < nbox ? lane : 0;
#else
        for (int i = 0; i < nbox; ++i) {
#endif
          const int tb = t0 + i * box_h;
          const int32_t page = __shfl_sync(0xffffffffu, my_page, tb / P - win);
#if KVX_TMA_LANES
          if (lane < nbox) {
#else
          if (lane == 0) {
#endif
            int pg = page;
            if (page < 0 || (int64_t)page >= gd.num_pages) {
              atomicOr(p.status, KVX_DEV_BAD_PAGE);
              pg = (int)gd.num_pages;  // whole box past the last page: loads zeros
            }
            const uint32_t d = kdst + (uint32_t)i * box_bytes;
            // Failure-detection test only: the chosen block arms its first
            // stage but loads nothing, so that stage's wait runs out.
            if (!(gs == 0 && (int)blockIdx.x == p.stall_block)) {
              tma_load_5d(d, tmk, 0, tb & (P - 1), 0, row, pg, full, pol);
              tma_load_5d(d + C::kTile, tmv, 0, tb & (P - 1), 0, row, pg, full, pol);
            }
          }
        }
      }
    }
    if (!waited) pdl_wait();
    // Do not leave while a load of ours may still be landing.
    if (lane == 0) {
      const int issued = gs;
      for (int s = 0; s < kStages && s < issued; ++s) {
        const int last = s + ((issued - 1 - s) / kStages) * kStages;
        if (!mbar_wait(full0 + 8 * s, (last / kStages) & 1, p.wait_ns))
          atomicOr(p.status, KVX_DEV_TIMEOUT);
      }
    }
  } else {
    // ----------------------------------------------------------- consumers
    constexpr int NK = D / 16;
    const int r = lane >> 2, c = lane & 3;
    const float sl2 = p.scale_log2;
    const int box_h = P < kStageTokens ? P : kStageTokens;
    // kept rows fill a stage as one 32-row tile
    const LaneAddr la = lane_addr<D>(lane, kKept ? 5 : 31 - __clz(box_h));
    int gs = 0;
    bool dead = false;
    for (int it = it0; it < it1; ++it) {
      const Item item = it == it0 ? item0 : p.items[it];
      const int b = item.bh / p.Hkv, h = item.bh - b * p.Hkv;
      if (warp == 0 && lane == 0) {
        const int L = __ldg(p.seq_len + b), bud = __ldg(p.head_budget + item.bh);
        if (min(L, bud) != __ldg(p.n_plan + item.bh))
          atomicOr(p.status, KVX_DEV_BAD_BUDGET);
      }
      uint32_t qf[NK][2];
      {
        const __nv_bfloat16 *qb = (const __nv_bfloat16 *)p.q +
                                  ((size_t)b * p.Hq + (size_t)h * g + r) * D;
#pragma unroll
        for (int j = 0; j < NK; ++j) {
          if (r < g) {
            qf[j][0] = __ldg((const uint32_t *)(qb + 16 * j + 2 * c));
            qf[j][1] = __ldg((const uint32_t *)(qb + 16 * j + 2 * c + 8));
          } else {
            qf[j][0] = qf[j][1] = 0u;
          }
        }
      }
      float o[NK][4];
#pragma unroll
      for (int dm = 0; dm < NK; ++dm) o[dm][0] = o[dm][1] = o[dm][2] = o[dm][3] = 0.f;
      float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
      const int nst = (item.end - item.begin + kStageTokens - 1) / kStageTokens;
      for (int st = 0; st < nst; ++st, ++gs) {
        if (gs % kCons != warp || dead) continue;
        const int slot = gs % kStages;
        bool ok = !*abort_flag;
        if (ok) ok = mbar_wait(full0 + 8 * slot, (gs / kStages) & 1, p.wait_ns);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
          if (lane == 0) {
            atomicOr(p.status, KVX_DEV_TIMEOUT);
            *abort_flag = 1;
          }
          dead = true;
          continue;
        }
        const int t0 = item.begin + st * kStageTokens;
        const int valid = min(kStageTokens, item.end - t0);
        const uint32_t kb = stage0 + slot * C::kStage;
        consume_stage<D>(kb, kb + C::kTile, la, valid, qf, o, m0, m1, l0, l1, sl2, lane);
        // Coverage record (test hook): one count per token this warp has
        // just fed to the softmax, taken here rather than from the plan.
        if (p.cover && lane < valid)
          atomicAdd(p.cover + (size_t)item.bh * p.cover_stride + t0 + lane, 1);
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * slot);
      }
      // ---- merge the consumer warps' partial states of this item
#pragma unroll
      for (int sh = 4; sh < 32; sh <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, sh);
        l1 += __shfl_xor_sync(0xffffffffu, l1, sh);
      }
      float *buf = merge + ((it - it0) % kMergeBufs) * kCons * C::kMW;
      float *mw = buf + warp * C::kMW;
#pragma unroll
      for (int dm = 0; dm < NK; ++dm) {
        mw[(2 * c) * C::kMS + 16 * dm + r] = o[dm][0];
        mw[(2 * c + 1) * C::kMS + 16 * dm + r] = o[dm][1];
        mw[(2 * c) * C::kMS + 16 * dm + r + 8] = o[dm][2];
        mw[(2 * c + 1) * C::kMS + 16 * dm + r + 8] = o[dm][3];
      }
      if (r == 0) {
        mw[8 * C::kMS + 2 * c] = m0;
        mw[8 * C::kMS + 2 * c + 1] = m1;
        mw[8 * C::kMS + 8 + 2 * c] = l0;
        mw[8 * C::kMS + 8 + 2 * c + 1] = l1;
      }
      consumer_sync(kCons * 32);
      const int tid = threadIdx.x;
      const bool in_cluster = kCluster && item.mode == kMergeCluster;
      float *obox = (float *)smem;  // cluster merge: this piece's (m, l, o), in the idle ring
      // Per query row, once: each warp's weight 2^(m_w - M) and the row's
      // 1 / sum, kept in the padding columns of warp 0's row.
      if (tid < g) {
        const int qi = tid;
        float M = -INFINITY, mw_[kCons];
#pragma unroll
        for (int w = 0; w < kCons; ++w) {
          mw_[w] = buf[w * C::kMW + 8 * C::kMS + qi];
          M = fmaxf(M, mw_[w]);
        }
        float Ls = 0.f;
        float *rf = buf + qi * C::kMS + D;
#pragma unroll
        for (int w = 0; w < kCons; ++w) {
          const float f = ex2(mw_[w] - M);
          rf[w] = f;
          Ls += f * buf[w * C::kMW + 8 * C::kMS + 8 + qi];
        }
        rf[3] = 1.f / Ls;
        if (in_cluster)
          reinterpret_cast<float2 *>(obox + g * D)[qi] = make_float2(M, Ls);
        else if (item.slot >= 0)
          p.part_ml[(size_t)item.slot * g + qi] = make_float2(M, Ls);
      }
      consumer_sync(kCons * 32);
      for (int q4 = tid; q4 < g * D / 4; q4 += kCons * 32) {
        const int qi = (4 * q4) / D, d4 = 4 * q4 - qi * D;
        const float4 rf = *reinterpret_cast<const float4 *>(buf + qi * C::kMS + D);
        const float fw[3] = {rf.x, rf.y, rf.z};
        float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kCons; ++w) {
          const float4 v = *reinterpret_cast<const float4 *>(buf + w * C::kMW + qi * C::kMS + d4);
          O.x = fmaf(fw[w], v.x, O.x);
          O.y = fmaf(fw[w], v.y, O.y);
          O.z = fmaf(fw[w], v.z, O.z);
          O.w = fmaf(fw[w], v.w, O.w);
        }
        if (in_cluster) {
          *reinterpret_cast<float4 *>(obox + qi * D + d4) = O;
        } else if (item.slot < 0) {
          *reinterpret_cast<float4 *>(p.out + ((size_t)b * p.Hq + (size_t)h * g + qi) * D + d4) =
              make_float4(O.x * rf.w, O.y * rf.w, O.z * rf.w, O.w * rf.w);
        } else {
          *reinterpret_cast<float4 *>(p.part_o + ((size_t)item.slot * g + qi) * D + d4) = O;
        }
      }
      // one merge buffer: the next item may overwrite it only after every
      // consumer has read it (a split item's ticket syncs below do that)
      if (kMergeBufs == 1 && item.slot < 0 && !in_cluster) consumer_sync(kCons * 32);
      if constexpr (kCluster) {
        if (in_cluster) {
          // This piece is the block's last item. Piece 0's block merges the
          // head; every other piece's block signals it once its (m, l, o) is
          // in its ring, and keeps that memory (it only waits at the final
          // cluster barrier, which the merging block passes after reading).
          fence_acq_rel_cluster();
          consumer_sync(kCons * 32);
          if (!phase0_done) {
            cluster_wait();
            phase0_done = true;
          }
          const SplitHead sh = p.split[item.split];
          // every rank the plan names must lie inside the cluster (never map
          // one outside; a damaged plan is reported, not followed)
          bool ranks_ok = sh.count >= 2 && sh.count <= 8;
          for (int j = 0; j < sh.count && j < 8; ++j)
            ranks_ok = ranks_ok && (int)((sh.ranks >> (4 * j)) & 15u) < p.cluster;
          if (!ranks_ok) {
            if (tid == 0) atomicOr(p.status, KVX_DEV_BAD_BUDGET);
          } else if (item.piece != 0) {
            if (tid == 0) mbar_arrive_remote(mapa_shared(inbox, sh.ranks & 15u));
          } else {
            const bool ok = __all_sync(0xffffffffu, mbar_wait_cluster(inbox, 0, p.wait_ns));
            if (ok)
              merge_cluster<D, kCons * 32, VM>(p, sh, tid, smem_u32(obox));
            else if (lane == 0)
              atomicOr(p.status, KVX_DEV_TIMEOUT);
          }
        }
      }
      if (!in_cluster && item.slot >= 0) {
        // Publish this piece; the block that finishes the head's last piece
        // merges all of them and rearms the counter for the next call. After
        // the barrier, one thread's acquire-release ticket releases every
        // partial write of the block (release is cumulative over the writes
        // the barrier ordered before it), and in the last block it acquires
        // the other blocks' partials for all its threads through the second
        // barrier.
        consumer_sync(kCons * 32);
        if (tid == 0)
          *last_flag = ticket_acq_rel(p.counters + item.split) == p.split[item.split].count - 1;
        consumer_sync(kCons * 32);
        if (*last_flag) {
          merge_split<D, kCons * 32, VM, 12>(p, p.split[item.split], tid);
          if (tid == 0) p.counters[item.split] = 0;
        }
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
  // Final cluster barrier: no block leaves while a merging block of its
  // cluster may still read its shared memory.
  if constexpr (kCluster) {
    if (!phase0_done) cluster_wait();
    cluster_arrive();
    cluster_wait();
  }
}

// Sets the kernel instance's shared-memory limit on the current device (once).
template <int D, int VM, bool kCluster, bool kKept>
cudaError_t configure_dv() {
  static int configured[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(attn_mma_kernel<D, VM, kCluster, kKept>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (kCluster ? Cfg<D>::kSmemCluster : Cfg<D>::kSmem));
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  return cudaSuccess;
}

template <int D, int VM, bool kCluster, bool kKept>
cudaError_t launch_dvc(const AttnParams &p, int num_ctas, cudaStream_t st) {
  cudaError_t e = configure_dv<D, VM, kCluster, kKept>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_ctas);
  cfg.blockDim = dim3((kCons + 1) * 32);
  cfg.dynamicSmemBytes = kCluster ? Cfg<D>::kSmemCluster : Cfg<D>::kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (kCluster) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)p.cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  e = cudaLaunchKernelEx(&cfg, attn_mma_kernel<D, VM, kCluster, kKept>, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int D, int VM>
cudaError_t launch_dv(const AttnParams &p, int num_ctas, cudaStream_t st) {
  if (p.kept)
    return p.cluster > 1 ? launch_dvc<D, VM, true, true>(p, num_ctas, st)
                         : launch_dvc<D, VM, false, true>(p, num_ctas, st);
  return p.cluster > 1 ? launch_dvc<D, VM, true, false>(p, num_ctas, st)
                       : launch_dvc<D, VM, false, false>(p, num_ctas, st);
}

template <int D, int VM>
int max_clusters_dv(int cluster) {
  if (configure_dv<D, VM, true, false>() != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)cluster);
  cfg.blockDim = dim3((kCons + 1) * 32);
  cfg.dynamicSmemBytes = Cfg<D>::kSmemCluster;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, attn_mma_kernel<D, VM, true, false>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

template <int D>
cudaError_t launch_d(const AttnParams &p, int num_ctas, cudaStream_t st) {
  constexpr int NT = kCons * 32;
  static_assert(KVX_MAX_GQA * D / 4 <= 3 * NT, "split merge: at most three groups per thread");
  const int n4 = p.g * D / 4;
  constexpr int VMAX = (KVX_MAX_GQA * D / 4 + NT - 1) / NT;
  if (n4 <= NT) return launch_dv<D, 1>(p, num_ctas, st);
  if constexpr (VMAX >= 2) {
    if (n4 <= 2 * NT) return launch_dv<D, 2>(p, num_ctas, st);
  }
  if constexpr (VMAX >= 3) return launch_dv<D, 3>(p, num_ctas, st);
  return cudaErrorInvalidValue;  // unreachable: g <= KVX_MAX_GQA
}

template <int D>
int max_clusters_d(int g, int cluster) {
  constexpr int NT = kCons * 32;
  constexpr int VMAX = (KVX_MAX_GQA * D / 4 + NT - 1) / NT;
  const int n4 = g * D / 4;
  if (n4 <= NT) return max_clusters_dv<D, 1>(cluster);
  if constexpr (VMAX >= 2) {
    if (n4 <= 2 * NT) return max_clusters_dv<D, 2>(cluster);
  }
  if constexpr (VMAX >= 3) return max_clusters_dv<D, 3>(cluster);
  return 0;
}

}  // namespace

int attn_mma_ctas_per_sm() { return KVX_ATTN_CTAS_PER_SM; }

int attn_mma_max_clusters(int D, int g, int cluster) {
  if (cluster < 2 || cluster > 8 || g < 1 || g > KVX_MAX_GQA) return 0;
  return D == 128 ? max_clusters_d<128>(g, cluster) : max_clusters_d<64>(g, cluster);
}

cudaError_t launch_attn_mma(const AttnParams &p, int num_ctas, cudaStream_t st) {
  if (num_ctas <= 0) return cudaSuccess;
  return p.D == 128 ? launch_d<128>(p, num_ctas, st) : launch_d<64>(p, num_ctas, st);
}

}  // namespace kvx
