// plan.cpp -- host planner of the kvx library (no device code).
//
// Builds, ahead of time and from static budgets only, the work split of the
// decode-attention kernels ("Tangram: Unlocking Non-Uniform KV Cache for
// Efficient Multi-turn LLM Serving", AOT Load Balancing, Figs. 4(c), 5, 13):
// each head's kept tokens are cut into items and the items are packed onto
// thread blocks so that every block streams about the same number of KV
// bytes. Also reports the head-group page counts (Fig. 8) and the footprint
// they imply (Fig. 7, M(r)).
#include <algorithm>
#include <chrono>
#include <cmath>
#include <cstring>
#include <new>

#include "kvx_internal.h"

namespace kvx {
int set_cuda_error(cudaError_t e);  // abi.cpp

// Cost, in tokens, charged per work item on top of its tokens: the query
// load, the cross-warp merge and the partial write of an item take about as
// long as streaming this many tokens (a per-block trace of a sparse layer fits
// 1.4 us per item against 16 ns per token, i.e. about 85 tokens).
#ifndef KVX_ITEM_OVERHEAD_TOKENS
#define KVX_ITEM_OVERHEAD_TOKENS 96
#endif
static int item_overhead_tokens() { return KVX_ITEM_OVERHEAD_TOKENS; }

static bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

// Granularity of the balanced plan's cuts: a piece of a head may start at
// any multiple of min(P, stage) tokens, because the attention kernels fetch a
// stage as boxes of min(P, stage) rows that never cross a page.
static int cut_tokens(const kvx_plan *p) { return std::min(p->shape.page_size, kStageTokens); }

static void finish_splits(kvx_plan *p) {
  const int H = p->shape.B * p->shape.Hkv;
  std::vector<int32_t> count(H, 0);
  for (const Item &it : p->items) count[it.bh]++;
  std::vector<int32_t> first(H, -1), split_of(H, -1);
  int32_t slots = 0;
  for (int bh = 0; bh < H; ++bh) {
    if (count[bh] > 1) {
      first[bh] = slots;
      split_of[bh] = (int32_t)p->split_heads.size();
      p->split_heads.push_back(SplitHead{bh, slots, count[bh], kMergeGlobal, 0u, 0, 0, 0});
      slots += count[bh];
    }
  }
  // Slots of a split head follow its items' token order.
  std::vector<int32_t> next(first);
  std::vector<size_t> order(p->items.size());
  for (size_t i = 0; i < order.size(); ++i) order[i] = i;
  std::stable_sort(order.begin(), order.end(), [&](size_t a, size_t b) {
    const Item &x = p->items[a], &y = p->items[b];
    return x.bh != y.bh ? x.bh < y.bh : x.begin < y.begin;
  });
  for (size_t i : order) {
    Item &it = p->items[i];
    it.slot = count[it.bh] > 1 ? next[it.bh]++ : -1;
    it.split = split_of[it.bh];
  }
  p->num_slots = slots;
  // Inside each block, run the pieces of split heads first: the block that
  // finishes a head's last piece merges its partials, and doing that early
  // keeps the merges off the end of the kernel, behind ongoing streaming.
  for (int c = 0; c < p->num_ctas; ++c)
    std::stable_partition(p->items.begin() + p->cta_off[c], p->items.begin() + p->cta_off[c + 1],
                          [&](const Item &it) { return count[it.bh] > 1; });
  p->cta_tokens.assign(p->num_ctas, 0);
  for (int c = 0; c < p->num_ctas; ++c)
    for (int i = p->cta_off[c]; i < p->cta_off[c + 1]; ++i)
      p->cta_tokens[c] += p->items[i].end - p->items[i].begin;
}

// Blocks dispatched last. A launch that follows another kernel gets its
// blocks placed, in index order, into the slots that kernel's blocks free as
// they leave; the last blocks start latest (up to about 2 us after the median
// on a short launch) and have had the least time to fill their rings before
// the dependency wait. The last kLateFrac of the blocks are therefore charged
// kLateTokens more (measured on back-to-back decode layers: the sparse step
// 2.3 % faster, the Qwen3-4B and 32k steps 0.2 %, Qwen2.5-32B unchanged).
constexpr double kLateFrac = 0.3;
constexpr double kLateTokens = 48.0;

// Greedy fill of `heads` (in order) into blocks of cost at most `cap` each,
// less kLateTokens for the last kLateFrac of the blocks (tokens + c0 per
// item; a head's last sliver under one cut may pass the cap), cutting at
// multiples of cut_tokens; returns the number of blocks used, or max_ctas + 1
// if they do not suffice (out is then partial).
static int fill_blocks(const kvx_plan *p, const std::vector<int> &heads, double cap, double c0,
                       int max_ctas, std::vector<std::vector<Item>> *out) {
  const int T = cut_tokens(p);
  int c = 0;
  double used = 0;
  if (out) out->assign(max_ctas, {});
  const int late0 = (int)std::ceil((1.0 - kLateFrac) * max_ctas);
  for (int bh : heads) {
    const int n = p->n[bh];
    int pos = 0;
    while (pos < n) {
      if (c >= max_ctas) return max_ctas + 1;
      const int rem = n - pos;
      const double left = cap - (c >= late0 ? kLateTokens : 0.0) - used;
      if (left >= rem + c0) {
        if (out) (*out)[c].push_back(Item{bh, pos, n, -1, -1, 0, 0, 0});
        used += rem + c0;
        pos = n;
        continue;
      }
      int k = (int)std::floor((left - c0) / T) * T;
      if (k >= T) {
        if (rem - k < T) k = rem;  // take a sliver along (the cap is passed by < T)
        if (out) (*out)[c].push_back(Item{bh, pos, pos + k, -1, -1, 0, 0, 0});
        pos += k;
        if (pos == n) {
          used += k + c0;
          continue;
        }
      }
      ++c;  // the block is full
      used = 0;
    }
  }
  return used > 0 ? c + 1 : c;
}

// Balanced: lay the heads' kept tokens end to end, charge each item its
// tokens plus a fixed overhead, and cut the stream into at most num_ctas
// blocks whose cost is at most a common cap (less the late charge for the
// blocks dispatched last), at multiples of cut_tokens; the cap is the smallest
// (to a token) with which the stream fits.
static void plan_balanced(kvx_plan *p, int num_ctas) {
  const int H = p->shape.B * p->shape.Hkv;
  const double c0 = item_overhead_tokens();
  std::vector<int> heads(H);
  double total = 0;
  for (int bh = 0; bh < H; ++bh) {
    heads[bh] = bh;
    total += p->n[bh] + c0;
  }
  double lo = std::max(total / num_ctas, c0 + cut_tokens(p)), hi = lo;
  while (fill_blocks(p, heads, hi, c0, num_ctas, nullptr) > num_ctas) hi += c0 + kStageTokens;
  while (hi - lo > 1.0) {
    const double mid = 0.5 * (lo + hi);
    if (fill_blocks(p, heads, mid, c0, num_ctas, nullptr) <= num_ctas)
      hi = mid;
    else
      lo = mid;
  }
  std::vector<std::vector<Item>> cta;
  fill_blocks(p, heads, hi, c0, num_ctas, &cta);
  p->num_ctas = num_ctas;
  p->cta_off.assign(1, 0);
  for (int i = 0; i < num_ctas; ++i) {
    for (const Item &it : cta[i]) p->items.push_back(it);
    p->cta_off.push_back((int32_t)p->items.size());
  }
}

// ---- cluster layout --------------------------------------------------------
// Every head is either whole on one block or cut into pieces on blocks of one
// cluster of C blocks; a block holds at most one such piece and runs it last,
// so that its pieces can be merged through distributed shared memory when the
// block has nothing else to do. Heads are placed longest first: whole on the
// least loaded block where it fits under the cost cap, else cut, at stage
// boundaries, over the free blocks of the cluster with the most room (largest
// room first). Returns false if that does not fit under the cap.
struct ClusterFill {
  std::vector<std::vector<Item>> whole;  // per block
  std::vector<Item> piece;               // per block; bh < 0: none
};

static bool fill_cluster(const kvx_plan *p, const std::vector<int> &order, int C, int K,
                         double cap, double c0, ClusterFill *out) {
  const int T = kStageTokens, NB = K * C;
  std::vector<double> used(NB, 0.0);
  std::vector<char> has_piece(NB, 0);
  std::vector<std::pair<int64_t, int>> room;
  if (out) {
    out->whole.assign(NB, {});
    out->piece.assign(NB, Item{-1, 0, 0, -1, -1, 0, kMergeGlobal, 0});
  }
  for (int bh : order) {
    const int n = p->n[bh];
    int best = -1;
    for (int c = 0; c < NB; ++c)
      if (cap - used[c] >= n + c0 && (best < 0 || used[c] < used[best])) best = c;
    if (best >= 0) {
      used[best] += n + c0;
      if (out) out->whole[best].push_back(Item{bh, 0, n, -1, -1, 0, kMergeGlobal, 0});
      continue;
    }
    int bk = -1;
    int64_t bk_room = -1;
    for (int k = 0; k < K; ++k) {
      int64_t r = 0;
      for (int j = 0; j < C; ++j) {
        const int c = k * C + j;
        const double left = cap - used[c] - c0;
        if (!has_piece[c] && left >= T) r += (int64_t)std::floor(left / T) * T;
      }
      if (r > bk_room) {
        bk_room = r;
        bk = k;
      }
    }
    if (bk < 0 || bk_room < n) return false;
    room.clear();
    for (int j = 0; j < C; ++j) {
      const int c = bk * C + j;
      const double left = cap - used[c] - c0;
      if (!has_piece[c] && left >= T) room.push_back({(int64_t)std::floor(left / T) * T, c});
    }
    std::stable_sort(room.begin(), room.end(),
                     [](const std::pair<int64_t, int> &a, const std::pair<int64_t, int> &b) {
                       return a.first > b.first;
                     });
    int pos = 0;
    for (const auto &rc : room) {
      if (pos >= n) break;
      const int k = (int)std::min<int64_t>(rc.first, n - pos);
      has_piece[rc.second] = 1;
      used[rc.second] += k + c0;
      if (out) out->piece[rc.second] = Item{bh, pos, pos + k, -1, -1, 0, kMergeCluster, 0};
      pos += k;
    }
  }
  return true;
}

// Cluster layout on num_ctas blocks (a multiple of C): the smallest cost cap
// (to a token) with which fill_cluster succeeds. Each block runs its whole
// heads, then its piece. Returns false if no cap works.
static bool plan_cluster(kvx_plan *p, int C, int num_ctas) {
  const int K = num_ctas / C, H = p->shape.B * p->shape.Hkv;
  if (K < 1 || C < 2 || C > 8) return false;
  const double c0 = item_overhead_tokens();
  std::vector<int> order(H);
  double total = 0;
  for (int bh = 0; bh < H; ++bh) {
    order[bh] = bh;
    total += p->n[bh] + c0;
  }
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return p->n[a] > p->n[b]; });
  double lo = std::max(total / (K * C), c0 + kStageTokens), hi = lo;
  for (int guard = 0; !fill_cluster(p, order, C, K, hi, c0, nullptr); ++guard) {
    if (guard > 400) return false;
    hi += std::max(c0 + kStageTokens, 0.125 * hi);
  }
  while (hi - lo > 1.0) {
    const double mid = 0.5 * (lo + hi);
    if (fill_cluster(p, order, C, K, mid, c0, nullptr))
      hi = mid;
    else
      lo = mid;
  }
  ClusterFill f;
  fill_cluster(p, order, C, K, hi, c0, &f);
  p->items.clear();
  p->cta_off.assign(1, 0);
  for (int c = 0; c < K * C; ++c) {
    for (const Item &it : f.whole[c]) p->items.push_back(it);
    if (f.piece[c].bh >= 0) p->items.push_back(f.piece[c]);
    p->cta_off.push_back((int32_t)p->items.size());
  }
  p->num_ctas = K * C;
  p->cluster = C;
  return true;
}

// Split-head records of a cluster layout: piece index in token order, the
// cluster rank of each piece's block; no workspace slots.
static void finish_cluster_splits(kvx_plan *p) {
  const int H = p->shape.B * p->shape.Hkv, C = p->cluster;
  std::vector<int32_t> count(H, 0);
  for (const Item &it : p->items) count[it.bh]++;
  std::vector<int32_t> split_of(H, -1);
  std::vector<std::vector<std::pair<int32_t, int32_t>>> pieces(H);  // (begin, item index)
  for (size_t i = 0; i < p->items.size(); ++i)
    if (count[p->items[i].bh] > 1) pieces[p->items[i].bh].push_back({p->items[i].begin, (int)i});
  std::vector<int32_t> cta_of(p->items.size());
  for (int c = 0; c < p->num_ctas; ++c)
    for (int i = p->cta_off[c]; i < p->cta_off[c + 1]; ++i) cta_of[i] = c;
  for (int bh = 0; bh < H; ++bh) {
    if (count[bh] < 2) continue;
    std::sort(pieces[bh].begin(), pieces[bh].end());
    uint32_t ranks = 0;
    for (size_t k = 0; k < pieces[bh].size(); ++k) {
      Item &it = p->items[pieces[bh][k].second];
      it.piece = (int32_t)k;
      it.split = (int32_t)p->split_heads.size();
      it.slot = -1;
      it.mode = kMergeCluster;
      ranks |= (uint32_t)(cta_of[pieces[bh][k].second] % C) << (4 * k);
    }
    p->split_heads.push_back(SplitHead{bh, -1, count[bh], kMergeCluster, ranks, 0, 0, 0});
  }
  for (Item &it : p->items)
    if (count[it.bh] < 2) {  // a head left in one piece is a whole head
      it.mode = kMergeGlobal;
      it.slot = -1;
      it.split = -1;
      it.piece = 0;
    }
  p->num_slots = 0;
  p->cta_tokens.assign(p->num_ctas, 0);
  for (int c = 0; c < p->num_ctas; ++c)
    for (int i = p->cta_off[c]; i < p->cta_off[c + 1]; ++i)
      p->cta_tokens[c] += p->items[i].end - p->items[i].begin;
}

// One block per head, no split.
static void plan_per_head(kvx_plan *p) {
  const int H = p->shape.B * p->shape.Hkv;
  p->cta_off.assign(1, 0);
  for (int bh = 0; bh < H; ++bh) {
    p->items.push_back(Item{bh, 0, p->n[bh], -1, -1, 0, 0, 0});
    p->cta_off.push_back((int32_t)p->items.size());
  }
  p->num_ctas = H;
}

// Every head cut into the same number of equal pieces, one block per piece.
static void plan_uniform(kvx_plan *p, int sms) {
  const int H = p->shape.B * p->shape.Hkv;
  const int T = kStageTokens;
  const int splits = std::max(1, (2 * sms + H - 1) / H);
  p->cta_off.assign(1, 0);
  for (int bh = 0; bh < H; ++bh) {
    const int n = p->n[bh];
    int chunk = (n + splits - 1) / splits;
    chunk = ((chunk + T - 1) / T) * T;
    for (int b0 = 0; b0 < n; b0 += chunk) {
      p->items.push_back(Item{bh, b0, std::min(n, b0 + chunk), -1, -1, 0, 0, 0});
      p->cta_off.push_back((int32_t)p->items.size());
    }
  }
  p->num_ctas = (int32_t)p->items.size();
}

}  // namespace kvx

using namespace kvx;

extern "C" int kvx_device_sm_count(int32_t *sms) {
  if (!sms) return KVX_EINVAL;
  int dev = 0, v = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return set_cuda_error(e);
  *sms = v;
  return KVX_OK;
}

extern "C" int kvx_plan_create(const kvx_shape *s, const int32_t *head_budget,
                               const int32_t *seq_len,
                               const int32_t *head_group, int32_t num_ctas,
                               int32_t policy, int32_t kernel,
                               kvx_plan **out) {
  if (!out) return KVX_EINVAL;
  *out = nullptr;
  if (!s || !head_budget || !seq_len || !head_group) return KVX_EINVAL;
  const auto t0 = std::chrono::steady_clock::now();
  if (s->B < 1 || s->Hkv < 1 || s->Hq < 1 || s->num_groups < 1)
    return KVX_EINVAL;
  if (s->Hkv > KVX_MAX_KV_HEADS || s->num_groups > KVX_MAX_GROUPS ||
      s->num_groups > s->Hkv)
    return KVX_EUNSUPPORTED;
  if (s->Hq % s->Hkv != 0) return KVX_EINVAL;
  const int g = s->Hq / s->Hkv;
  if (g > KVX_MAX_GQA) return KVX_EUNSUPPORTED;
  if (s->D != 64 && s->D != 128) return KVX_EUNSUPPORTED;
  if (!is_pow2(s->page_size) || s->page_size < 8 || s->page_size > 128)
    return KVX_EUNSUPPORTED;
  if (s->dtype != KVX_F32 && s->dtype != KVX_BF16) return KVX_EUNSUPPORTED;
  if (s->layout != KVX_LAYOUT_HEAD_MAJOR && s->layout != KVX_LAYOUT_TOKEN_MAJOR)
    return KVX_EUNSUPPORTED;
  if (policy < KVX_PLAN_BALANCED || policy > KVX_PLAN_CLUSTER_8)
    return KVX_EINVAL;
  if (kernel < KVX_KERNEL_AUTO || kernel > KVX_KERNEL_SIMT) return KVX_EINVAL;
  int resolved = kernel;
  if (resolved == KVX_KERNEL_AUTO)
    resolved = s->dtype == KVX_BF16 ? KVX_KERNEL_MMA : KVX_KERNEL_SIMT;
  if (resolved == KVX_KERNEL_MMA && s->dtype != KVX_BF16)
    return KVX_EUNSUPPORTED;
  if (num_ctas < 0) return KVX_EINVAL;
  const int cluster_req = policy == KVX_PLAN_CLUSTER_2   ? 2
                          : policy == KVX_PLAN_CLUSTER_4 ? 4
                          : policy == KVX_PLAN_CLUSTER_8 ? 8
                                                         : 1;
  if (cluster_req > 1) {
    if (resolved != KVX_KERNEL_MMA) return KVX_EUNSUPPORTED;
    if (num_ctas % cluster_req != 0) return KVX_EINVAL;
  }

  const int B = s->B, Hkv = s->Hkv, G = s->num_groups, P = s->page_size;
  for (int h = 0; h < Hkv; ++h)
    if (head_group[h] < 0 || head_group[h] >= G) return KVX_EINVAL;
  for (int b = 0; b < B; ++b)
    if (seq_len[b] < 1) return KVX_EINVAL;
  for (int i = 0; i < B * Hkv; ++i)
    if (head_budget[i] < 1) return KVX_EINVAL;

  int sms = 0;
  if (((policy == KVX_PLAN_BALANCED || cluster_req > 1) && num_ctas == 0) ||
      policy == KVX_PLAN_UNIFORM) {
    if (num_ctas > 0) {
      sms = num_ctas;
    } else {
      int rc = kvx_device_sm_count(&sms);
      if (rc != KVX_OK) return rc;
    }
  }

  kvx_plan *p = new (std::nothrow) kvx_plan();
  if (!p) return KVX_ENOMEM;
  try {
    p->shape = *s;
    p->policy = policy;
    p->kernel = resolved;
    p->num_ctas = 0;
    p->cluster = 1;
    p->num_slots = 0;
    p->d_buf = nullptr;
    p->d_items = nullptr;
    p->d_cta_off = nullptr;
    p->d_n = nullptr;
    p->d_split = nullptr;
    p->d_trace = nullptr;
    p->d_cover = nullptr;
    p->cover_stride = 0;
    p->stall_block = -1;
    p->wait_ns = 2000000000ull;
    p->early_kv = 0;
    p->pf_tokens = 0;
    // Deterministic Budget Allocation: n = min(L, budget).
    p->n.resize((size_t)B * Hkv);
    for (int b = 0; b < B; ++b)
      for (int h = 0; h < Hkv; ++h)
        p->n[(size_t)b * Hkv + h] =
            std::min(seq_len[b], head_budget[(size_t)b * Hkv + h]);
    // Head groups: rows within a group in ascending head order.
    p->head_group.assign(head_group, head_group + Hkv);
    p->head_row.assign(Hkv, 0);
    p->group_size.assign(G, 0);
    for (int h = 0; h < Hkv; ++h) p->head_row[h] = p->group_size[head_group[h]]++;
    for (int gi = 0; gi < G; ++gi)
      if (p->group_size[gi] == 0) {
        delete p;
        return KVX_EINVAL;
      }
    p->group_pages.assign((size_t)G * B, 0);
    for (int b = 0; b < B; ++b)
      for (int h = 0; h < Hkv; ++h) {
        int32_t &pg = p->group_pages[(size_t)head_group[h] * B + b];
        pg = std::max(pg, (p->n[(size_t)b * Hkv + h] + P - 1) / P);
      }
    const int g = s->Hq / s->Hkv;
    const int resident = sms * (resolved == KVX_KERNEL_MMA ? attn_mma_ctas_per_sm() : 1);
    if (policy == KVX_PLAN_BALANCED) {
      plan_balanced(p, num_ctas > 0 ? num_ctas : resident);
      finish_splits(p);
    } else if (cluster_req > 1) {
      int nb = num_ctas;
      if (nb == 0) nb = std::min(attn_mma_max_clusters(s->D, g, cluster_req),
                                 resident / cluster_req) * cluster_req;
      if (nb < cluster_req || !plan_cluster(p, cluster_req, nb)) {
        delete p;
        return KVX_EUNSUPPORTED;
      }
      finish_cluster_splits(p);
    } else {
      if (policy == KVX_PLAN_PER_HEAD)
        plan_per_head(p);
      else
        plan_uniform(p, sms);
      finish_splits(p);
    }
    // L2 warm-up amount (short launches only)
    int64_t total = 0;
    for (int64_t v : p->cta_tokens) total += v;
    const int64_t mean = total / std::max(p->num_ctas, 1);
    const int64_t per_token = 2ll * s->D * (s->dtype == KVX_BF16 ? 2 : 4);
    p->pf_tokens = 0;
    if (mean <= KVX_ATTN_PREFETCH_MAX_BLOCK_TOKENS)
      p->pf_tokens = (int32_t)std::min<int64_t>(
          mean, ((int64_t)KVX_ATTN_PREFETCH_MB << 20) / (std::max(p->num_ctas, 1) * per_token));
  } catch (const std::bad_alloc &) {
    delete p;
    return KVX_ENOMEM;
  }
  p->plan_us = std::chrono::duration<double, std::micro>(
                   std::chrono::steady_clock::now() - t0)
                   .count();
  *out = p;
  return KVX_OK;
}

extern "C" int kvx_plan_upload(kvx_plan *p, void *stream) {
  if (!p) return KVX_EINVAL;
  if (p->d_buf) return KVX_OK;
  const size_t ni = p->items.size(), nc = p->cta_off.size(), nn = p->n.size(),
               ns = p->split_heads.size();
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t o_items = 0, o_cta = al(o_items + ni * sizeof(Item)),
               o_n = al(o_cta + nc * sizeof(int32_t)),
               o_split = al(o_n + nn * sizeof(int32_t)),
               total = al(o_split + std::max<size_t>(ns, 1) * sizeof(SplitHead));
  void *buf = nullptr;
  cudaError_t e = cudaMalloc(&buf, total);
  if (e != cudaSuccess) return set_cuda_error(e);
  char *b = (char *)buf;
  cudaStream_t st = (cudaStream_t)stream;
  e = cudaMemcpyAsync(b + o_items, p->items.data(), ni * sizeof(Item),
                      cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(b + o_cta, p->cta_off.data(), nc * sizeof(int32_t),
                        cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(b + o_n, p->n.data(), nn * sizeof(int32_t),
                        cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess && ns)
    e = cudaMemcpyAsync(b + o_split, p->split_heads.data(),
                        ns * sizeof(SplitHead), cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) {
    cudaFree(buf);
    return set_cuda_error(e);
  }
  p->d_buf = buf;
  p->d_items = (Item *)(b + o_items);
  p->d_cta_off = (int32_t *)(b + o_cta);
  p->d_n = (int32_t *)(b + o_n);
  p->d_split = (SplitHead *)(b + o_split);
  return KVX_OK;
}

AttnWs kvx::attn_ws_layout(const kvx_plan *p) {
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t g = (size_t)(p->shape.Hq / p->shape.Hkv);
  const size_t slots = (size_t)p->num_slots;
  AttnWs w;
  w.counters = KVX_WS_HEADER_BYTES;
  w.part_ml = al(w.counters + 4 * p->split_heads.size());
  w.part_o = al(w.part_ml + slots * g * sizeof(float2));
  w.total = w.part_o + slots * g * p->shape.D * sizeof(float);
  return w;
}

extern "C" int kvx_plan_workspace_bytes(const kvx_plan *p, size_t *bytes) {
  if (!p || !bytes) return KVX_EINVAL;
  *bytes = attn_ws_layout(p).total;
  return KVX_OK;
}

extern "C" int kvx_plan_get_stats(const kvx_plan *p, kvx_plan_stats *st) {
  if (!p || !st) return KVX_EINVAL;
  std::memset(st, 0, sizeof(*st));
  st->num_ctas = p->num_ctas;
  st->num_items = (int32_t)p->items.size();
  st->num_slots = p->num_slots;
  st->num_split_heads = (int32_t)p->split_heads.size();
  st->kernel = p->kernel;
  st->policy = p->policy;
  int64_t tot = 0, mx = 0;
  for (int32_t v : p->n) tot += v;
  for (int64_t v : p->cta_tokens) mx = std::max(mx, v);
  st->total_tokens = tot;
  st->max_cta_tokens = mx;
  st->mean_cta_tokens = p->num_ctas ? (double)tot / p->num_ctas : 0.0;
  const int B = p->shape.B, G = p->shape.num_groups, P = p->shape.page_size;
  int64_t alloc = 0;
  for (int gi = 0; gi < G; ++gi)
    for (int b = 0; b < B; ++b)
      alloc += (int64_t)p->group_pages[(size_t)gi * B + b] * p->group_size[gi] * P;
  st->slots_allocated = alloc;
  st->item_overhead = item_overhead_tokens();
  st->cluster = p->cluster;
  st->slots_used = tot;
  st->plan_us = p->plan_us;
  return KVX_OK;
}

extern "C" int kvx_plan_kept(const kvx_plan *p, int32_t *n) {
  if (!p || !n) return KVX_EINVAL;
  std::memcpy(n, p->n.data(), p->n.size() * sizeof(int32_t));
  return KVX_OK;
}

extern "C" int kvx_plan_group_pages(const kvx_plan *p, int32_t *pages) {
  if (!p || !pages) return KVX_EINVAL;
  std::memcpy(pages, p->group_pages.data(),
              p->group_pages.size() * sizeof(int32_t));
  return KVX_OK;
}

extern "C" int kvx_plan_items(const kvx_plan *p, int32_t *items,
                              int32_t *cta_off) {
  if (!p || !items || !cta_off) return KVX_EINVAL;
  for (size_t i = 0; i < p->items.size(); ++i) {
    items[4 * i + 0] = p->items[i].bh;
    items[4 * i + 1] = p->items[i].begin;
    items[4 * i + 2] = p->items[i].end;
    items[4 * i + 3] = p->items[i].slot;
  }
  std::memcpy(cta_off, p->cta_off.data(), p->cta_off.size() * sizeof(int32_t));
  return KVX_OK;
}

extern "C" int kvx_plan_cta_tokens(const kvx_plan *p, int64_t *tokens) {
  if (!p || !tokens) return KVX_EINVAL;
  std::memcpy(tokens, p->cta_tokens.data(),
              p->cta_tokens.size() * sizeof(int64_t));
  return KVX_OK;
}

extern "C" int kvx_plan_set_trace(kvx_plan *p, int64_t *dev_trace) {
  if (!p) return KVX_EINVAL;
  p->d_trace = dev_trace;
  return KVX_OK;
}

static int32_t plan_max_n(const kvx_plan *p) {
  int32_t mx = 1;
  for (int32_t v : p->n) mx = std::max(mx, v);
  return mx;
}

extern "C" int kvx_plan_coverage(const kvx_plan *p, int32_t *count) {
  if (!p || !count) return KVX_EINVAL;
  const int32_t mx = plan_max_n(p);
  std::memset(count, 0, sizeof(int32_t) * p->n.size() * (size_t)mx);
  for (const Item &it : p->items) {
    if (it.bh < 0 || (size_t)it.bh >= p->n.size() || it.begin < 0 || it.end > mx)
      return KVX_ERANGE;  // not reachable for a plan built by kvx_plan_create
    int32_t *row = count + (size_t)it.bh * mx;
    for (int32_t t = it.begin; t < it.end; ++t) row[t] += 1;
  }
  return KVX_OK;
}

extern "C" int kvx_plan_set_coverage_record(kvx_plan *p, int32_t *dev_count, int32_t stride) {
  if (!p) return KVX_EINVAL;
  if (dev_count && stride < plan_max_n(p)) return KVX_ERANGE;
  p->d_cover = dev_count;
  p->cover_stride = dev_count ? stride : 0;
  return KVX_OK;
}

extern "C" int kvx_plan_inject_stall(kvx_plan *p, int32_t block, uint64_t wait_limit_ns) {
  if (!p) return KVX_EINVAL;
  if (wait_limit_ns < 1000000ull || wait_limit_ns > 10000000000ull) return KVX_ERANGE;
  p->stall_block = block < 0 ? -1 : block;
  p->wait_ns = wait_limit_ns;
  return KVX_OK;
}

extern "C" int kvx_plan_set_early_kv(kvx_plan *p, int32_t enable) {
  if (!p || enable < 0 || enable > 1) return KVX_EINVAL;
  p->early_kv = enable;
  return KVX_OK;
}

extern "C" void kvx_plan_destroy(kvx_plan *p) {
  if (!p) return;
  if (p->d_buf) cudaFree(p->d_buf);
  delete p;
}
