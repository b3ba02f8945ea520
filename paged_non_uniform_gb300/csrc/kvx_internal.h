// kvx_internal.h -- structures shared by the host planner, the C ABI and the
// kernels of the kvx library. Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "kvx.h"

struct kvx_plan;

namespace kvx {

// Tokens one pipeline stage of the attention kernels covers (a multiple of
// every supported page size up to 32, and two 16-row MMA tiles).
constexpr int kStageTokens = 32;

// How a split head's partials are merged.
constexpr int kMergeGlobal = 0;   // partials in the workspace, last piece's block merges
constexpr int kMergeCluster = 1;  // pieces on blocks of one cluster, merged through
                                  // distributed shared memory by piece 0's block

// One work item: tokens [begin, end) of head bh = b*Hkv + h. split >= 0
// names the head's entry in the plan's split-head list. With a global merge,
// slot >= 0 is the partial-result slot; slot < 0 means the item covers the
// whole head and writes the final output. With a cluster merge, piece is the
// item's index among the head's pieces (token order) and the item is the last
// of its block.
struct alignas(16) Item {
  int32_t bh, begin, end, slot;
  int32_t split, piece, mode, pad;
};

// A split head: count pieces. Global merge: partials in slots [slot_begin,
// slot_begin + count). Cluster merge: piece i runs on the block of cluster
// rank (ranks >> 4i) & 15 of the cluster (at most 8 pieces).
struct SplitHead {
  int32_t bh, slot_begin, count, mode;
  uint32_t ranks;
  int32_t pad0, pad1, pad2;
};

struct GroupDesc {
  const int32_t *page_table;  // [B][stride]
  const void *k_pool;         // [num_pages][size][P][D]
  const void *v_pool;
  int64_t num_pages;
  int32_t stride;
  int32_t size;
};

// L2 warm-up by the tensor-core kernel while the previous kernel of the
// stream finishes: up to KVX_ATTN_PREFETCH_MB of K/V over the whole grid,
// and only for short launches (mean block load at most
// KVX_ATTN_PREFETCH_MAX_BLOCK_TOKENS), where the start-up is a large share of
// the launch; a long launch gains nothing and its first loads would queue
// behind the prefetches.
#ifndef KVX_ATTN_PREFETCH_MB
#define KVX_ATTN_PREFETCH_MB 16
#endif
#ifndef KVX_ATTN_PREFETCH_MAX_BLOCK_TOKENS
#define KVX_ATTN_PREFETCH_MAX_BLOCK_TOKENS 1024
#endif

// Kernel parameters of the attention kernels (passed by value as a
// __grid_constant__ argument; the tensor maps keep their 128-byte alignment).
struct alignas(128) AttnParams {
  CUtensorMap tmK[KVX_MAX_GROUPS];
  CUtensorMap tmV[KVX_MAX_GROUPS];
  GroupDesc grp[KVX_MAX_GROUPS];
  const Item *items;
  const int32_t *cta_off;
  const SplitHead *split;      // [split heads]
  int32_t *counters;           // [split heads] finished pieces, back to 0 after the merge
  const int32_t *n_plan;       // [B*Hkv]
  const int32_t *head_budget;  // [B*Hkv] device, for the plan check
  const int32_t *seq_len;      // [B] device
  const void *q;               // [B][Hq][D]
  float *out;                  // [B][Hq][D]
  float *part_o;               // [slots][g][D]
  float2 *part_ml;             // [slots][g] = (max in log2 units, sum)
  uint32_t *status;
  int64_t *trace;
  int32_t *cover;              // coverage record [B*Hkv][cover_stride], or null
  int32_t cover_stride;
  int32_t B, Hq, Hkv, D, g, P, num_groups, layout;
  float scale_log2;            // scale * log2(e)
  int32_t cluster;             // blocks per thread-block cluster (1: no clusters)
  int32_t stall_block;         // failure-detection test: block whose first stage gets no loads (-1: none)
  int32_t pf_tokens;           // tokens per block warmed into L2 before the dependency wait
  int32_t early_kv;            // 1: the producer may fill its ring before the dependency wait
  uint64_t wait_ns;            // limit of every pipeline wait
  // Kept-row attention (kvx_decode_attn_kept): token i of head bh is row
  // kept[bh * kept_stride + i] of the dense kdense / vdense [B*Hkv][Lmax][D];
  // null kept: head-group pages through the tensor maps.
  const int32_t *kept;
  const void *kdense;
  const void *vdense;
  int32_t kept_stride;
  int32_t Lmax;
  int8_t head_grp[KVX_MAX_KV_HEADS];
  int8_t head_row[KVX_MAX_KV_HEADS];
};

// Launchers (defined in the .cu files). Return cudaGetLastError().
cudaError_t launch_attn_mma(const AttnParams &p, int num_ctas, cudaStream_t st);
int attn_mma_ctas_per_sm();  // resident blocks per SM of the tensor-core kernel
// Clusters of `cluster` blocks of the tensor-core kernel (head dim D, GQA g)
// that can be resident at once on the current device; 0 if none or on error.
int attn_mma_max_clusters(int D, int g, int cluster);
cudaError_t launch_attn_simt(const AttnParams &p, int dtype, int num_ctas,
                             cudaStream_t st);

struct GatherParams {
  const int32_t *block_table;  // [S][max_blocks]
  const int32_t *num_blocks;   // [S]
  const void *pools[KVX_MAX_GATHER_TENSORS];
  void *stagings[KVX_MAX_GATHER_TENSORS];
  uint32_t *status;
  int64_t *totals;       // [0] runs, [1] live blocks
  int32_t *run_count;    // [S]
  int32_t *row_blocks;   // [S], -1 for a rejected row
  int32_t *run_off;      // [S+1] first run of each row in `runs`
  int64_t *row_bstart;   // [S+1] first live block of each row, all rows laid end to end
  int4 *runs;            // [total runs] = {first physical block or -1, row, first logical block, length}
  int64_t *run_bstart;   // [total runs] global index of each run's first block
  int64_t num_phys, block_bytes, row_bytes;
  int32_t S, max_blocks, num_tensors, flags;
};

// Workspace layout of decode attention (offsets in bytes from its start):
// header (status word) | split-head counters | partial (m, l) | partial o.
struct AttnWs {
  size_t counters, part_ml, part_o, total;
};
AttnWs attn_ws_layout(const kvx_plan *plan);

// Workspace layout of the gather (offsets in bytes from the workspace start).
struct GatherWs {
  size_t run_count, row_blocks, run_off, row_bstart, runs, run_bstart, total;
};
GatherWs gather_ws_layout(int S, int max_blocks);

cudaError_t launch_gather(const GatherParams &p, cudaStream_t st);
int set_cuda_error(cudaError_t e);  // records e for kvx_last_cuda_error


}  // namespace kvx

// The opaque plan.
struct kvx_plan {
  kvx_shape shape;
  int32_t policy, kernel, num_ctas;
  int32_t cluster;                   // blocks per cluster (1: no clusters)
  std::vector<int32_t> n;            // [B*Hkv]
  std::vector<int32_t> head_group;   // [Hkv]
  std::vector<int32_t> head_row;     // [Hkv]
  std::vector<int32_t> group_size;   // [G]
  std::vector<int32_t> group_pages;  // [G][B]
  std::vector<kvx::Item> items;
  std::vector<int32_t> cta_off;
  std::vector<kvx::SplitHead> split_heads;
  std::vector<int64_t> cta_tokens;
  int32_t num_slots;
  double plan_us;
  // device copies (kvx_plan_upload)
  void *d_buf;
  kvx::Item *d_items;
  int32_t *d_cta_off;
  int32_t *d_n;
  kvx::SplitHead *d_split;
  int64_t *d_trace;
  int32_t *d_cover;     // kvx_plan_set_coverage_record
  int32_t cover_stride;
  int32_t stall_block;  // kvx_plan_inject_stall
  uint64_t wait_ns;
  int32_t pf_tokens;    // tokens per block warmed into L2 before the dependency wait
  int32_t early_kv;     // kvx_plan_set_early_kv
};
