// abi.cpp -- the C ABI entry points of kvx that launch device work:
// argument validation (everything is checked before anything is launched),
// bulk-tensor map encoding, kernel launches and workspace helpers.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "kvx_internal.h"

namespace kvx {

static thread_local int g_last_cuda_error = 0;

int set_cuda_error(cudaError_t e) {
  g_last_cuda_error = (int)e;
  return KVX_ECUDA;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t,
                                  void *, const cuuint64_t *, const cuuint64_t *,
                                  const cuuint32_t *, const cuuint32_t *,
                                  CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, []() {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)f;
  });
  return fn;
}

// A 5-D bf16 tensor map over one head-group pool, dims (innermost first)
// {64 elements, P slots, D/64 halves, |G| heads, pages}: one box
// {64, box_rows, D/64, 1, 1} fetches box_rows token rows of one head of one
// page and lands in shared memory as [half][row][128 B], 128-byte swizzled,
// zero-filled out of bounds. The two page layouts differ only in strides.
static bool encode_pool_map(CUtensorMap *tm, const void *base, int64_t pages,
                            int gsize, int P, int D, int layout, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t row = (cuuint64_t)D * 2;  // bytes of one token row of one head
  const cuuint32_t halves = (cuuint32_t)(D / 64);
  cuuint64_t dims[5] = {64u, (cuuint64_t)P, halves, (cuuint64_t)gsize, (cuuint64_t)pages};
  cuuint64_t strides[4];
  if (layout == KVX_LAYOUT_HEAD_MAJOR) {  // [|G|][P][D]
    strides[0] = row;                     // slot
    strides[2] = row * P;                 // head
  } else {                                // [P][|G|][D]
    strides[0] = row * gsize;             // slot
    strides[2] = row;                     // head
  }
  strides[1] = 128u;                      // half
  strides[3] = row * P * gsize;           // page
  cuuint32_t box[5] = {64u, (cuuint32_t)box_rows, halves, 1u, 1u};
  cuuint32_t estr[5] = {1u, 1u, 1u, 1u, 1u};
  CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

static bool aligned(const void *p, uintptr_t a) { return ((uintptr_t)p % a) == 0; }

}  // namespace kvx

using namespace kvx;

extern "C" const char *kvx_status_string(int s) {
  switch (s) {
    case KVX_OK: return "ok";
    case KVX_EINVAL: return "invalid argument";
    case KVX_ERANGE: return "index or length out of range";
    case KVX_ENOMEM: return "out of host memory";
    case KVX_ECUDA: return "CUDA runtime error";
    case KVX_EUNSUPPORTED: return "unsupported shape, page size, dtype or GQA factor";
    case KVX_ESTATE: return "plan not uploaded";
    case KVX_ENOBLOCKS: return "fewer free physical blocks than asked";
    case KVX_ESCRATCH: return "problem needs more scratch than the static buffer of kvx_gather_coalesce_noalloc holds";
    default: return "unknown status";
  }
}

extern "C" int kvx_last_cuda_error(void) { return g_last_cuda_error; }

namespace kvx {

// Checks and fills what both decode entry points share: the plan, q, out,
// the per-call device arrays, the workspace and the scale.
static int attn_common(const kvx_plan *plan, const void *q, const int32_t *head_budget,
                       const int32_t *seq_len, float scale, float *out, void *workspace,
                       size_t workspace_bytes, AttnParams &p) {
  if (!plan || !q || !head_budget || !seq_len || !out || !workspace) return KVX_EINVAL;
  if (!plan->d_buf) return KVX_ESTATE;
  const kvx_shape &s = plan->shape;
  size_t need = 0;
  kvx_plan_workspace_bytes(plan, &need);
  if (workspace_bytes < need || !aligned(workspace, 256)) return KVX_EINVAL;
  if (!std::isfinite(scale) || scale < 0.f) return KVX_EINVAL;
  if (!aligned(q, 16) || !aligned(out, 16)) return KVX_EINVAL;
  std::memset(&p, 0, sizeof(p));
  for (int h = 0; h < s.Hkv; ++h) {
    p.head_grp[h] = (int8_t)plan->head_group[h];
    p.head_row[h] = (int8_t)plan->head_row[h];
  }
  char *ws = (char *)workspace;
  const AttnWs lay = attn_ws_layout(plan);
  p.items = plan->d_items;
  p.cta_off = plan->d_cta_off;
  p.split = plan->d_split;
  p.counters = (int32_t *)(ws + lay.counters);
  p.n_plan = plan->d_n;
  p.head_budget = head_budget;
  p.seq_len = seq_len;
  p.q = q;
  p.out = out;
  p.status = (uint32_t *)ws;
  p.part_ml = (float2 *)(ws + lay.part_ml);
  p.part_o = (float *)(ws + lay.part_o);
  p.trace = plan->d_trace;
  p.cover = plan->d_cover;
  p.cover_stride = plan->cover_stride;
  p.B = s.B;
  p.Hq = s.Hq;
  p.Hkv = s.Hkv;
  p.D = s.D;
  p.g = s.Hq / s.Hkv;
  p.P = s.page_size;
  p.num_groups = s.num_groups;
  p.layout = s.layout;
  p.cluster = plan->cluster;
  p.stall_block = plan->stall_block;
  p.wait_ns = plan->wait_ns;
  const float sc = scale == 0.f ? 1.0f / std::sqrt((float)s.D) : scale;
  p.scale_log2 = (float)((double)sc * 1.4426950408889634);
  return KVX_OK;
}

}  // namespace kvx

extern "C" int kvx_decode_attn(const kvx_plan *plan, const void *q,
                               const void *const *k_pools,
                               const void *const *v_pools,
                               const int64_t *pool_pages,
                               const int32_t *const *page_tables,
                               const int32_t *page_table_stride,
                               const int32_t *head_budget,
                               const int32_t *seq_len, float scale, float *out,
                               void *workspace, size_t workspace_bytes,
                               void *stream) {
  if (!k_pools || !v_pools || !pool_pages || !page_tables || !page_table_stride)
    return KVX_EINVAL;
  AttnParams p;
  const int rc = attn_common(plan, q, head_budget, seq_len, scale, out, workspace,
                             workspace_bytes, p);
  if (rc != KVX_OK) return rc;
  const kvx_shape &s = plan->shape;
  const int G = s.num_groups, B = s.B, P = s.page_size, D = s.D;
  for (int gi = 0; gi < G; ++gi) {
    if (!k_pools[gi] || !v_pools[gi] || !page_tables[gi]) return KVX_EINVAL;
    if (!aligned(k_pools[gi], 16) || !aligned(v_pools[gi], 16)) return KVX_EINVAL;
    if (pool_pages[gi] < 1) return KVX_EINVAL;
    if (pool_pages[gi] >= ((int64_t)1 << 31) - 1) return KVX_ERANGE;
    int32_t mx = 0;
    for (int b = 0; b < B; ++b) mx = std::max(mx, plan->group_pages[(size_t)gi * B + b]);
    if (page_table_stride[gi] < std::max(mx, 1)) return KVX_ERANGE;
    GroupDesc &gd = p.grp[gi];
    gd.page_table = page_tables[gi];
    gd.k_pool = k_pools[gi];
    gd.v_pool = v_pools[gi];
    gd.num_pages = pool_pages[gi];
    gd.stride = page_table_stride[gi];
    gd.size = plan->group_size[gi];
    if (plan->kernel == KVX_KERNEL_MMA) {
      const int box = std::min(P, kStageTokens);
      if (!encode_pool_map(&p.tmK[gi], k_pools[gi], pool_pages[gi], plan->group_size[gi], P, D,
                           s.layout, box) ||
          !encode_pool_map(&p.tmV[gi], v_pools[gi], pool_pages[gi], plan->group_size[gi], P, D,
                           s.layout, box))
        return set_cuda_error(cudaErrorInvalidValue);
    }
  }
  p.early_kv = plan->early_kv;
  // with early loads into the ring, the L2 warm-up only competes with them
  p.pf_tokens = plan->early_kv ? 0 : plan->pf_tokens;

  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = plan->kernel == KVX_KERNEL_MMA
                      ? launch_attn_mma(p, plan->num_ctas, st)
                      : launch_attn_simt(p, s.dtype, plan->num_ctas, st);
  if (e != cudaSuccess) return set_cuda_error(e);
  return KVX_OK;
}

extern "C" int kvx_decode_attn_kept(const kvx_plan *plan, const void *q, const void *keys,
                                    const void *values, int32_t Lmax,
                                    const int32_t *kept_idx, int32_t kept_stride,
                                    const int32_t *head_budget, const int32_t *seq_len,
                                    float scale, float *out, void *workspace,
                                    size_t workspace_bytes, void *stream) {
  if (!keys || !values || !kept_idx) return KVX_EINVAL;
  AttnParams p;
  const int rc = attn_common(plan, q, head_budget, seq_len, scale, out, workspace,
                             workspace_bytes, p);
  if (rc != KVX_OK) return rc;
  if (plan->shape.dtype != KVX_BF16 || plan->kernel != KVX_KERNEL_MMA) return KVX_EUNSUPPORTED;
  if (Lmax < 1 || kept_stride < 1) return KVX_EINVAL;
  if (!aligned(keys, 16) || !aligned(values, 16)) return KVX_EINVAL;
  int32_t maxn = 0;
  for (int32_t v : plan->n) maxn = std::max(maxn, v);
  if (maxn > kept_stride) return KVX_ERANGE;
  p.kept = kept_idx;
  p.kdense = keys;
  p.vdense = values;
  p.kept_stride = kept_stride;
  p.Lmax = Lmax;
  // the kept list comes from the work before the call: no loads before the
  // dependency wait, and no L2 warm-up (it walks page tables)
  p.early_kv = 0;
  p.pf_tokens = 0;
  cudaError_t e = launch_attn_mma(p, plan->num_ctas, (cudaStream_t)stream);
  if (e != cudaSuccess) return set_cuda_error(e);
  return KVX_OK;
}

extern "C" int kvx_workspace_status(const void *workspace, uint32_t *status) {
  if (!workspace || !status) return KVX_EINVAL;
  cudaError_t e = cudaMemcpy(status, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return set_cuda_error(e);
  return KVX_OK;
}

extern "C" int kvx_workspace_clear(void *workspace, size_t bytes, void *stream) {
  if (!workspace || bytes < KVX_WS_HEADER_BYTES) return KVX_EINVAL;
  cudaError_t e = cudaMemsetAsync(workspace, 0, bytes, (cudaStream_t)stream);
  if (e != cudaSuccess) return set_cuda_error(e);
  return KVX_OK;
}

extern "C" int kvx_gather_workspace_bytes(int32_t S, int32_t max_blocks, size_t *bytes) {
  if (!bytes || S < 0 || max_blocks < 0) return KVX_EINVAL;
  *bytes = gather_ws_layout(S, max_blocks).total;
  return KVX_OK;
}

extern "C" int kvx_gather_coalesce(const int32_t *block_table,
                                   const int32_t *num_blocks, int32_t S,
                                   int32_t max_blocks, int32_t num_tensors,
                                   const void *const *pools,
                                   int64_t num_phys_blocks, int64_t block_bytes,
                                   void *const *stagings,
                                   int64_t staging_row_bytes, int32_t flags,
                                   void *workspace, size_t workspace_bytes,
                                   void *stream) {
  if (!block_table || !num_blocks || !pools || !stagings || !workspace) return KVX_EINVAL;
  if (S < 0 || max_blocks < 0 || num_tensors < 1 || num_tensors > KVX_MAX_GATHER_TENSORS)
    return KVX_EINVAL;
  if (num_phys_blocks < 1 || block_bytes < 16 || block_bytes % 16 != 0 ||
      staging_row_bytes < 0 || staging_row_bytes % 16 != 0)
    return KVX_EINVAL;
  if (flags & ~KVX_ZERO_TAIL) return KVX_EINVAL;
  const GatherWs w = gather_ws_layout(S, max_blocks);
  if (workspace_bytes < w.total || !aligned(workspace, 256)) return KVX_EINVAL;
  GatherParams p;
  std::memset(&p, 0, sizeof(p));
  for (int t = 0; t < num_tensors; ++t) {
    if (!pools[t] || !stagings[t] || !aligned(pools[t], 16) || !aligned(stagings[t], 16))
      return KVX_EINVAL;
    p.pools[t] = pools[t];
    p.stagings[t] = stagings[t];
  }
  char *ws = (char *)workspace;
  p.block_table = block_table;
  p.num_blocks = num_blocks;
  p.status = (uint32_t *)ws;
  p.totals = (int64_t *)(ws + 16);
  p.run_count = (int32_t *)(ws + w.run_count);
  p.row_blocks = (int32_t *)(ws + w.row_blocks);
  p.run_off = (int32_t *)(ws + w.run_off);
  p.row_bstart = (int64_t *)(ws + w.row_bstart);
  p.runs = (int4 *)(ws + w.runs);
  p.run_bstart = (int64_t *)(ws + w.run_bstart);
  p.num_phys = num_phys_blocks;
  p.block_bytes = block_bytes;
  p.row_bytes = staging_row_bytes;
  p.S = S;
  p.max_blocks = max_blocks;
  p.num_tensors = num_tensors;
  p.flags = flags;
  cudaError_t e = launch_gather(p, (cudaStream_t)stream);
  if (e != cudaSuccess) return set_cuda_error(e);
  return KVX_OK;
}

extern "C" int kvx_gather_read_runs(const void *workspace, int32_t S,
                                    int32_t max_blocks, int32_t *run_count,
                                    int32_t *runs) {
  if (!workspace || !run_count || !runs || S < 0 || max_blocks < 0) return KVX_EINVAL;
  const GatherWs w = gather_ws_layout(S, max_blocks);
  const char *ws = (const char *)workspace;
  std::vector<int32_t> off((size_t)S + 1);
  cudaError_t e = cudaMemcpy(run_count, ws + w.run_count, 4 * (size_t)S, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess)
    e = cudaMemcpy(off.data(), ws + w.run_off, 4 * ((size_t)S + 1), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return set_cuda_error(e);
  const int64_t total = off[S];
  std::vector<int4> all((size_t)std::max<int64_t>(total, 1));
  if (total > 0) {
    e = cudaMemcpy(all.data(), ws + w.runs, 16 * (size_t)total, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return set_cuda_error(e);
  }
  std::memset(runs, 0, sizeof(int32_t) * 3 * (size_t)S * (size_t)max_blocks);
  for (int s = 0; s < S; ++s) {
    // the counts come from the device: never index past either array
    const int64_t n = std::min<int64_t>({run_count[s], max_blocks, total - off[s]});
    for (int r = 0; r < n; ++r) {
      const int4 &d = all[(size_t)off[s] + r];
      int32_t *o = runs + ((size_t)s * max_blocks + r) * 3;
      o[0] = d.x;
      o[1] = d.z;
      o[2] = d.w;
    }
  }
  return KVX_OK;
}
