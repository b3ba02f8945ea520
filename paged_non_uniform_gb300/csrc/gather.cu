// gather.cu -- KV-RM movement step: merge a fragmented block table into runs
// and copy each run into a fixed-shape staging buffer.
//
// "KV-RM: Regularizing KV-Cache Movement for Static-Graph LLM Serving",
// Fig. 3 (descriptor merging turns fragmented page descriptors into a few
// large transfers) and abstract / Fig. 2 (the transfers fill the fixed-shape
// buffer the static attention kernel reads). The page's own transport uses
// DMA copy engines on A100s; here the copies are SM kernels with 16-byte
// streaming loads and stores, balanced over the GPU by bytes.
//
// Kernels, in stream order:
//   count  one block per row: validate the row, count its runs;
//   scan   one block: exclusive prefix sums of run counts and live blocks;
//   emit   one block per row: write the row's runs {src, row, dst, len}
//          at its offset and the global index of each run's first block;
//   copy   persistent blocks, each owns an equal share of all live blocks,
//          walks the runs covering it and copies them contiguously;
//   tail   (KVX_ZERO_TAIL) zero every row past its live blocks.
#include <mutex>

#include "kvx_internal.h"
#include "ptx.cuh"

namespace kvx {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ bool valid_block(int32_t id, int64_t num_phys) {
  return id >= 0 && (int64_t)id < num_phys;
}

// Block j of `row` starts a new run unless it and block j-1 are both valid
// and physically consecutive.
__device__ __forceinline__ int run_start(const int32_t *row, int j,
                                         int64_t num_phys) {
  if (j == 0) return 1;
  const int32_t a = row[j - 1], b = row[j];
  return !(valid_block(a, num_phys) && valid_block(b, num_phys) &&
           (int64_t)b == (int64_t)a + 1);
}

__device__ __forceinline__ bool row_ok(const GatherParams &p, int nb) {
  return nb >= 0 && nb <= p.max_blocks && (int64_t)nb * p.block_bytes <= p.row_bytes;
}

// Exclusive block-wide scan of one int per thread; returns the block total.
__device__ __forceinline__ int block_excl_scan(int v, int &excl) {
  __shared__ int wsum[kThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int sh = 1; sh < 32; sh <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, sh);
    if (lane >= sh) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kThreads / 32 ? wsum[lane] : 0;
#pragma unroll
    for (int sh = 1; sh < 32; sh <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, sh);
      if (lane >= sh) w += y;
    }
    if (lane < kThreads / 32) wsum[lane] = w;
  }
  __syncthreads();
  const int before = warp ? wsum[warp - 1] : 0;
  const int total = wsum[kThreads / 32 - 1];
  excl = before + x - v;
  __syncthreads();
  return total;
}

__global__ void __launch_bounds__(kThreads) gather_count_kernel(const GatherParams p) {
  const int s = blockIdx.x;
  const int nb = p.num_blocks[s];
  if (!row_ok(p, nb)) {
    if (threadIdx.x == 0) {
      atomicOr(p.status, KVX_DEV_BAD_LENGTH);
      p.run_count[s] = 0;
      p.row_blocks[s] = -1;
    }
    return;
  }
  const int32_t *row = p.block_table + (size_t)s * p.max_blocks;
  int cnt = 0;
  for (int j = threadIdx.x; j < nb; j += kThreads) cnt += run_start(row, j, p.num_phys);
  int excl;
  const int total = block_excl_scan(cnt, excl);
  if (threadIdx.x == 0) {
    p.run_count[s] = total;
    p.row_blocks[s] = nb;
  }
}

__global__ void __launch_bounds__(kThreads) gather_scan_kernel(const GatherParams p) {
  __shared__ int64_t carry_runs, carry_blocks;
  if (threadIdx.x == 0) carry_runs = carry_blocks = 0;
  __syncthreads();
  for (int base = 0; base < p.S; base += kThreads) {
    const int s = base + threadIdx.x;
    const int rc = s < p.S ? p.run_count[s] : 0;
    const int rb = s < p.S ? max(p.row_blocks[s], 0) : 0;
    int er, eb;
    const int tr = block_excl_scan(rc, er);
    const int tb = block_excl_scan(rb, eb);
    if (s < p.S) {
      p.run_off[s] = (int32_t)(carry_runs + er);
      p.row_bstart[s] = carry_blocks + eb;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      carry_runs += tr;
      carry_blocks += tb;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    p.run_off[p.S] = (int32_t)carry_runs;
    p.row_bstart[p.S] = carry_blocks;
    p.totals[0] = carry_runs;
    p.totals[1] = carry_blocks;
  }
}

__global__ void __launch_bounds__(kThreads) gather_emit_kernel(const GatherParams p) {
  const int s = blockIdx.x;
  const int nb = p.row_blocks[s];
  if (nb <= 0) return;
  const int32_t *row = p.block_table + (size_t)s * p.max_blocks;
  const int base = p.run_off[s];
  int idx0 = 0;
  for (int j0 = 0; j0 < nb; j0 += kThreads) {
    const int j = j0 + threadIdx.x;
    int st = 0, src = -1;
    if (j < nb) {
      st = run_start(row, j, p.num_phys);
      src = row[j];
      if (!valid_block(src, p.num_phys)) {
        atomicOr(p.status, KVX_DEV_BAD_BLOCK);
        src = -1;
      }
    }
    int excl;
    const int tot = block_excl_scan(st, excl);
    if (st) p.runs[base + idx0 + excl] = make_int4(src, s, j, 0);
    idx0 += tot;
  }
  __syncthreads();
  const int cnt = p.run_count[s];
  for (int r = threadIdx.x; r < cnt; r += kThreads) {
    const int j = p.runs[base + r].z;
    const int next = r + 1 < cnt ? p.runs[base + r + 1].z : nb;
    p.runs[base + r].w = next - j;
    p.run_bstart[base + r] = p.row_bstart[s] + j;
  }
}

__device__ __forceinline__ void copy_span(const uint8_t *src, uint8_t *dst,
                                          int64_t bytes) {
  constexpr int U = 8;
  const int64_t nv = bytes >> 4;
  const uint4 *s = reinterpret_cast<const uint4 *>(src);
  uint4 *d = reinterpret_cast<uint4 *>(dst);
  for (int64_t b0 = 0; b0 < nv; b0 += (int64_t)kThreads * U) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = b0 + u * kThreads + threadIdx.x;
      if (i < nv) v[u] = __ldcs(s + i);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = b0 + u * kThreads + threadIdx.x;
      if (i < nv) __stcs(d + i, v[u]);
    }
  }
}

__global__ void __launch_bounds__(kThreads) gather_copy_kernel(const GatherParams p) {
  const int64_t total = p.totals[1], nruns = p.totals[0];
  if (total <= 0 || nruns <= 0) return;
  const int64_t lo = total * blockIdx.x / gridDim.x;
  const int64_t hi = total * (blockIdx.x + 1) / gridDim.x;
  if (lo >= hi) return;
  int64_t a = 0, z = nruns - 1;  // last run whose first block is <= lo
  while (a < z) {
    const int64_t mid = (a + z + 1) >> 1;
    if (p.run_bstart[mid] <= lo)
      a = mid;
    else
      z = mid - 1;
  }
  int64_t r = a;
  int4 d = p.runs[r];
  int64_t gb = p.run_bstart[r];
  const int64_t bb = p.block_bytes;
  for (int64_t g = lo; g < hi;) {
    int4 dn = d;
    int64_t gbn = gb;
    if (r + 1 < nruns) {  // prefetch the next descriptor while copying
      dn = p.runs[r + 1];
      gbn = p.run_bstart[r + 1];
    }
    const int64_t off = g - gb;
    const int64_t n = min((int64_t)d.w - off, hi - g);
    if (d.x >= 0) {
      for (int t = 0; t < p.num_tensors; ++t)
        copy_span((const uint8_t *)p.pools[t] + ((int64_t)d.x + off) * bb,
                  (uint8_t *)p.stagings[t] + (int64_t)d.y * p.row_bytes + ((int64_t)d.z + off) * bb,
                  n * bb);
    }
    g += n;
    if (g >= gb + d.w) {
      ++r;
      d = dn;
      gb = gbn;
    }
  }
}

__global__ void __launch_bounds__(kThreads) gather_tail_kernel(const GatherParams p) {
  const int s = blockIdx.x;
  const int nb = p.row_blocks[s];
  if (nb < 0) return;
  const int64_t from = (int64_t)nb * p.block_bytes;
  const int64_t nv = (p.row_bytes - from) >> 4;
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  for (int t = 0; t < p.num_tensors; ++t) {
    uint4 *d = reinterpret_cast<uint4 *>((uint8_t *)p.stagings[t] + (int64_t)s * p.row_bytes + from);
    for (int64_t i = (int64_t)blockIdx.y * kThreads + threadIdx.x; i < nv;
         i += (int64_t)gridDim.y * kThreads)
      __stcs(d + i, z);
  }
}

int sm_count_cached() {
  static int sms[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 132;
  if (!sms[dev]) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
      v = 132;
    sms[dev] = v;
  }
  return sms[dev];
}

}  // namespace

GatherWs gather_ws_layout(int S, int max_blocks) {
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  GatherWs w;
  w.run_count = KVX_WS_HEADER_BYTES;
  w.row_blocks = al(w.run_count + 4 * (size_t)S);
  w.run_off = al(w.row_blocks + 4 * (size_t)S);
  w.row_bstart = al(w.run_off + 4 * ((size_t)S + 1));
  w.runs = al(w.row_bstart + 8 * ((size_t)S + 1));
  const size_t cap = std::max<size_t>((size_t)S * (size_t)max_blocks, 1);
  w.run_bstart = al(w.runs + 16 * cap);
  w.total = al(w.run_bstart + 8 * cap);
  return w;
}

cudaError_t launch_gather(const GatherParams &p, cudaStream_t st) {
  if (p.S <= 0) return cudaSuccess;
  gather_count_kernel<<<p.S, kThreads, 0, st>>>(p);
  gather_scan_kernel<<<1, kThreads, 0, st>>>(p);
  gather_emit_kernel<<<p.S, kThreads, 0, st>>>(p);
  gather_copy_kernel<<<8 * sm_count_cached(), kThreads, 0, st>>>(p);
  if (p.flags & KVX_ZERO_TAIL) gather_tail_kernel<<<dim3(p.S, 8), kThreads, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace kvx

// ---------------------------------------------------------------------------
// Allocation-free variant of the gather.
//
// Some callers cannot call cudaMalloc: code that runs inside a host callback
// or a custom allocator's own paths, runtimes that hand out only their own
// pre-planned device memory, or processes that forbid allocation after
// start-up so their memory footprint stays fixed. For them the gather's
// scratch memory (block-table runs, prefix sums, the status word) lives in
// this file-scope device array instead of a caller workspace. Every GPU that
// loads the library holds it until the process exits.
#define KVX_GATHER_STATIC_SCRATCH_BYTES KVX_GATHER_NOALLOC_SCRATCH_BYTES

namespace kvx {
namespace {

static __device__ __align__(256) unsigned char g_gather_scratch[KVX_GATHER_STATIC_SCRATCH_BYTES];

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

// Process-unique id of the CUDA context current on this thread, or 0 when
// there is none yet (or the driver cannot tell).
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, []() {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = (CtxGetCurrentFn)f;
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = (CtxGetIdFn)f;
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of g_gather_scratch in the current device's context. The
// array's host-side name is only a stand-in, not a device address, so the
// address is looked up with cudaGetSymbolAddress the first time a context
// of the device calls, and again whenever the current context is not the one
// the cached address belongs to (a device reset destroys the context, and
// the array may land elsewhere in the next one). Returns nullptr and sets
// *err if the lookup fails.
void *static_scratch(cudaError_t *err) {
  static std::mutex mu;
  static void *addr[64] = {nullptr};
  static unsigned long long ctx_of[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) {
    *err = e != cudaSuccess ? e : cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  const unsigned long long ctx = current_context_id();
  if (!addr[dev] || ctx == 0 || ctx != ctx_of[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_gather_scratch);
    if (e != cudaSuccess) {
      *err = e;
      return nullptr;
    }
    addr[dev] = p;
    ctx_of[dev] = current_context_id();  // the lookup made the context current
  }
  *err = cudaSuccess;
  return addr[dev];
}

}  // namespace
}  // namespace kvx

extern "C" int kvx_gather_coalesce_noalloc(
    const int32_t *block_table, const int32_t *num_blocks, int32_t S,
    int32_t max_blocks, int32_t num_tensors, const void *const *pools,
    int64_t num_phys_blocks, int64_t block_bytes, void *const *stagings,
    int64_t staging_row_bytes, int32_t flags, uint32_t *status, void *stream) {
  using namespace kvx;
  if (!block_table || !num_blocks || !pools || !stagings) return KVX_EINVAL;
  if (S < 0 || max_blocks < 0 || num_tensors < 1 || num_tensors > KVX_MAX_GATHER_TENSORS)
    return KVX_EINVAL;
  if (num_phys_blocks < 1 || block_bytes < 16 || block_bytes % 16 != 0 ||
      staging_row_bytes < 0 || staging_row_bytes % 16 != 0)
    return KVX_EINVAL;
  if (flags & ~KVX_ZERO_TAIL) return KVX_EINVAL;
  if (status && ((uintptr_t)status % 4) != 0) return KVX_EINVAL;
  const GatherWs w = gather_ws_layout(S, max_blocks);
  if (w.total > KVX_GATHER_STATIC_SCRATCH_BYTES) return KVX_ESCRATCH;
  GatherParams p;
  memset(&p, 0, sizeof(p));
  for (int t = 0; t < num_tensors; ++t) {
    if (!pools[t] || !stagings[t] || ((uintptr_t)pools[t] % 16) != 0 ||
        ((uintptr_t)stagings[t] % 16) != 0)
      return KVX_EINVAL;
    p.pools[t] = pools[t];
    p.stagings[t] = stagings[t];
  }
  cudaError_t e = cudaSuccess;
  char *ws = (char *)static_scratch(&e);
  if (!ws) return set_cuda_error(e);
  cudaStream_t st = (cudaStream_t)stream;
  // The array keeps the previous call's contents: clear the header (status
  // word and totals) that the kernels accumulate into.
  e = cudaMemsetAsync(ws, 0, KVX_WS_HEADER_BYTES, st);
  if (e != cudaSuccess) return set_cuda_error(e);
  p.block_table = block_table;
  p.num_blocks = num_blocks;
  p.status = status ? status : (uint32_t *)ws;
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
  e = launch_gather(p, st);
  if (e != cudaSuccess) return set_cuda_error(e);
  return KVX_OK;
}
