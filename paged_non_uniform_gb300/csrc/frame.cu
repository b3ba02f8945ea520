// frame.cu -- KV-RM block pager and Frame commit.
//
// "KV-RM" (Fig. 2, Fig. 3): the logical KV history of every sequence maps to
// physical blocks through a block pager; runtime variability (lengths that
// differ, sequences that end, histories that fragment) is expressed as
// mapping edits -- Alias, Trim, Reserve -- and sealed once per decode step by
// a Frame commit that swaps a shadow descriptor in as the active one. The
// descriptor is what the coalesced gather reads: block_table [S][max_blocks]
// and num_blocks [S].
//
// Host side (this file, plain C++): the edited view, per-block reference
// counts, and a free-block index (a segment tree over 64-block bitmap words
// holding, per node, the free prefix, suffix and longest free run) that
// answers "lowest run of c free blocks" and "lowest free block" in
// O(log(N/64)) plus one word scan. Every edited table entry and row is
// stamped with the frame it changed in.
//
// Device side: two descriptors (active, shadow). A commit writes, as one
// array of (index, value) records in mapped pinned host memory, every entry
// and row length that changed in this frame or the one before -- the shadow
// was last current two frames ago -- and one small kernel reads them in
// place and scatters them into the shadow, which then becomes active. A
// commit is one launch, or nothing when no entry changed in two frames.
#include <cuda_runtime.h>

#include <algorithm>
#include <chrono>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "kvx.h"
#include "kvx_internal.h"

namespace kvx {
namespace {

constexpr int kApplyThreads = 256;

// Records [0, ne) set block_table[rec.x] = rec.y; records [ne, ne + nr) set
// num_blocks[rec.x] = rec.y. The records live in mapped pinned host memory
// (plain loads). Indices are built by the host in range; the
// checks only keep a damaged record list from writing outside the buffers.
__global__ void __launch_bounds__(kApplyThreads)
    frame_apply_kernel(int32_t *__restrict__ bt, int32_t *__restrict__ nb,
                       const int2 *rec, int32_t ne, int32_t nr, int64_t bt_len,
                       int32_t S) {
  const int64_t i = (int64_t)blockIdx.x * kApplyThreads + threadIdx.x;
  if (i >= (int64_t)ne + nr) return;
  const int2 r = rec[i];
  if (i < ne) {
    if (r.x >= 0 && r.x < bt_len) bt[r.x] = r.y;
  } else {
    if (r.x >= 0 && r.x < S) nb[r.x] = r.y;
  }
}

// Free-block index. Leaf w covers blocks [64w, 64w+64); bit i set = block
// 64w+i free (bits past N stay clear).
class FreeIndex {
 public:
  bool init(int32_t N) {
    N_ = N;
    words_ = (N + 63) / 64;
    leaves_ = 1;
    while (leaves_ < words_) leaves_ <<= 1;
    try {
      bits_.assign(leaves_, 0ull);
      pref_.assign(2 * leaves_, 0);
      suf_.assign(2 * leaves_, 0);
      best_.assign(2 * leaves_, 0);
      len_.assign(2 * leaves_, 0);
    } catch (const std::bad_alloc &) {
      return false;
    }
    for (int32_t w = 0; w < words_; ++w) {
      const int32_t n = std::min(64, N - 64 * w);
      bits_[w] = n == 64 ? ~0ull : ((1ull << n) - 1ull);
    }
    for (int32_t w = 0; w < leaves_; ++w) leaf(w);
    for (int32_t v = leaves_ - 1; v >= 1; --v) pull(v);
    free_ = N;
    return true;
  }
  int64_t free_count() const { return free_; }
  void set(int32_t p, bool fr) {
    const uint64_t m = 1ull << (p & 63);
    uint64_t &w = bits_[p >> 6];
    if (((w & m) != 0) == fr) return;
    w = fr ? (w | m) : (w & ~m);
    free_ += fr ? 1 : -1;
    int32_t v = leaves_ + (p >> 6);
    leaf(p >> 6);
    for (v >>= 1; v >= 1; v >>= 1) pull(v);
  }
  // Lowest p with [p, p+c) all free, or -1.
  int64_t find_run(int32_t c) const {
    if (c <= 0 || best_[1] < c) return -1;
    int32_t v = 1;
    int64_t start = 0;
    while (v < leaves_) {
      const int32_t l = 2 * v, r = 2 * v + 1;
      if (best_[l] >= c) {
        v = l;
      } else if (suf_[l] + pref_[r] >= c) {
        return start + len_[l] - suf_[l];
      } else {
        start += len_[l];
        v = r;
      }
    }
    // inside one word: lowest start of c consecutive set bits
    const uint64_t x = bits_[v - leaves_];
    int32_t run = 0;
    for (int i = 0; i < 64; ++i) {
      run = ((x >> i) & 1ull) ? run + 1 : 0;
      if (run == c) return start + i - c + 1;
    }
    return -1;  // unreachable: best >= c
  }

 private:
  void leaf(int32_t w) {
    const uint64_t x = bits_[w];
    const int32_t v = leaves_ + w;
    len_[v] = 64;
    pref_[v] = x == ~0ull ? 64 : __builtin_ctzll(~x);
    suf_[v] = x == ~0ull ? 64 : __builtin_clzll(~x);
    int32_t b = 0;
    for (uint64_t y = x; y; y &= y >> 1) ++b;
    best_[v] = b;
  }
  void pull(int32_t v) {
    const int32_t l = 2 * v, r = 2 * v + 1;
    len_[v] = len_[l] + len_[r];
    pref_[v] = pref_[l] == len_[l] ? len_[l] + pref_[r] : pref_[l];
    suf_[v] = suf_[r] == len_[r] ? len_[r] + suf_[l] : suf_[r];
    best_[v] = std::max(std::max(best_[l], best_[r]), suf_[l] + pref_[r]);
  }
  int32_t N_ = 0, words_ = 0, leaves_ = 1;
  int64_t free_ = 0;
  std::vector<uint64_t> bits_;
  std::vector<int32_t> pref_, suf_, best_, len_;
};

}  // namespace
}  // namespace kvx

using namespace kvx;

struct kvx_frame {
  int32_t S = 0, M = 0, N = 0;
  std::vector<int32_t> table;  // [S][M], -1 past nb
  std::vector<int32_t> nb;     // [S]
  std::vector<int32_t> rc;     // [N]
  FreeIndex fi;
  // dirty tracking: stamp = frame in which the entry / row last changed
  int64_t frame = 0;  // number of the frame being edited (= commits so far)
  std::vector<int64_t> entry_stamp, row_stamp;
  std::vector<int32_t> cur_entries, prev_entries, cur_rows, prev_rows;
  std::vector<int32_t> scratch;  // Alias source snapshot
  // device side (allocated on first use)
  bool dev_ready = false;
  int32_t *d_bt[2] = {nullptr, nullptr};
  int32_t *d_nb[2] = {nullptr, nullptr};
  int active = 0;
  int2 *h_rec[2] = {nullptr, nullptr};  // pinned, mapped: the apply kernel reads them in place
  int2 *d_rec[2] = {nullptr, nullptr};  // device address of h_rec
  int64_t rec_cap[2] = {0, 0};
  cudaEvent_t ev[2] = {nullptr, nullptr};
  bool ev_used[2] = {false, false};
  // stats
  int64_t last_records = 0, last_bytes = 0, launches = 0, wait_ns = 0;

  void touch_entry(int64_t e) {
    if (entry_stamp[e] != frame) {
      entry_stamp[e] = frame;
      cur_entries.push_back((int32_t)e);
    }
  }
  void touch_row(int32_t s) {
    if (row_stamp[s] != frame) {
      row_stamp[s] = frame;
      cur_rows.push_back(s);
    }
  }
  void release(int32_t p) {
    if (--rc[p] == 0) fi.set(p, true);
  }
  void acquire(int32_t p) {
    if (rc[p]++ == 0) fi.set(p, false);
  }
  int ensure_device();
  void free_device();
};

int kvx_frame::ensure_device() {
  if (dev_ready) return KVX_OK;
  const size_t bt_bytes = sizeof(int32_t) * (size_t)S * (size_t)M;
  cudaError_t e = cudaSuccess;
  for (int i = 0; i < 2 && e == cudaSuccess; ++i) {
    e = cudaMalloc(&d_bt[i], bt_bytes);
    if (e == cudaSuccess) e = cudaMalloc(&d_nb[i], sizeof(int32_t) * (size_t)S);
    if (e == cudaSuccess) e = cudaMemset(d_bt[i], 0xff, bt_bytes);
    if (e == cudaSuccess) e = cudaMemset(d_nb[i], 0, sizeof(int32_t) * (size_t)S);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming);
  }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    free_device();
    return set_cuda_error(e);
  }
  dev_ready = true;
  return KVX_OK;
}

void kvx_frame::free_device() {
  for (int i = 0; i < 2; ++i) {
    if (ev[i]) {
      if (ev_used[i]) cudaEventSynchronize(ev[i]);
      cudaEventDestroy(ev[i]);
    }
    if (d_bt[i]) cudaFree(d_bt[i]);
    if (d_nb[i]) cudaFree(d_nb[i]);
    if (h_rec[i]) cudaFreeHost(h_rec[i]);
    ev[i] = nullptr;
    d_bt[i] = d_nb[i] = nullptr;
    d_rec[i] = nullptr;
    h_rec[i] = nullptr;
    rec_cap[i] = 0;
    ev_used[i] = false;
  }
  dev_ready = false;
}

extern "C" int kvx_frame_create(int32_t S, int32_t max_blocks, int32_t num_phys_blocks,
                                kvx_frame **out) {
  if (!out) return KVX_EINVAL;
  *out = nullptr;
  if (S < 1 || max_blocks < 1 || num_phys_blocks < 1) return KVX_EINVAL;
  if ((int64_t)S * max_blocks + S > INT32_MAX) return KVX_ERANGE;
  kvx_frame *f = new (std::nothrow) kvx_frame;
  if (!f) return KVX_ENOMEM;
  f->S = S;
  f->M = max_blocks;
  f->N = num_phys_blocks;
  try {
    f->table.assign((size_t)S * max_blocks, -1);
    f->nb.assign(S, 0);
    f->rc.assign(num_phys_blocks, 0);
    f->entry_stamp.assign((size_t)S * max_blocks, -1);
    f->row_stamp.assign(S, -1);
  } catch (const std::bad_alloc &) {
    delete f;
    return KVX_ENOMEM;
  }
  if (!f->fi.init(num_phys_blocks)) {
    delete f;
    return KVX_ENOMEM;
  }
  *out = f;
  return KVX_OK;
}

extern "C" int kvx_frame_destroy(kvx_frame *f) {
  if (!f) return KVX_EINVAL;
  f->free_device();
  delete f;
  return KVX_OK;
}

extern "C" int kvx_frame_reserve(kvx_frame *f, int32_t seq, int32_t count, int32_t *ids) {
  if (!f || seq < 0 || seq >= f->S || count < 0) return KVX_EINVAL;
  if ((int64_t)f->nb[seq] + count > f->M) return KVX_ERANGE;
  if (count > f->fi.free_count()) return KVX_ENOBLOCKS;
  if (count == 0) return KVX_OK;
  int32_t *row = f->table.data() + (size_t)seq * f->M;
  const int32_t base = f->nb[seq];
  const int64_t start = f->fi.find_run(count);
  for (int32_t i = 0; i < count; ++i) {
    const int32_t p = start >= 0 ? (int32_t)(start + i) : (int32_t)f->fi.find_run(1);
    f->acquire(p);
    row[base + i] = p;
    f->touch_entry((int64_t)seq * f->M + base + i);
    if (ids) ids[i] = p;
  }
  f->nb[seq] = base + count;
  f->touch_row(seq);
  return KVX_OK;
}

extern "C" int kvx_frame_alias(kvx_frame *f, int32_t dst, int32_t dst_block, int32_t src,
                               int32_t src_block, int32_t count) {
  if (!f || dst < 0 || dst >= f->S || src < 0 || src >= f->S || count < 0) return KVX_EINVAL;
  if (src_block < 0 || (int64_t)src_block + count > f->nb[src]) return KVX_ERANGE;
  if (dst_block < 0 || dst_block > f->nb[dst] || (int64_t)dst_block + count > f->M)
    return KVX_ERANGE;
  if (count == 0) return KVX_OK;
  const int32_t *srow = f->table.data() + (size_t)src * f->M;
  int32_t *drow = f->table.data() + (size_t)dst * f->M;
  f->scratch.assign(srow + src_block, srow + src_block + count);
  // take the new references before dropping the old ones, so a block that
  // stays referenced never passes through the free index
  for (int32_t i = 0; i < count; ++i) f->acquire(f->scratch[i]);
  for (int32_t i = 0; i < count; ++i) {
    const int32_t j = dst_block + i;
    if (j < f->nb[dst]) f->release(drow[j]);
    drow[j] = f->scratch[i];
    f->touch_entry((int64_t)dst * f->M + j);
  }
  if (dst_block + count > f->nb[dst]) {
    f->nb[dst] = dst_block + count;
    f->touch_row(dst);
  }
  return KVX_OK;
}

extern "C" int kvx_frame_trim(kvx_frame *f, int32_t seq, int32_t begin_block,
                              int32_t end_block) {
  if (!f || seq < 0 || seq >= f->S) return KVX_EINVAL;
  if (begin_block < 0 || begin_block > end_block || end_block > f->nb[seq]) return KVX_ERANGE;
  int32_t *row = f->table.data() + (size_t)seq * f->M;
  const int32_t n = f->nb[seq];
  for (int32_t j = 0; j < begin_block; ++j) f->release(row[j]);
  for (int32_t j = end_block; j < n; ++j) f->release(row[j]);
  const int32_t keep = end_block - begin_block;
  if (begin_block > 0) {
    for (int32_t j = 0; j < keep; ++j) {
      row[j] = row[begin_block + j];
      f->touch_entry((int64_t)seq * f->M + j);
    }
  }
  for (int32_t j = keep; j < n; ++j) {
    row[j] = -1;
    f->touch_entry((int64_t)seq * f->M + j);
  }
  if (keep != n) {
    f->nb[seq] = keep;
    f->touch_row(seq);
  }
  return KVX_OK;
}

extern "C" int kvx_frame_edit(kvx_frame *f, const int32_t *ops, int32_t n, int32_t *status,
                              int32_t *ids, int64_t ids_cap, int64_t *ids_written) {
  if (!f || n < 0 || (n > 0 && !ops) || ids_cap < 0) return KVX_EINVAL;
  int first = KVX_OK;
  int64_t written = 0;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t *o = ops + 6 * (size_t)i;
    int rc;
    switch (o[0]) {
      case KVX_EDIT_RESERVE:
        if (ids && o[2] > 0 && written + o[2] > ids_cap) {
          rc = KVX_ERANGE;  // no room for its ids: the edit is not applied
        } else {
          rc = kvx_frame_reserve(f, o[1], o[2], ids ? ids + written : nullptr);
          if (rc == KVX_OK && ids) written += o[2];
        }
        break;
      case KVX_EDIT_ALIAS: rc = kvx_frame_alias(f, o[1], o[2], o[3], o[4], o[5]); break;
      case KVX_EDIT_TRIM: rc = kvx_frame_trim(f, o[1], o[2], o[3]); break;
      default: rc = KVX_EINVAL;
    }
    if (status) status[i] = rc;
    if (rc != KVX_OK && first == KVX_OK) first = rc;
  }
  if (ids_written) *ids_written = written;
  return first;
}

extern "C" int kvx_frame_commit(kvx_frame *f, void *stream) {
  if (!f) return KVX_EINVAL;
  int rc = f->ensure_device();
  if (rc != KVX_OK) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  const int slot = (int)(f->frame & 1);
  // entries and rows changed in this frame or the previous one (the shadow
  // was last brought up to date two frames ago)
  int64_t ne = (int64_t)f->cur_entries.size(), nr = (int64_t)f->cur_rows.size();
  for (int32_t e : f->prev_entries) ne += f->entry_stamp[e] != f->frame;
  for (int32_t s : f->prev_rows) nr += f->row_stamp[s] != f->frame;
  const int64_t n = ne + nr;
  if (n > 0) {
    if (f->ev_used[slot]) {
      // the record buffers of this slot were last used two commits ago
      const auto t0 = std::chrono::steady_clock::now();
      cudaError_t e = cudaEventSynchronize(f->ev[slot]);
      f->wait_ns += std::chrono::duration_cast<std::chrono::nanoseconds>(
                        std::chrono::steady_clock::now() - t0)
                        .count();
      if (e != cudaSuccess) return set_cuda_error(e);
    }
    if (f->rec_cap[slot] < n) {
      int64_t cap = std::max<int64_t>(4096, f->rec_cap[slot]);
      while (cap < n) cap *= 2;
      if (f->h_rec[slot]) cudaFreeHost(f->h_rec[slot]);
      f->d_rec[slot] = nullptr;
      f->h_rec[slot] = nullptr;
      f->rec_cap[slot] = 0;
      void *hp = nullptr, *dp = nullptr;
      cudaError_t e = cudaHostAlloc(&hp, sizeof(int2) * (size_t)cap, cudaHostAllocMapped);
      if (e == cudaSuccess) {
        f->h_rec[slot] = (int2 *)hp;
        e = cudaHostGetDevicePointer(&dp, hp, 0);
      }
      if (e != cudaSuccess) return set_cuda_error(e);
      f->d_rec[slot] = (int2 *)dp;
      f->rec_cap[slot] = cap;
    }
    int2 *h = f->h_rec[slot];
    int64_t k = 0;
    for (int32_t e : f->cur_entries) h[k++] = make_int2(e, f->table[e]);
    for (int32_t e : f->prev_entries)
      if (f->entry_stamp[e] != f->frame) h[k++] = make_int2(e, f->table[e]);
    for (int32_t s : f->cur_rows) h[k++] = make_int2(s, f->nb[s]);
    for (int32_t s : f->prev_rows)
      if (f->row_stamp[s] != f->frame) h[k++] = make_int2(s, f->nb[s]);
    const int sh = 1 - f->active;
    const int64_t blocks = (n + kApplyThreads - 1) / kApplyThreads;
    frame_apply_kernel<<<(unsigned)blocks, kApplyThreads, 0, st>>>(
        f->d_bt[sh], f->d_nb[sh], f->d_rec[slot], (int32_t)ne, (int32_t)nr,
        (int64_t)f->S * f->M, f->S);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaEventRecord(f->ev[slot], st);
    if (e != cudaSuccess) return set_cuda_error(e);
    f->ev_used[slot] = true;
    f->launches += 1;
  }
  f->active = 1 - f->active;
  f->last_records = n;
  f->last_bytes = n * (int64_t)sizeof(int2);
  f->prev_entries.swap(f->cur_entries);
  f->cur_entries.clear();
  f->prev_rows.swap(f->cur_rows);
  f->cur_rows.clear();
  f->frame += 1;
  return KVX_OK;
}

extern "C" int kvx_frame_active(kvx_frame *f, const int32_t **block_table,
                                const int32_t **num_blocks) {
  if (!f || !block_table || !num_blocks) return KVX_EINVAL;
  int rc = f->ensure_device();
  if (rc != KVX_OK) return rc;
  *block_table = f->d_bt[f->active];
  *num_blocks = f->d_nb[f->active];
  return KVX_OK;
}

extern "C" int kvx_frame_view(const kvx_frame *f, int32_t *block_table, int32_t *num_blocks,
                              int32_t *refcount) {
  if (!f) return KVX_EINVAL;
  if (block_table) std::memcpy(block_table, f->table.data(), sizeof(int32_t) * f->table.size());
  if (num_blocks) std::memcpy(num_blocks, f->nb.data(), sizeof(int32_t) * f->nb.size());
  if (refcount) std::memcpy(refcount, f->rc.data(), sizeof(int32_t) * f->rc.size());
  return KVX_OK;
}

extern "C" int kvx_frame_get_stats(const kvx_frame *f, kvx_frame_stats *out) {
  if (!f || !out) return KVX_EINVAL;
  out->commits = f->frame;
  out->free_blocks = f->fi.free_count();
  out->pending_entries = (int64_t)f->cur_entries.size();
  out->pending_rows = (int64_t)f->cur_rows.size();
  out->last_records = f->last_records;
  out->last_bytes = f->last_bytes;
  out->launches = f->launches;
  out->wait_ns = f->wait_ns;
  return KVX_OK;
}
