/*
 * kvx.h -- C ABI of the kvx library: decode-step attention over a paged KV
 * cache with non-uniform per-head budgets, the coalesced KV gather and the
 * block pager behind it, and kept-set selection for sparse decode.
 *
 * Sources of the operations:
 *  - "Tangram: Unlocking Non-Uniform KV Cache for Efficient Multi-turn LLM
 *    Serving": static per-head budgets (Deterministic Budget Allocation),
 *    head-group page tables (Head Group Page, Fig. 8), and a work split
 *    computed ahead of time from the static budgets (AOT Load Balancing,
 *    Figs. 4(c), 5 and 13).
 *  - "KV-RM: Regularizing KV-Cache Movement for Static-Graph LLM Serving":
 *    descriptor merging of fragmented block mappings into a few large
 *    transfers that fill a fixed-shape staging buffer (Figs. 2 and 3), and
 *    mapping edits sealed by a Frame commit (Fig. 3).
 *  - "KVDrive": decode over each head's top-K critical KV entries (Fig. 7,
 *    Fig. 16).
 *
 * Conventions for every entry point:
 *  - Every function returns an int status: KVX_OK (0) or a negative code
 *    (kvx_status_string() names it). Nothing throws across the ABI.
 *  - The caller owns all device memory (inputs, outputs, workspaces) and all
 *    host arrays passed in. The library owns only its opaque objects: the
 *    plan (host arrays plus a device copy made by kvx_plan_upload, freed by
 *    kvx_plan_destroy) and the frame (host view, two device descriptors and
 *    record buffers, freed by kvx_frame_destroy).
 *  - Device calls are asynchronous on the stream passed as `void *stream`
 *    (a cudaStream_t; NULL = the legacy default stream). They never
 *    synchronise and never allocate device memory on the hot path (a frame
 *    allocates its descriptors on first use). Argument errors are found on
 *    the host, before anything is launched.
 *  - Errors found on the device (a page id outside its pool, a budget that
 *    disagrees with the plan, a block id outside the pool, a wait that ran
 *    out) set bits in a status word at the start of the caller's workspace
 *    (KVX_DEV_* below); the affected reads are replaced by zeros and the
 *    kernel still terminates. The word is sticky: kvx_workspace_status reads
 *    it, kvx_workspace_clear resets it. A fresh workspace must be zero-filled
 *    (kvx_workspace_clear over its whole size) once before first use, and
 *    again after a call that reported KVX_DEV_TIMEOUT.
 *  - All layouts are dense row-major C arrays, outermost index first.
 */
#ifndef KVX_H
#define KVX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---------------------------------------------------- */
#define KVX_OK 0
#define KVX_EINVAL (-1)       /* a null pointer, bad size or inconsistent argument */
#define KVX_ERANGE (-2)       /* an index or length outside its declared range */
#define KVX_ENOMEM (-3)       /* host allocation failed */
#define KVX_ECUDA (-4)        /* a CUDA runtime call failed; see kvx_last_cuda_error */
#define KVX_EUNSUPPORTED (-5) /* head_dim / page size / dtype / GQA combination */
#define KVX_ESTATE (-6)       /* plan used before kvx_plan_upload */
#define KVX_ESCRATCH (-7)     /* kvx_gather_coalesce_noalloc: problem too large for its static scratch */
#define KVX_ENOBLOCKS (-8)    /* kvx_frame_reserve: fewer free physical blocks than asked */

/* ---- device status bits (workspace status word) ---------------------- */
#define KVX_DEV_BAD_PAGE 1u    /* a page-table entry outside [0, pool_pages) */
#define KVX_DEV_BAD_BUDGET 2u  /* min(seq_len, head_budget) differs from the plan */
#define KVX_DEV_TIMEOUT 4u     /* a pipeline wait gave up after its time limit */
#define KVX_DEV_BAD_BLOCK 8u   /* a block-table entry outside [0, num_phys_blocks);
                                  a kept index outside [0, Lmax) (packing,
                                  kept-row attention) */
#define KVX_DEV_BAD_LENGTH 16u /* num_blocks[s] outside [0, max_blocks] or the row;
                                  a selection seq_len outside [0, Lmax] */

/* ---- element types --------------------------------------------------- */
#define KVX_F32 0
#define KVX_BF16 1

/* ---- work-split policies (kvx_plan_create) ---------------------------- */
/* Ahead-of-time balanced split (Tangram, AOT Load Balancing): the kept tokens
 * of all heads are laid end to end and cut into num_ctas spans of equal cost;
 * a head cut across spans is split into partials merged by log-sum-exp
 * through the workspace. */
#define KVX_PLAN_BALANCED 0
/* One thread block per (sequence, KV head); no split (naive baseline). */
#define KVX_PLAN_PER_HEAD 1
/* Every head split into the same number of equal pieces, sized so the grid
 * covers the GPU twice; one block per piece (the uniform split of Tangram
 * Fig. 4(c), whose stragglers the balanced plan removes). */
#define KVX_PLAN_UNIFORM 2
/* Cluster layout (tensor-core kernel only), thread-block clusters of 2, 4 or 8
 * blocks on this GPU: every head is either whole on one block or cut into
 * pieces on blocks of one cluster, at most one piece per block, run as that
 * block's last item; the pieces are merged through distributed shared memory
 * by the block of the head's first piece, with no workspace partials. The
 * cost cap per block is the smallest with which that placement fits (heads
 * placed longest first). num_ctas must be a multiple of the cluster size;
 * 0 = as many clusters as can be resident on the current device.
 * KVX_EUNSUPPORTED if no placement fits. */
#define KVX_PLAN_CLUSTER_2 3
#define KVX_PLAN_CLUSTER_4 4
#define KVX_PLAN_CLUSTER_8 5

/* ---- kernel choice ----------------------------------------------------- */
#define KVX_KERNEL_AUTO 0 /* tensor-core kernel for bf16, CUDA-core kernel for fp32 */
#define KVX_KERNEL_MMA 1  /* bf16 only: bulk-tensor loads + warp-level MMA */
#define KVX_KERNEL_SIMT 2 /* CUDA-core kernel, fp32 or bf16 */

/* ---- page layouts ------------------------------------------------------ */
/* A head-group page holds P token slots for each of the |G| heads of its
 * group, for K and (in a separate pool) for V:
 *  HEAD_MAJOR  [|G|][P][D]: the slots of one head are contiguous
 *              (Tangram's head-group page, Fig. 8(b));
 *  TOKEN_MAJOR [P][|G|][D]: the heads of one token are contiguous, the block
 *              layout of KV-RM's block pager and staging buffer (Fig. 2). */
#define KVX_LAYOUT_HEAD_MAJOR 0
#define KVX_LAYOUT_TOKEN_MAJOR 1

/* ---- gather flags ------------------------------------------------------ */
#define KVX_ZERO_TAIL 1 /* zero each staging row past its live blocks */

/* ---- limits ------------------------------------------------------------ */
#define KVX_MAX_GROUPS 16
#define KVX_MAX_KV_HEADS 64
#define KVX_MAX_GQA 8
#define KVX_MAX_GATHER_TENSORS 4
#define KVX_WS_HEADER_BYTES 256

typedef struct kvx_shape {
  int32_t B;          /* sequences in the batch */
  int32_t Hq;         /* query heads; Hq = g * Hkv, 1 <= g <= KVX_MAX_GQA */
  int32_t Hkv;        /* KV heads, <= KVX_MAX_KV_HEADS */
  int32_t D;          /* head dimension: 64 or 128 */
  int32_t page_size;  /* P, tokens per page: 8, 16, 32, 64 or 128 */
  int32_t num_groups; /* head groups, <= KVX_MAX_GROUPS */
  int32_t dtype;      /* KVX_F32 or KVX_BF16 (q, K and V share it) */
  int32_t layout;     /* page layout: KVX_LAYOUT_HEAD_MAJOR or KVX_LAYOUT_TOKEN_MAJOR */
} kvx_shape;

typedef struct kvx_plan kvx_plan;

typedef struct kvx_plan_stats {
  int32_t num_ctas;          /* thread blocks the attention kernel launches */
  int32_t num_items;         /* work items (head, token range) */
  int32_t num_slots;         /* partial results written for split heads */
  int32_t num_split_heads;   /* heads cut into more than one item */
  int32_t kernel;            /* KVX_KERNEL_MMA or KVX_KERNEL_SIMT (resolved) */
  int32_t policy;            /* KVX_PLAN_* */
  int64_t total_tokens;      /* sum of kept tokens over all heads */
  int64_t max_cta_tokens;    /* largest token load of one thread block */
  double mean_cta_tokens;    /* mean token load per thread block */
  int64_t slots_allocated;   /* token slots in allocated group pages (all heads) */
  int64_t slots_used;        /* token slots holding kept tokens (= total_tokens) */
  double plan_us;            /* host time spent building the plan */
  int32_t item_overhead;     /* tokens the balanced plan charges per item on top of
                                its tokens (the per-item cost of query load,
                                cross-warp merge and partial write) */
  int32_t cluster;           /* blocks per thread-block cluster of the launch
                                (1: no clusters, split heads merged through the
                                workspace) */
} kvx_plan_stats;

/* Text for a status code. Never NULL. */
const char *kvx_status_string(int status);

/* The cudaError_t of the last failed CUDA call in this thread (0 if none). */
int kvx_last_cuda_error(void);

/* Streaming multiprocessors of the current device (queries the driver). */
int kvx_device_sm_count(int32_t *sms);

/* ---------------------------------------------------------------------------
 * kvx_plan_create -- host only, no device work.
 *
 * Resolves the kept-token count of every head (Tangram, Deterministic Budget
 * Allocation: a static budget per head):
 *     n[b][h] = min(seq_len[b], head_budget[b*Hkv + h]),  head_budget >= 1,
 * groups the KV heads (Tangram, Fig. 8: heads with similar budgets share one
 * head-group page table) and builds the ahead-of-time work split.
 *
 *   shape        problem shape (host).
 *   head_budget  int32 [B*Hkv], tokens each (sequence, KV head) keeps (host).
 *   seq_len      int32 [B], tokens in each sequence, >= 1 (host).
 *   head_group   int32 [Hkv], group of each KV head, in [0, num_groups); every
 *                group non-empty (host). Within a group, heads take page-slot
 *                rows 0, 1, ... in ascending head order.
 *   num_ctas     thread blocks for KVX_PLAN_BALANCED and KVX_PLAN_CLUSTER_*;
 *                0 = as many as stay resident on the current device (2 per SM
 *                for the tensor-core kernel, 1 for the CUDA-core kernel);
 *                ignored by the other policies.
 *   policy       KVX_PLAN_*.   kernel  KVX_KERNEL_*.
 *   out          receives the plan (owned by the caller; kvx_plan_destroy).
 * Errors: KVX_EINVAL, KVX_EUNSUPPORTED, KVX_ENOMEM; *out is NULL on error.
 * ------------------------------------------------------------------------- */
int kvx_plan_create(const kvx_shape *shape, const int32_t *head_budget,
                    const int32_t *seq_len, const int32_t *head_group,
                    int32_t num_ctas, int32_t policy, int32_t kernel,
                    kvx_plan **out);

/* Copies the plan's work list to the device (allocates plan-owned device
 * memory; call once, outside any hot loop). Stream-ordered on `stream`. */
int kvx_plan_upload(kvx_plan *plan, void *stream);

/* Bytes of device workspace kvx_decode_attn needs with this plan: a
 * KVX_WS_HEADER_BYTES header (status word), one counter per split head and
 * the split partials. The counters return to zero at the end of every call. */
int kvx_plan_workspace_bytes(const kvx_plan *plan, size_t *bytes);

int kvx_plan_get_stats(const kvx_plan *plan, kvx_plan_stats *stats);

/* Kept-token counts n, int32 [B*Hkv] (host). */
int kvx_plan_kept(const kvx_plan *plan, int32_t *n);

/* Pages each head group needs per sequence: int32 [num_groups][B] (host),
 * pages[g][b] = ceil(max_{h in g} n[b][h] / P). A group's page table row for
 * sequence b must hold at least that many valid page ids. */
int kvx_plan_group_pages(const kvx_plan *plan, int32_t *pages);

/* The work list (host copies): items int32 [num_items][4] =
 * {b*Hkv + h, first token, end token, partial slot or -1}, and cta_off
 * int32 [num_ctas + 1]: thread block c runs items cta_off[c] .. cta_off[c+1]-1.
 * Token t of head (b,h) is the head's t-th kept token in ascending position. */
int kvx_plan_items(const kvx_plan *plan, int32_t *items, int32_t *cta_off);

/* Per-block token loads, int64 [num_ctas] (host). */
int kvx_plan_cta_tokens(const kvx_plan *plan, int64_t *tokens);

/* Token coverage of the plan (host only). The ahead-of-time split must read
 * every kept token of every head exactly once (Tangram, AOT Load Balancing,
 * Fig. 13: the static plan cuts each head's kept tokens across thread blocks;
 * the cut changes where tokens are read, never which). Fills
 *     count int32 [B*Hkv][max_n],  max_n = max(1, max over heads of n[b][h]),
 *     count[bh*max_n + t] = number of work items containing token t of head bh,
 * so a correct plan gives 1 for t < n[bh] and 0 from n[bh] on.
 * Errors: KVX_EINVAL (null argument). */
int kvx_plan_coverage(const kvx_plan *plan, int32_t *count);

/* Device coverage record (test hook; no effect unless set). dev_count is a
 * device buffer of int32 [B*Hkv][stride], stride >= max_n above, zeroed by
 * the caller. Every subsequent kvx_decode_attn with this plan adds 1 to
 * dev_count[bh*stride + t] for each kept token t of head bh at the point
 * where a consumer warp feeds it to the softmax (after its K/V data has
 * arrived; counted from what the kernel consumed, not from the plan). A
 * correct launch leaves exactly kvx_plan_coverage's array. NULL turns the
 * record off. Errors: KVX_EINVAL, KVX_ERANGE (stride too small). */
int kvx_plan_set_coverage_record(kvx_plan *plan, int32_t *dev_count, int32_t stride);

/* Optional per-block timing trace: dev_trace is a device buffer of int64
 * [num_ctas][4] = {SM id, start ns, end ns, tokens}, written by every
 * subsequent kvx_decode_attn with this plan; NULL turns it off. */
int kvx_plan_set_trace(kvx_plan *plan, int64_t *dev_trace);

/* Failure-detection test hook (no effect unless called). The tensor-core
 * kernel's thread block `block` arms the barrier of its first pipeline stage
 * but issues none of its loads, so the wait for that stage runs out after
 * wait_limit_ns (1 ms .. 10 s; every pipeline wait uses this limit, 2 s by
 * default). The call then finishes with KVX_DEV_TIMEOUT set in the workspace
 * status word; its output is undefined, the CUDA context stays usable, and the
 * workspace must be cleared before the next call. block < 0 turns the stall
 * off (the limit stays as given). Errors: KVX_EINVAL, KVX_ERANGE. */
int kvx_plan_inject_stall(kvx_plan *plan, int32_t block, uint64_t wait_limit_ns);

/* Early K/V loads (off by default; tensor-core kernel). The decode call is
 * launched as a programmatic dependent of the kernel before it on the stream,
 * and waits for that kernel on the device before it reads its inputs. With
 * enable = 1, each block's load warp reads page-table entries and K/V pages
 * before that wait: it fills its empty ring with its first stages, except a
 * stage that holds a head's newest page (the page of its last kept token),
 * and waits before anything else. q, seq_len and head_budget are still read
 * after the wait, and the L2 warm-up of short launches is skipped.
 * Precondition: if the kernel before the call lets its dependents start early
 * (programmatic dependent launch), it writes none of the page-table entries
 * or K/V pages the call reads, except each head's newest page and that page's
 * page-table entry (the load warp reads the entries again after the wait and
 * loads the newest page only then). An ordinary
 * kernel lets its dependents start only when it has completed, so any kernel
 * qualifies that does not use programmatic launch; so do the library's own
 * kernels, none of which write pages or page tables while a dependent may run.
 * enable: 0 or 1. Errors: KVX_EINVAL. */
int kvx_plan_set_early_kv(kvx_plan *plan, int32_t enable);

void kvx_plan_destroy(kvx_plan *plan);

/* ---------------------------------------------------------------------------
 * kvx_decode_attn -- one decode step of attention for one layer.
 *
 * For sequence b, query head j, KV head h = floor(j / g) (g = Hq / Hkv), over
 * the n[b][h] kept tokens t of head h:
 *     s_t = scale * <q[b][j], k_t>,   out[b][j] = sum_t softmax(s)_t * v_t.
 * (Tangram, Fig. 2: attention over each head's kept tokens; the split-K
 * partials of a cut head are merged by log-sum-exp, which leaves the result
 * unchanged up to rounding. The merge runs inside the same kernel launch, in
 * the block that finishes the head's last piece, in a fixed order.)
 *
 * Head-group page addressing (Tangram, Fig. 8(b)): head h belongs to group
 * G = head_group[h] and has row r = its rank within G. Its t-th kept token is
 * in physical page p = page_tables[G][b * page_table_stride[G] + t / P],
 * at k_pools[G] + ((p * |G| + r) * P + t % P) * D elements with the
 * head-major layout, or k_pools[G] + ((p * P + t % P) * |G| + r) * D with
 * the token-major layout (same for V).
 *
 *   plan              an uploaded plan built for these shapes and budgets.
 *   q                 [B][Hq][D] of the plan's dtype (device), 16-byte aligned.
 *   k_pools, v_pools  host arrays [num_groups] of device pointers, each a
 *                     pool of pool_pages[G] pages, [|G|][P][D] (head-major)
 *                     or [P][|G|][D] (token-major) of the plan's dtype,
 *                     16-byte aligned.
 *   pool_pages        host int64 [num_groups], pages in each pool.
 *   page_tables       host array [num_groups] of device int32 pointers, each
 *                     [B][page_table_stride[G]].
 *   page_table_stride host int32 [num_groups]; must be >= the pages the plan
 *                     says the group needs (kvx_plan_group_pages).
 *   head_budget       device int32 [B*Hkv]; seq_len device int32 [B]: checked
 *                     on the device against the plan (KVX_DEV_BAD_BUDGET).
 *   scale             score scale; 0 means 1/sqrt(D).
 *   out               device fp32 [B][Hq][D].
 *   workspace         device, >= kvx_plan_workspace_bytes, 256-byte aligned.
 * Padding slots of partly filled pages are never read into the result.
 * Launch: one kernel, as a programmatic dependent of the kernel before it on
 * the stream. It may start while that kernel drains. It reads no input but
 * the plan's device copy until that kernel has completed, except that a plan
 * of short blocks prefetches its first K/V pages into L2, which changes no
 * data. The call may be captured into a CUDA graph once the plan has made
 * one call on the device (that call sets the kernel's shared-memory limit);
 * the graph keeps the pointers, strides and scale of the captured call.
 * Errors: KVX_EINVAL, KVX_ERANGE, KVX_ESTATE, KVX_ECUDA (nothing launched on
 * argument errors).
 * ------------------------------------------------------------------------- */
int kvx_decode_attn(const kvx_plan *plan, const void *q,
                    const void *const *k_pools, const void *const *v_pools,
                    const int64_t *pool_pages,
                    const int32_t *const *page_tables,
                    const int32_t *page_table_stride,
                    const int32_t *head_budget, const int32_t *seq_len,
                    float scale, float *out, void *workspace,
                    size_t workspace_bytes, void *stream);

/* Reads the workspace status word (synchronous device-to-host copy). */
int kvx_workspace_status(const void *workspace, uint32_t *status);

/* Zeroes the first `bytes` bytes of a workspace (stream-ordered): pass the
 * whole workspace size before first use; KVX_WS_HEADER_BYTES clears only the
 * status word. bytes >= KVX_WS_HEADER_BYTES. */
int kvx_workspace_clear(void *workspace, size_t bytes, void *stream);

/* ---------------------------------------------------------------------------
 * kvx_gather_coalesce -- KV-RM movement step.
 *
 * (1) Descriptor merging (KV-RM, Fig. 3): the block table of each sequence is
 *     cut into runs, maximal stretches of logically consecutive blocks whose
 *     physical ids are consecutive; the runs are written to the workspace.
 * (2) Coalesced gather (KV-RM, abstract and Fig. 2): every run is copied as
 *     one contiguous transfer into the fixed-shape staging buffer, so that
 *     for s < S, j < num_blocks[s]:
 *         staging_t[s*row_bytes + j*block_bytes ...+block_bytes]
 *           = pools_t[block_table[s*max_blocks + j] * block_bytes ...]
 *     for every tensor t < num_tensors (e.g. K and V). Staging bytes of a row
 *     past num_blocks[s]*block_bytes are left untouched, or zeroed with
 *     KVX_ZERO_TAIL.
 *
 *   block_table   device int32 [S][max_blocks]; entries past num_blocks[s]
 *                 are ignored.
 *   num_blocks    device int32 [S], each in [0, max_blocks] with
 *                 num_blocks[s]*block_bytes <= row_bytes (else the row is
 *                 skipped and KVX_DEV_BAD_LENGTH is set).
 *   pools         host array [num_tensors] of device pointers, each
 *                 [num_phys_blocks][block_bytes] bytes, 16-byte aligned.
 *   stagings      host array [num_tensors] of device pointers, each
 *                 [S][staging_row_bytes] bytes, 16-byte aligned.
 *   block_bytes, staging_row_bytes  multiples of 16.
 *   workspace     device, >= kvx_gather_workspace_bytes(S, max_blocks).
 * Blocks with an id outside the pool are not copied (KVX_DEV_BAD_BLOCK).
 * ------------------------------------------------------------------------- */
int kvx_gather_workspace_bytes(int32_t S, int32_t max_blocks, size_t *bytes);

int kvx_gather_coalesce(const int32_t *block_table, const int32_t *num_blocks,
                        int32_t S, int32_t max_blocks, int32_t num_tensors,
                        const void *const *pools, int64_t num_phys_blocks,
                        int64_t block_bytes, void *const *stagings,
                        int64_t staging_row_bytes, int32_t flags,
                        void *workspace, size_t workspace_bytes, void *stream);

/* Reads the runs of the last kvx_gather_coalesce on this workspace
 * (synchronous): run_count int32 [S]; runs int32 [S][max_blocks][3] =
 * {first physical block, first logical block, length in blocks}. */
int kvx_gather_read_runs(const void *workspace, int32_t S, int32_t max_blocks,
                         int32_t *run_count, int32_t *runs);

/* ---------------------------------------------------------------------------
 * KV-RM block pager and Frame commit ("KV-RM", Fig. 2: block pager; Fig. 3:
 * runtime variability expressed as mapping edits Alias, Trim and Reserve,
 * sealed by a single Frame commit that swaps a shadow descriptor in as the
 * active one).
 *
 * A frame object holds, for S sequences, the logical view of each sequence:
 * a list of at most max_blocks physical block ids out of a pool of
 * num_phys_blocks. A block may appear in several views (after Alias); it is
 * free when no view names it. Edits change the host view only; a commit
 * publishes it as the device descriptor that kvx_gather_coalesce reads:
 *     block_table int32 [S][max_blocks], entries past num_blocks[s] are -1;
 *     num_blocks  int32 [S].
 * Two device descriptors are kept (active and shadow). kvx_frame_commit
 * writes the entries and lengths that changed since the shadow was last
 * current (this frame and the one before) as records in mapped pinned host
 * memory and enqueues on `stream` one kernel that reads them and writes them
 * into the shadow, then makes the shadow active. Work that reads a descriptor must be ordered before the
 * commit after the one that made it active (it becomes the shadow that
 * commit writes); on one stream this holds by construction.
 *
 * Placement: Reserve(s, c) takes the lowest-addressed run of c consecutive
 * free blocks if there is one, else the c lowest-numbered free blocks in
 * ascending order (runs keep descriptor merging effective).
 *
 * Errors: KVX_EINVAL (null frame, sequence outside [0, S), negative count),
 * KVX_ERANGE (block index or length out of range), KVX_ENOBLOCKS (fewer free
 * blocks than asked), KVX_ENOMEM (host), KVX_ECUDA. A failed edit changes
 * nothing. Device memory is allocated on first use (commit or active). One
 * frame is used by one host thread at a time.
 * ------------------------------------------------------------------------- */
typedef struct kvx_frame kvx_frame;

typedef struct {
  int64_t commits;         /* frames committed so far */
  int64_t free_blocks;     /* physical blocks no view names */
  int64_t pending_entries; /* table entries edited since the last commit */
  int64_t pending_rows;    /* view lengths changed since the last commit */
  int64_t last_records;    /* (index, value) records the last commit uploaded */
  int64_t last_bytes;      /* bytes of those records (read by the device from host memory) */
  int64_t launches;        /* apply-kernel launches so far */
  int64_t wait_ns;         /* host time commits spent waiting for the record
                              buffers of the commit before last (stream work
                              queued ahead of it) */
} kvx_frame_stats;

/* S >= 1, max_blocks >= 1, num_phys_blocks >= 1; S * max_blocks + S must fit
 * in int32 (KVX_ERANGE). All views start empty, all blocks free. */
int kvx_frame_create(int32_t S, int32_t max_blocks, int32_t num_phys_blocks,
                     kvx_frame **out);
/* Frees host and device memory; call after the work reading its descriptors. */
int kvx_frame_destroy(kvx_frame *frame);
/* Reserve: appends count new blocks to the view of seq (nb[seq] + count <=
 * max_blocks); writes their ids to ids[0..count) when ids is not NULL. */
int kvx_frame_reserve(kvx_frame *frame, int32_t seq, int32_t count, int32_t *ids);
/* Alias: view entries [dst_block, dst_block+count) of dst name the blocks
 * that entries [src_block, src_block+count) of src name (all read before
 * any is written, so overlapping ranges of one view are fine). dst_block <=
 * nb[dst]; the view of dst grows to max(nb[dst], dst_block+count) <=
 * max_blocks. Blocks no longer named become free. */
int kvx_frame_alias(kvx_frame *frame, int32_t dst, int32_t dst_block, int32_t src,
                    int32_t src_block, int32_t count);
/* Trim: seq keeps view entries [begin_block, end_block), renumbered from 0
 * (0 <= begin <= end <= nb[seq]); the others are released. Trim(s, 0, 0)
 * ends a sequence; Trim(s, k, nb) drops its k oldest blocks. */
int kvx_frame_trim(kvx_frame *frame, int32_t seq, int32_t begin_block, int32_t end_block);
/* Several edits in one call, applied in order exactly as the single-edit
 * calls would apply them: ops [n][6] int32, one of
 *     {KVX_EDIT_RESERVE, seq, count, 0, 0, 0}
 *     {KVX_EDIT_ALIAS, dst, dst_block, src, src_block, count}
 *     {KVX_EDIT_TRIM, seq, begin_block, end_block, 0, 0}
 * status [n] (may be NULL) receives each edit's status (KVX_EINVAL for an
 * unknown kind). A failed edit changes nothing and the later ones are still
 * applied. ids (may be NULL) receives the block ids of every successful
 * Reserve, concatenated in edit order; a Reserve whose ids would not fit in
 * ids_cap entries fails with KVX_ERANGE. *ids_written (may be NULL) gets the
 * number of ids written. Returns KVX_OK, or the status of the first failed
 * edit. */
#define KVX_EDIT_RESERVE 0
#define KVX_EDIT_ALIAS 1
#define KVX_EDIT_TRIM 2
int kvx_frame_edit(kvx_frame *frame, const int32_t *ops, int32_t n, int32_t *status,
                   int32_t *ids, int64_t ids_cap, int64_t *ids_written);
/* Frame commit (see above). Asynchronous on `stream`: the apply kernel reads
 * the commit's records from mapped pinned host memory, which is reused two
 * commits later, after that kernel ended. */
int kvx_frame_commit(kvx_frame *frame, void *stream);
/* Device pointers of the active descriptor (valid until the frame is
 * destroyed; their contents change with the second commit after this one). */
int kvx_frame_active(kvx_frame *frame, const int32_t **block_table,
                     const int32_t **num_blocks);
/* Host copy of the edited view (including edits not yet committed):
 * block_table [S][max_blocks], num_blocks [S], refcount [num_phys_blocks];
 * any may be NULL. */
int kvx_frame_view(const kvx_frame *frame, int32_t *block_table, int32_t *num_blocks,
                   int32_t *refcount);
int kvx_frame_get_stats(const kvx_frame *frame, kvx_frame_stats *out);

/* ---------------------------------------------------------------------------
 * kvx_select_topk -- kept-set selection for sparse long-context decode
 * ("KVDrive", Fig. 7 and Fig. 16: decode attends to the top-K critical KV
 * entries of each head; here together with a recent window).
 *
 * For sequence b and KV head h, with Q = the sum of h's g = Hq/Hkv query
 * vectors (the grouped query heads score a token by the sum of their dot
 * products):
 *     score_t = <k_t, Q>   (fp32)            for t < L_b - recent,
 *     kept    = the min(top, L_b - recent) largest scores (equal scores:
 *               lower position first), then [max(0, L_b - recent), L_b);
 *               ascending positions.
 *   keys        device bf16 [B][Hkv][Lmax][D], D = 64 or 128, 16-byte aligned;
 *               Lmax <= 262144 (KVX_EUNSUPPORTED beyond).
 *   q           device bf16 [B][Hq][D].
 *   seq_len     device int32 [B], each in [0, Lmax]; a length outside that
 *               range selects nothing for its sequence (count 0) and sets
 *               KVX_DEV_BAD_LENGTH in the workspace status word
 *               (kvx_workspace_status).
 *   kept_idx    device int32 [B*Hkv][top + recent]; entries past the count
 *               are set to -1.
 *   kept_count  device int32 [B*Hkv].
 *   workspace   device, >= kvx_select_workspace_bytes(B, Hkv, Lmax), 256-byte
 *               aligned (holds the scores, the first digit of the largest
 *               score of every 8 positions and a per-head histogram, which
 *               the call clears on `stream` first).
 * The cut is decided on fp32 scores: positions whose scores lie within fp32
 * rounding of the cut may be exchanged with respect to an exact selection.
 * Launch: a kernel that clears the histograms, a programmatic dependent of
 * the work before it on `stream` that waits for that work on the device
 * before it writes; the score pass, a programmatic dependent of it that
 * waits only before adding its counts;
 * then the cut pass, a programmatic dependent of the score pass that waits
 * for it on the device: one thread-block cluster of 4 blocks per head (this
 * GPU only). Each block reads only the score groups whose largest first digit
 * reaches the cut's bucket, and sends the bucket's keys to the cluster's
 * first block through distributed shared memory, which finds the cut there.
 * ------------------------------------------------------------------------- */
int kvx_select_workspace_bytes(int32_t B, int32_t Hkv, int32_t Lmax, size_t *bytes);

int kvx_select_topk(const void *keys, const void *q, const int32_t *seq_len,
                    int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t Lmax,
                    int32_t top, int32_t recent, int32_t *kept_idx,
                    int32_t *kept_count, void *workspace, size_t workspace_bytes,
                    void *stream);

/* ---------------------------------------------------------------------------
 * kvx_pack_kept -- compaction of kept rows into head-group pages (Tangram,
 * Fig. 8(b)). For every head (b, h) of the plan and i < n[b][h] (the plan's
 * kept count), copies row kept_idx[(b*Hkv + h) * kept_stride + i] of the
 * dense keys and values into token i of the head's pages, with the plan's
 * page layout and groups (same addressing as kvx_decode_attn).
 *   keys, values  device bf16 [B][Hkv][Lmax][D], 16-byte aligned.
 *   pools, page tables: as for kvx_decode_attn (written here).
 *   workspace     device, >= KVX_WS_HEADER_BYTES: its status word collects
 *                 KVX_DEV_BAD_BLOCK (a kept index outside [0, Lmax)) and
 *                 KVX_DEV_BAD_PAGE; such rows are not copied.
 * Errors: KVX_EINVAL, KVX_ERANGE, KVX_ESTATE, KVX_EUNSUPPORTED (fp32 plans).
 * ------------------------------------------------------------------------- */
int kvx_pack_kept(const kvx_plan *plan, const void *keys, const void *values,
                  int32_t Lmax, const int32_t *kept_idx, int32_t kept_stride,
                  void *const *k_pools, void *const *v_pools,
                  const int64_t *pool_pages, const int32_t *const *page_tables,
                  const int32_t *page_table_stride, void *workspace,
                  size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * kvx_decode_attn_kept -- decode attention straight over the kept rows of a
 * dense cache, without packing them into pages first. The result is that of
 * kvx_decode_attn over the pages kvx_pack_kept would fill from the same kept
 * lists with the same plan, bit for bit: the same items, the same stages of
 * 32 kept tokens, the same arithmetic ("KVDrive", Fig. 7: decode attends to
 * each head's selected critical entries; Tangram, Fig. 13: the plan's split).
 *   plan        bf16 plan whose kept count n[b][h] is the number of entries of
 *               head (b, h)'s kept list that it attends to (for example
 *               kvx_select_topk's kept_count, copied to the host, as the
 *               head_budget of kvx_plan_create); any page size, layout and
 *               work-split policy (pages play no part here).
 *   q, out, head_budget, seq_len, scale, workspace: as for kvx_decode_attn.
 *   keys, values  device bf16 [B][Hkv][Lmax][D], 16-byte aligned.
 *   kept_idx    device int32 [B*Hkv][kept_stride]: token i of head
 *               bh = b*Hkv + h is row kept_idx[bh*kept_stride + i] of that
 *               head's keys and values, for i < n[b][h]; any order. An index
 *               outside [0, Lmax) reads as a zero row and sets KVX_DEV_BAD_BLOCK
 *               in the workspace status word.
 * Launch: as kvx_decode_attn, except that the load warps read the kept list
 * only after the dependency wait (it usually comes from the kernel before,
 * e.g. kvx_select_topk), so kvx_plan_set_early_kv and the L2 warm-up of short
 * launches do not apply. Each load warp copies a stage's 32 rows of K and V
 * with 16-byte asynchronous copies (cp.async) that arrive on the stage's
 * barrier as they land.
 * Errors: KVX_EINVAL, KVX_ERANGE (kept_stride below the plan's largest kept
 * count), KVX_ESTATE, KVX_EUNSUPPORTED (fp32 plans, CUDA-core kernel plans),
 * KVX_ECUDA.
 * ------------------------------------------------------------------------- */
int kvx_decode_attn_kept(const kvx_plan *plan, const void *q, const void *keys,
                         const void *values, int32_t Lmax, const int32_t *kept_idx,
                         int32_t kept_stride, const int32_t *head_budget,
                         const int32_t *seq_len, float scale, float *out, void *workspace,
                         size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * kvx_gather_coalesce_noalloc -- kvx_gather_coalesce without a workspace.
 *
 * The pages have no counterpart of this entry point: it exists for callers
 * that cannot allocate device memory (code running inside host callbacks or
 * allocator paths, runtimes that only hand out pre-planned memory, processes
 * that keep a fixed device footprint after start-up). It computes exactly what
 * kvx_gather_coalesce computes, with the same arguments except the workspace:
 * its scratch (runs, prefix sums) lives in a static device array of
 * KVX_GATHER_NOALLOC_SCRATCH_BYTES (8 MiB) that every GPU loading the library
 * holds until the process exits. It allocates nothing.
 *
 *  - Size limit: the scratch must hold kvx_gather_workspace_bytes(S,
 *    max_blocks) bytes, about 24 * S * max_blocks + 32 * S (S = 256,
 *    max_blocks = 1024 fits); larger problems return KVX_ESCRATCH before
 *    anything is launched.
 *  - status: optional device uint32 (may be NULL) into which device-detected
 *    errors (KVX_DEV_BAD_BLOCK, KVX_DEV_BAD_LENGTH) are OR-ed; the caller
 *    zeroes it. With NULL they are not reported.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current, and a call looks it
 *    up again when the device's CUDA context has changed since (after
 *    cudaDeviceReset, the array may sit elsewhere in the new context). Make
 *    that first call before any stream capture. A call with S = 0 does only
 *    this set-up (plus the header clear below) and copies nothing: use it to
 *    prepare a device ahead of time.
 *  - Every call shares the one array and clears its header on `stream` first;
 *    calls whose work overlaps on the GPU (different streams, different
 *    threads) race on it and must be ordered by the caller.
 *  - Run lists are not readable afterwards (kvx_gather_read_runs needs a
 *    caller workspace).
 * ------------------------------------------------------------------------- */
#define KVX_GATHER_NOALLOC_SCRATCH_BYTES (8u << 20)
int kvx_gather_coalesce_noalloc(const int32_t *block_table,
                                const int32_t *num_blocks, int32_t S,
                                int32_t max_blocks, int32_t num_tensors,
                                const void *const *pools,
                                int64_t num_phys_blocks, int64_t block_bytes,
                                void *const *stagings,
                                int64_t staging_row_bytes, int32_t flags,
                                uint32_t *status, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* KVX_H */
