/*
 * oracle.h -- plain, slow, obviously correct CPU reference for the
 * non-uniform paged decode-attention path and the coalesced KV gather.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product (the kvx library and its
 * Python binding) may include, link, load or call this code. Only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg use it.
 * It shares no source, header, table or helper with the CUDA path.
 *
 * All floating point is IEEE double. The oracle never sees pages, head groups
 * or a work plan: attention is computed from dense, unpaged K/V plus the
 * explicit set of token positions each head keeps, which is the definition
 * the paged form must reproduce ("Tangram: Unlocking Non-Uniform KV Cache for
 * Efficient Multi-turn LLM Serving", Fig. 2 caption: each head keeps its most
 * critical tokens, which carry most of the attention output; abstract: the
 * accuracy of the serving system is unchanged by its memory layout).
 *
 * Return codes: 0 on success, -1 on invalid arguments (nothing is written).
 */
#ifndef KV_ORACLE_H
#define KV_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Number of tokens head (b,h) keeps: n = min(seq_len[b], budget[b*Hkv+h]).
 * A budget below 1 is invalid (a decode query always sees its own token).
 * Tangram, abstract and Sec. "Deterministic Budget Allocation": every head
 * has a static token budget. Writes n[B*Hkv]. */
int oracle_resolve_budget(int B, int Hkv, const int32_t *budget,
                          const int32_t *seq_len, int32_t *n);

/* Softmax attention of the g query heads that share one KV head, over the
 * n kept positions idx[0..n) (strictly increasing, each in [0, L)).
 *   s_t = scale * <q_j, k_{idx_t}>,  w_t = exp(s_t - max s) / sum_u exp(s_u - max s),
 *   out_j = sum_t w_t v_{idx_t}.
 * q: [g][D]; k, v: [L][D] dense rows (rows outside idx are never read);
 * out: [g][D]; w (optional, may be NULL): [g][n] softmax weights. */
int oracle_attn_head(int D, int g, int L, const double *q, const double *k,
                     const double *v, int n, const int32_t *idx, double scale,
                     double *out, double *w);

/* Decode attention for a whole batch. Query head j of sequence b reads KV
 * head floor(j / (Hq/Hkv)) (contiguous grouped-query mapping).
 * q: [B][Hq][D]; k, v: [B][Hkv][Lmax][D]; kept_off: [B*Hkv+1] offsets into
 * kept_idx (positions of head (b,h) are kept_idx[kept_off[bh] .. kept_off[bh+1]));
 * each kept position must be < seq_len[b] <= Lmax. out: [B][Hq][D].
 * Parallel over (b, h) with OpenMP when available; every head is computed
 * exactly as oracle_attn_head computes it. */
int oracle_decode_attn(int B, int Hq, int Hkv, int D, int Lmax,
                       const int32_t *seq_len, const double *q,
                       const double *k, const double *v,
                       const int64_t *kept_off, const int32_t *kept_idx,
                       double scale, double *out);

/* Pages each head group needs per sequence: the group's page table for
 * sequence b holds ceil(max_{h in group} n[b*Hkv+h] / P) pages, because a
 * group page has one slot row per head of the group and every head of the
 * group advances through the same pages (Tangram, Fig. 8(b): each head group
 * keeps its own page table). head_group[h] in [0, G). pages: [G][B]. */
int oracle_group_pages(int B, int Hkv, const int32_t *n,
                       const int32_t *head_group, int G, int P,
                       int32_t *pages);

/* Guaranteed KV footprint, in bytes, of sequence b for one layer: the sum
 * over groups of pages * |group| * P * 2 (K and V) * D * dtype_bytes
 * (Tangram, Fig. 7 caption: the footprint M(r) in terms of the head
 * dimension and the data-type size; the printed formula is lost, this is the
 * exact page count times page bytes). bytes: [B]. */
int oracle_footprint_bytes(int B, int Hkv, const int32_t *n,
                           const int32_t *head_group, int G, int P, int D,
                           int dtype_bytes, int64_t *bytes);

/* Token coverage of a work plan. items: [nitems][4] = {bh, tok_begin,
 * tok_end, slot}. count: [nheads][maxn] is filled with the number of items
 * that cover each token of each head. Returns the number of violations
 * (a token of [0, n) covered other than exactly once, any token >= n
 * covered, an empty or out-of-range item), or -1 on invalid arguments.
 * Tangram, Fig. 13 and abstract: the ahead-of-time plan splits each head's
 * kept tokens across thread blocks; splitting must not change what is read. */
int64_t oracle_plan_coverage(int nheads, const int32_t *n, int maxn,
                             int nitems, const int32_t *items,
                             int32_t *count);

/* Runs of a block table: maximal stretches of logically consecutive blocks
 * j, j+1, ... of one sequence whose physical ids are p, p+1, ...
 * ("KV-RM: Regularizing KV-Cache Movement for Static-Graph LLM Serving",
 * Fig. 3: descriptor merging turns fragmented page descriptors into a few
 * large transfers). bt: [S][max_blocks]; nb: [S].
 * run_count: [S]; runs: [S][max_blocks][3] = {first physical block,
 * first logical block, length in blocks}, in logical order.
 * Returns the total number of runs, or -1. */
int64_t oracle_runs(int S, int max_blocks, const int32_t *bt,
                    const int32_t *nb, int32_t *run_count, int32_t *runs);

/* Brute-force gather into a fixed-shape staging buffer (KV-RM, abstract and
 * Fig. 2: non-contiguous mappings are materialised into the buffer a
 * fixed-shape attention kernel reads). For every sequence s and logical
 * block j < nb[s]: bytes [j*block_bytes, (j+1)*block_bytes) of staging row s
 * are a copy of physical block bt[s][j] of pool. Bytes of a row past
 * nb[s]*block_bytes are left as they are, or set to zero if zero_tail != 0.
 * pool: [num_phys][block_bytes]; staging: [S][row_bytes]. */
int oracle_gather(int S, int max_blocks, const int32_t *bt, const int32_t *nb,
                  const uint8_t *pool, int64_t num_phys, int64_t block_bytes,
                  uint8_t *staging, int64_t row_bytes, int zero_tail);

/* Kept set of one KV head for sparse long-context decode ("KVDrive", Fig. 7
 * and Fig. 16: attention over the critical top-K entries plus a recent
 * window). With Q = sum of the head's g query vectors,
 *   score_t = <k_t, Q> for t in [0, L - recent),
 *   kept = the min(top, L - recent) positions with the largest scores (equal
 *          scores: lower position first) and every position of
 *          [max(0, L - recent), L), in ascending order.
 * q: [g][D]; k: [L][D]; kept: room for top + recent entries; scores
 * (optional, may be NULL): [L], score_t for t < L - recent, 0 after.
 * Returns the number of kept positions, or -1. */
int oracle_select_topk(int L, int D, int g, const double *q, const double *k,
                       int top, int recent, int32_t *kept, double *scores);

/* Number of OpenMP threads the oracle uses (1 without OpenMP). */
int oracle_num_threads(void);

/* ---- KV-RM block pager and Frame commit (KV-RM, Fig. 2 and Fig. 3) ----
 * The logical KV view of sequence s is a list of physical block ids
 * table[s][0 .. nb[s]); a physical block may be referenced from several
 * places (after Alias) and is free when nothing references it. Runtime
 * variability is expressed as three mapping edits; a Frame commit publishes
 * the edited view as the one descriptor of the next decode step, so the
 * committed state is exactly the state after all edits so far.
 *
 * Placement (not fixed by the pages; stated here): Reserve(s, c) takes the
 * lowest-addressed run of c consecutive free blocks if one exists, else the
 * c lowest-numbered free blocks, ascending.
 *
 * Edits return 0, -1 (bad sequence or negative count), -2 (index range), or
 * -3 (not enough free blocks); a failed edit changes nothing. */
typedef struct oracle_frame oracle_frame;
oracle_frame *oracle_frame_new(int S, int max_blocks, int32_t num_phys);
void oracle_frame_free(oracle_frame *f);
/* Appends c new blocks to sequence s; their ids go to out[0..c) if out. */
int oracle_frame_reserve(oracle_frame *f, int s, int c, int32_t *out);
/* Logical blocks [dj, dj+c) of dst refer to the physical blocks that
 * logical blocks [sj, sj+c) of src refer to (read before any write);
 * dj <= nb[dst]; the view of dst grows to max(nb[dst], dj+c). */
int oracle_frame_alias(oracle_frame *f, int dst, int dj, int src, int sj, int c);
/* Sequence s keeps logical blocks [begin, end) of its view, renumbered from
 * 0; the others are released (Trim(s, 0, 0) ends the sequence). */
int oracle_frame_trim(oracle_frame *f, int s, int begin, int end);
/* The committed descriptor: table [S][max_blocks] (-1 past nb[s]), nb [S];
 * refcount [num_phys] (may be NULL). */
void oracle_frame_state(const oracle_frame *f, int32_t *table, int32_t *nb,
                        int32_t *refcount);
#ifdef __cplusplus
}
#endif
#endif
