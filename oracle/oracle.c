/*
 * oracle.c -- plain fp64 CPU reference (test infrastructure only; see
 * oracle.h). Written from the definitions in the pages, step by step, with
 * no blocking, fusion or reordering beyond what the definition states.
 *
 * ORACLE_MUTANT: when the test suite compiles this file with
 * -DORACLE_MUTANT=<k>, one deliberate mistake is planted so that the tests
 * can show that their pins catch it. The normal build never defines it.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Tangram, Sec. "Deterministic Budget Allocation": a static budget per head;
 * a head never keeps more tokens than its sequence has. */
int oracle_resolve_budget(int B, int Hkv, const int32_t *budget,
                          const int32_t *seq_len, int32_t *n) {
  if (B < 0 || Hkv <= 0 || !budget || !seq_len || !n) return -1;
  for (int b = 0; b < B; ++b) {
    if (seq_len[b] < 1) return -1;
    for (int h = 0; h < Hkv; ++h)
      if (budget[b * Hkv + h] < 1) return -1;
  }
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < Hkv; ++h) {
      int32_t c = budget[b * Hkv + h];
      int32_t L = seq_len[b];
#if ORACLE_MUTANT == 15
      n[b * Hkv + h] = c > L ? c : L;
#else
      n[b * Hkv + h] = c < L ? c : L;
#endif
    }
  return 0;
}

/* Softmax attention over the kept set of one KV head, for its g query
 * heads (Tangram, Fig. 2: attention output over each head's critical tokens;
 * plain scaled dot-product softmax attention). */
int oracle_attn_head(int D, int g, int L, const double *q, const double *k,
                     const double *v, int n, const int32_t *idx, double scale,
                     double *out, double *w) {
  if (D <= 0 || g <= 0 || L <= 0 || n <= 0 || n > L || !q || !k || !v ||
      !idx || !out)
    return -1;
  for (int t = 0; t < n; ++t) {
    if (idx[t] < 0 || idx[t] >= L) return -1;
    if (t > 0 && idx[t] <= idx[t - 1]) return -1;
  }
  double *s = (double *)malloc(sizeof(double) * (size_t)n);
  if (!s) return -1;
  for (int j = 0; j < g; ++j) {
    const double *qj = q + (size_t)j * D;
    /* scores s_t = scale * <q_j, k_t> over the kept positions */
    for (int t = 0; t < n; ++t) {
#if ORACLE_MUTANT == 5
      const double *kt = k + (size_t)t * D;
#else
      const double *kt = k + (size_t)idx[t] * D;
#endif
      double dot = 0.0;
      for (int d = 0; d < D; ++d) dot += qj[d] * kt[d];
#if ORACLE_MUTANT == 2
      s[t] = dot;
#elif ORACLE_MUTANT == 8
      s[t] = -scale * dot;
#else
      s[t] = scale * dot;
#endif
    }
    /* softmax: subtract the maximum, exponentiate, normalise */
    double m = s[0];
    for (int t = 1; t < n; ++t)
      if (s[t] > m) m = s[t];
#if ORACLE_MUTANT == 3
    m = 0.0;
#endif
    double z = 0.0;
    for (int t = 0; t < n; ++t) {
      s[t] = exp(s[t] - m);
      z += s[t];
    }
#if ORACLE_MUTANT == 4
    z = 1.0;
#endif
    for (int t = 0; t < n; ++t) s[t] = s[t] / z;
    if (w)
      for (int t = 0; t < n; ++t) w[(size_t)j * n + t] = s[t];
    /* out_j = sum_t w_t v_t */
    double *oj = out + (size_t)j * D;
    for (int d = 0; d < D; ++d) {
      double acc = 0.0;
#if ORACLE_MUTANT == 6
      int nt = n > 1 ? n - 1 : n;
#else
      int nt = n;
#endif
      for (int t = 0; t < nt; ++t) {
#if ORACLE_MUTANT == 7
        acc += s[t] * v[(size_t)d * L + idx[t]];
#else
        acc += s[t] * v[(size_t)idx[t] * D + d];
#endif
      }
      oj[d] = acc;
    }
  }
  free(s);
  return 0;
}

int oracle_decode_attn(int B, int Hq, int Hkv, int D, int Lmax,
                       const int32_t *seq_len, const double *q,
                       const double *k, const double *v,
                       const int64_t *kept_off, const int32_t *kept_idx,
                       double scale, double *out) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Lmax <= 0 || Hq % Hkv != 0 ||
      !seq_len || !q || !k || !v || !kept_off || !kept_idx || !out)
    return -1;
  const int g = Hq / Hkv;
  for (int b = 0; b < B; ++b)
    if (seq_len[b] < 1 || seq_len[b] > Lmax) return -1;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int bh = 0; bh < B * Hkv; ++bh) {
    int b = bh / Hkv, h = bh % Hkv;
    int64_t n64 = kept_off[bh + 1] - kept_off[bh];
    if (n64 < 1 || n64 > seq_len[b]) {
      bad |= 1;
      continue;
    }
    /* query heads of KV head h: j = h*g .. h*g+g-1 */
    for (int jj = 0; jj < g; ++jj) {
      int j = h * g + jj;
#if ORACLE_MUTANT == 1
      int hk = j % Hkv;
#else
      int hk = j / g;
#endif
      const double *kh = k + ((size_t)b * Hkv + hk) * (size_t)Lmax * D;
      const double *vh = v + ((size_t)b * Hkv + hk) * (size_t)Lmax * D;
      const int32_t *ix = kept_idx + kept_off[b * Hkv + hk];
      int nn = (int)(kept_off[b * Hkv + hk + 1] - kept_off[b * Hkv + hk]);
      if (oracle_attn_head(D, 1, seq_len[b], q + ((size_t)b * Hq + j) * D, kh,
                           vh, nn, ix, scale, out + ((size_t)b * Hq + j) * D,
                           NULL) != 0)
        bad |= 1;
    }
  }
  return bad ? -1 : 0;
}

/* Tangram, Fig. 8(b)/(c): a head group has its own page table; all heads of
 * the group walk the same pages, so the group needs as many pages as its
 * longest head. */
int oracle_group_pages(int B, int Hkv, const int32_t *n,
                       const int32_t *head_group, int G, int P,
                       int32_t *pages) {
  if (B < 0 || Hkv <= 0 || G <= 0 || P <= 0 || !n || !head_group || !pages)
    return -1;
  for (int h = 0; h < Hkv; ++h)
    if (head_group[h] < 0 || head_group[h] >= G) return -1;
  for (int gi = 0; gi < G; ++gi)
    for (int b = 0; b < B; ++b) {
      int32_t mx = 0;
#if ORACLE_MUTANT == 10
      mx = 0x7fffffff;
#endif
      for (int h = 0; h < Hkv; ++h) {
        if (head_group[h] != gi) continue;
        int32_t c = n[b * Hkv + h];
#if ORACLE_MUTANT == 10
        if (c < mx) mx = c;
#else
        if (c > mx) mx = c;
#endif
      }
#if ORACLE_MUTANT == 10
      if (mx == 0x7fffffff) mx = 0;
#endif
#if ORACLE_MUTANT == 9
      pages[gi * B + b] = mx / P;
#else
      pages[gi * B + b] = (mx + P - 1) / P;
#endif
    }
  return 0;
}

int oracle_footprint_bytes(int B, int Hkv, const int32_t *n,
                           const int32_t *head_group, int G, int P, int D,
                           int dtype_bytes, int64_t *bytes) {
  if (D <= 0 || dtype_bytes <= 0 || !bytes || G <= 0 || B < 0) return -1;
  int32_t *pages = (int32_t *)malloc(sizeof(int32_t) * (size_t)(G * B + 1));
  if (!pages) return -1;
  if (oracle_group_pages(B, Hkv, n, head_group, G, P, pages) != 0) {
    free(pages);
    return -1;
  }
  for (int b = 0; b < B; ++b) {
    int64_t tot = 0;
    for (int gi = 0; gi < G; ++gi) {
      int64_t size = 0;
      for (int h = 0; h < Hkv; ++h) size += (head_group[h] == gi);
      tot += (int64_t)pages[gi * B + b] * size * P * 2 * D * dtype_bytes;
    }
    bytes[b] = tot;
  }
  free(pages);
  return 0;
}

int64_t oracle_plan_coverage(int nheads, const int32_t *n, int maxn,
                             int nitems, const int32_t *items,
                             int32_t *count) {
  if (nheads < 0 || maxn < 0 || nitems < 0 || !n || !count ||
      (nitems > 0 && !items))
    return -1;
  for (int bh = 0; bh < nheads; ++bh)
    if (n[bh] < 0 || n[bh] > maxn) return -1;
  memset(count, 0, sizeof(int32_t) * (size_t)nheads * (size_t)maxn);
  int64_t bad = 0;
  for (int i = 0; i < nitems; ++i) {
    int32_t bh = items[4 * i + 0], b0 = items[4 * i + 1],
            e0 = items[4 * i + 2];
    if (bh < 0 || bh >= nheads || b0 < 0 || e0 <= b0 || e0 > maxn) {
      ++bad;
      continue;
    }
    for (int t = b0; t < e0; ++t) count[(size_t)bh * maxn + t] += 1;
  }
  for (int bh = 0; bh < nheads; ++bh)
    for (int t = 0; t < maxn; ++t) {
      int32_t c = count[(size_t)bh * maxn + t];
#if ORACLE_MUTANT == 14
      if (t < n[bh] && c != 1) ++bad;
#else
      if (t < n[bh] ? c != 1 : c != 0) ++bad;
#endif
    }
  return bad;
}

/* KV-RM, Fig. 3: descriptor merging. A run continues while both the logical
 * block index and the physical block id advance by one. */
int64_t oracle_runs(int S, int max_blocks, const int32_t *bt,
                    const int32_t *nb, int32_t *run_count, int32_t *runs) {
  if (S < 0 || max_blocks < 0 || !bt || !nb || !run_count || !runs) return -1;
  for (int s = 0; s < S; ++s)
    if (nb[s] < 0 || nb[s] > max_blocks) return -1;
  int64_t total = 0;
  for (int s = 0; s < S; ++s) {
    const int32_t *row = bt + (size_t)s * max_blocks;
    int32_t *out = runs + (size_t)s * max_blocks * 3;
    int r = -1;
    for (int j = 0; j < nb[s]; ++j) {
#if ORACLE_MUTANT == 11
      int cont = (j > 0) && (row[j] == row[j - 1]);
#else
      int cont = (j > 0) && (row[j] == row[j - 1] + 1);
#endif
      if (!cont) {
        ++r;
        out[3 * r + 0] = row[j];
        out[3 * r + 1] = j;
        out[3 * r + 2] = 1;
      } else {
        out[3 * r + 2] += 1;
      }
    }
    run_count[s] = r + 1;
    total += r + 1;
  }
  return total;
}

/* KV-RM, abstract and Fig. 2: every live block of a sequence lands in its
 * logical position of the fixed-shape staging row. */
int oracle_gather(int S, int max_blocks, const int32_t *bt, const int32_t *nb,
                  const uint8_t *pool, int64_t num_phys, int64_t block_bytes,
                  uint8_t *staging, int64_t row_bytes, int zero_tail) {
  if (S < 0 || max_blocks < 0 || !bt || !nb || !pool || !staging ||
      num_phys <= 0 || block_bytes <= 0 || row_bytes < 0)
    return -1;
  for (int s = 0; s < S; ++s) {
    if (nb[s] < 0 || nb[s] > max_blocks) return -1;
    if ((int64_t)nb[s] * block_bytes > row_bytes) return -1;
    for (int j = 0; j < nb[s]; ++j) {
      int32_t p = bt[(size_t)s * max_blocks + j];
      if (p < 0 || p >= num_phys) return -1;
    }
  }
#pragma omp parallel for schedule(dynamic, 1)
  for (int s = 0; s < S; ++s) {
    uint8_t *row = staging + (size_t)s * row_bytes;
#if ORACLE_MUTANT == 13
    int last = nb[s] + 1 <= max_blocks &&
                       (int64_t)(nb[s] + 1) * block_bytes <= row_bytes
                   ? nb[s] + 1
                   : nb[s];
#else
    int last = nb[s];
#endif
    for (int j = 0; j < last; ++j) {
      int32_t p = bt[(size_t)s * max_blocks + j];
      if (p < 0 || p >= num_phys) continue;
#if ORACLE_MUTANT == 12
      int64_t dst = (int64_t)(p % (last > 0 ? last : 1)) * block_bytes;
#else
      int64_t dst = (int64_t)j * block_bytes;
#endif
      memcpy(row + dst, pool + (size_t)p * (size_t)block_bytes,
             (size_t)block_bytes);
    }
    if (zero_tail) {
      int64_t used = (int64_t)nb[s] * block_bytes;
      memset(row + used, 0, (size_t)(row_bytes - used));
    }
  }
  return 0;
}

/* KVDrive, Fig. 7 / Fig. 16: the critical KV entries of a head are those
 * with the largest attention scores; the grouped query heads of one KV head
 * score a token by the sum of their dot products, i.e. <k_t, sum_j q_j>. */
typedef struct {
  double s;
  int32_t t;
} oracle_scored;

static int oracle_cmp_scored(const void *a, const void *b) {
  const oracle_scored *x = (const oracle_scored *)a, *y = (const oracle_scored *)b;
  if (x->s != y->s) return x->s > y->s ? -1 : 1; /* larger score first */
#if ORACLE_MUTANT == 16
  return x->t > y->t ? -1 : (x->t < y->t); /* ties: higher position first */
#else
  return x->t < y->t ? -1 : (x->t > y->t); /* ties: lower position first */
#endif
}

static int oracle_cmp_i32(const void *a, const void *b) {
  const int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
  return x < y ? -1 : (x > y);
}

int oracle_select_topk(int L, int D, int g, const double *q, const double *k,
                       int top, int recent, int32_t *kept, double *scores) {
  if (L <= 0 || D <= 0 || g <= 0 || top < 0 || recent < 0 || !q || !k || !kept)
    return -1;
  double *Q = (double *)calloc((size_t)D, sizeof(double));
  if (!Q) return -1;
#if ORACLE_MUTANT == 17
  for (int d = 0; d < D; ++d) Q[d] = q[d]; /* only the first query head */
#else
  for (int j = 0; j < g; ++j)
    for (int d = 0; d < D; ++d) Q[d] += q[(size_t)j * D + d];
#endif
  const int n = L - recent > 0 ? L - recent : 0;
  oracle_scored *c = (oracle_scored *)malloc(sizeof(oracle_scored) * (size_t)(n > 0 ? n : 1));
  if (!c) {
    free(Q);
    return -1;
  }
  for (int t = 0; t < n; ++t) {
    double s = 0.0;
    for (int d = 0; d < D; ++d) s += k[(size_t)t * D + d] * Q[d];
    c[t].s = s;
    c[t].t = t;
  }
  if (scores) {
    for (int t = 0; t < L; ++t) scores[t] = t < n ? c[t].s : 0.0;
  }
  qsort(c, (size_t)n, sizeof(oracle_scored), oracle_cmp_scored);
  const int ntop = top < n ? top : n;
  int cnt = 0;
  for (int i = 0; i < ntop; ++i) kept[cnt++] = c[i].t;
#if ORACLE_MUTANT == 18
  for (int t = n + 1; t < L; ++t) kept[cnt++] = t; /* recent window one short */
#else
  for (int t = n; t < L; ++t) kept[cnt++] = t;
#endif
  qsort(kept, (size_t)cnt, sizeof(int32_t), oracle_cmp_i32);
  free(c);
  free(Q);
  return cnt;
}

/* KV-RM, Fig. 2 (block pager) and Fig. 3 (Alias, Trim, Reserve sealed by
 * one Frame commit). Plain arrays; every edit validates first and then
 * applies, so a failed edit changes nothing. */
struct oracle_frame {
  int S, M;
  int32_t N;
  int32_t *table; /* [S][M], -1 past nb */
  int32_t *nb;    /* [S] */
  int32_t *rc;    /* [N] references from table entries */
};

oracle_frame *oracle_frame_new(int S, int max_blocks, int32_t num_phys) {
  if (S <= 0 || max_blocks <= 0 || num_phys <= 0) return NULL;
  oracle_frame *f = (oracle_frame *)calloc(1, sizeof(oracle_frame));
  if (!f) return NULL;
  f->S = S;
  f->M = max_blocks;
  f->N = num_phys;
  f->table = (int32_t *)malloc(sizeof(int32_t) * (size_t)S * (size_t)max_blocks);
  f->nb = (int32_t *)calloc((size_t)S, sizeof(int32_t));
  f->rc = (int32_t *)calloc((size_t)num_phys, sizeof(int32_t));
  if (!f->table || !f->nb || !f->rc) {
    oracle_frame_free(f);
    return NULL;
  }
  for (size_t i = 0; i < (size_t)S * (size_t)max_blocks; ++i) f->table[i] = -1;
  return f;
}

void oracle_frame_free(oracle_frame *f) {
  if (!f) return;
  free(f->table);
  free(f->nb);
  free(f->rc);
  free(f);
}

static void oracle_frame_release(oracle_frame *f, int32_t p) {
#if ORACLE_MUTANT != 20
  f->rc[p] -= 1;
#else
  (void)f;
  (void)p;
#endif
}

int oracle_frame_reserve(oracle_frame *f, int s, int c, int32_t *out) {
  if (!f || s < 0 || s >= f->S || c < 0) return -1;
  if (f->nb[s] + c > f->M) return -2;
  int32_t nfree = 0;
  for (int32_t p = 0; p < f->N; ++p) nfree += f->rc[p] == 0;
  if (c > nfree) return -3;
  if (c == 0) return 0;
  int32_t *pick = (int32_t *)malloc(sizeof(int32_t) * (size_t)c);
  if (!pick) return -1;
  /* lowest-addressed run of c consecutive free blocks */
  int32_t start = -1, run = 0;
  for (int32_t p = 0; p < f->N; ++p) {
    run = f->rc[p] == 0 ? run + 1 : 0;
    if (run == c) {
#if ORACLE_MUTANT == 19
      start = p - c; /* off by one */
      if (start < 0) start = 0;
#else
      start = p - c + 1;
#endif
      break;
    }
  }
  if (start >= 0) {
    for (int i = 0; i < c; ++i) pick[i] = start + i;
  } else {
    /* no such run: the c lowest-numbered free blocks */
    int i = 0;
#if ORACLE_MUTANT == 23
    for (int32_t p = f->N - 1; p >= 0 && i < c; --p)
#else
    for (int32_t p = 0; p < f->N && i < c; ++p)
#endif
      if (f->rc[p] == 0) pick[i++] = p;
  }
  for (int i = 0; i < c; ++i) {
    f->table[(size_t)s * f->M + f->nb[s] + i] = pick[i];
    f->rc[pick[i]] += 1;
    if (out) out[i] = pick[i];
  }
  f->nb[s] += c;
  free(pick);
  return 0;
}

int oracle_frame_alias(oracle_frame *f, int dst, int dj, int src, int sj, int c) {
  if (!f || dst < 0 || dst >= f->S || src < 0 || src >= f->S || c < 0) return -1;
  if (sj < 0 || sj + c > f->nb[src]) return -2;
  if (dj < 0 || dj > f->nb[dst] || dj + c > f->M) return -2;
  if (c == 0) return 0;
  int32_t *val = (int32_t *)malloc(sizeof(int32_t) * (size_t)c);
  if (!val) return -1;
  int32_t *srow = f->table + (size_t)src * f->M;
  int32_t *drow = f->table + (size_t)dst * f->M;
#if ORACLE_MUTANT == 21
  /* reads each source after the earlier writes */
  for (int i = 0; i < c; ++i) {
    int32_t v = srow[sj + i];
    if (dj + i < f->nb[dst]) oracle_frame_release(f, drow[dj + i]);
    drow[dj + i] = v;
    f->rc[v] += 1;
  }
#else
  for (int i = 0; i < c; ++i) val[i] = srow[sj + i];
  for (int i = 0; i < c; ++i) {
    if (dj + i < f->nb[dst]) oracle_frame_release(f, drow[dj + i]);
    drow[dj + i] = val[i];
    f->rc[val[i]] += 1;
  }
#endif
  if (dj + c > f->nb[dst]) f->nb[dst] = dj + c;
  free(val);
  return 0;
}

int oracle_frame_trim(oracle_frame *f, int s, int begin, int end) {
  if (!f || s < 0 || s >= f->S) return -1;
  if (begin < 0 || begin > end || end > f->nb[s]) return -2;
  int32_t *row = f->table + (size_t)s * f->M;
  const int n = f->nb[s];
#if ORACLE_MUTANT != 24
  for (int j = 0; j < begin; ++j) oracle_frame_release(f, row[j]);
#endif
#if ORACLE_MUTANT == 22
  for (int j = end + 1; j < n; ++j) oracle_frame_release(f, row[j]);
#else
  for (int j = end; j < n; ++j) oracle_frame_release(f, row[j]);
#endif
  for (int j = 0; j < end - begin; ++j) row[j] = row[begin + j];
  for (int j = end - begin; j < n; ++j) row[j] = -1;
  f->nb[s] = end - begin;
  return 0;
}

void oracle_frame_state(const oracle_frame *f, int32_t *table, int32_t *nb,
                        int32_t *refcount) {
  memcpy(table, f->table, sizeof(int32_t) * (size_t)f->S * (size_t)f->M);
  memcpy(nb, f->nb, sizeof(int32_t) * (size_t)f->S);
  if (refcount) memcpy(refcount, f->rc, sizeof(int32_t) * (size_t)f->N);
}
