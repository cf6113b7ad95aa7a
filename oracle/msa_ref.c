/* MSA CPU oracle -- TEST INFRASTRUCTURE ONLY (see msa_ref.h).
 *
 * Every function follows "MiniMax 模型迭代与竞品分析：从 Text-01、M1、M2 到 M3",
 * section 2 ("从 Lightning Attention 到 MSA"), in the order the page gives:
 *
 *   step 1  global scoring: per GQA group a light index query Q_idx is scored
 *           against the index key K_idx that all groups share, over the whole
 *           causal context;
 *   step 2  token -> block: 128-token KV blocks, block score = max of its
 *           token scores;
 *   step 3  selection: 16 blocks per query and group, the local block forced
 *           in as one of the 16;
 *   step 4  exact computation: standard softmax attention over the selected
 *           blocks only (at most 16 x 128 = 2048 tokens), the per-head
 *           equation s = q.k / sqrt(d_k), alpha = softmax over j <= t,
 *           o = sum alpha v given in the same section; GQA only decides which
 *           KV head a query head reads.
 *
 * Readings where the page is silent (kept identical in the CUDA library):
 *   - the index score is the raw dot product <Q_idx, K_idx> (no scale, no
 *     activation); ranking uses raw pooled scores (no exp);
 *   - the local block is lb = floor(t / block); candidates are blocks < lb;
 *     with fewer than topk causal blocks, all lb + 1 are selected;
 *   - equal pooled scores rank the lower block id first;
 *   - selected ids are stored ascending and padded with -1;
 *   - one softmax runs jointly over all selected tokens <= t, per query head,
 *     with the KV head of its group (group g = h / (H/G)).
 *
 * Arithmetic is double throughout; bf16 inputs widen exactly.
 */
#include "msa_ref.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

static double bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static int dims_ok(const msa_ref_dims *p) {
  return p && p->H > 0 && p->G > 0 && p->H % p->G == 0 && p->D > 0 && p->Di > 0 &&
         p->block > 0 && p->topk > 0;
}

typedef struct {
  double score;
  int32_t blk;
} cand_t;

/* Ranking of candidate blocks: higher pooled score first, lower id on ties. */
static int cand_cmp(const void *a, const void *b) {
  const cand_t *x = (const cand_t *)a, *y = (const cand_t *)b;
  if (x->score > y->score) return -1;
  if (x->score < y->score) return 1;
  return (x->blk > y->blk) - (x->blk < y->blk);
}

static int int_cmp(const void *a, const void *b) {
  int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
  return (x > y) - (x < y);
}

int msa_ref_select(const msa_ref_dims *p, int64_t t, const uint16_t *q_idx_t,
                   const uint16_t *k_idx, int32_t *sel_t, double *pooled) {
  if (!dims_ok(p) || t < 0 || !q_idx_t || !k_idx || !sel_t) return -1;
  const int64_t lb = t / p->block; /* local block: the one holding t */
  cand_t *cand = (cand_t *)malloc((size_t)(lb > 0 ? lb : 1) * sizeof(cand_t));
  if (!cand) return -1;
  for (int g = 0; g < p->G; ++g) {
    const uint16_t *qg = q_idx_t + (size_t)g * p->Di;
    /* steps 1 + 2: score every causal token of every candidate block, keep
     * the block maximum */
    for (int64_t blk = 0; blk < lb; ++blk) {
      double best = -INFINITY;
      for (int64_t tok = blk * p->block; tok < (blk + 1) * p->block && tok <= t; ++tok) {
        const uint16_t *kr = k_idx + (size_t)tok * p->Di;
        double s = 0.0;
        for (int d = 0; d < p->Di; ++d) s += bf16_to_double(qg[d]) * bf16_to_double(kr[d]);
        if (s > best) best = s;
      }
      cand[blk].score = best;
      cand[blk].blk = (int32_t)blk;
      if (pooled) pooled[(size_t)g * lb + blk] = best;
    }
    /* step 3: full sort of the candidates, local block first, then the best
     * topk-1 others */
    qsort(cand, (size_t)lb, sizeof(cand_t), cand_cmp);
    int64_t nsel = lb + 1 < p->topk ? lb + 1 : p->topk;
    int32_t *s = sel_t + (size_t)g * p->topk;
    s[0] = (int32_t)lb;
    for (int64_t i = 1; i < nsel; ++i) s[i] = cand[i - 1].blk;
    qsort(s, (size_t)nsel, sizeof(int32_t), int_cmp);
    for (int64_t i = nsel; i < p->topk; ++i) s[i] = -1;
  }
  free(cand);
  return 0;
}

/* Softmax of the logits z[0..n) against the value rows vrow[0..n): out[D]. */
static void softmax_combine(int n, const double *z, const uint16_t *const *vrow, int D,
                            double *out) {
  double m = -INFINITY;
  for (int i = 0; i < n; ++i)
    if (z[i] > m) m = z[i];
  double l = 0.0;
  for (int d = 0; d < D; ++d) out[d] = 0.0;
  for (int i = 0; i < n; ++i) {
    double w = exp(z[i] - m);
    l += w;
    for (int d = 0; d < D; ++d) out[d] += w * bf16_to_double(vrow[i][d]);
  }
  for (int d = 0; d < D; ++d) out[d] /= l;
}

static int attend_tokens(const msa_ref_dims *p, int64_t t, const uint16_t *q_t,
                         const uint16_t *k, const uint16_t *v, const int32_t *sel_t,
                         int dense, double *out_t) {
  const int hpg = p->H / p->G;
  const size_t row = (size_t)p->G * p->D; /* one token's K (or V) row, all heads */
  const int64_t maxn = dense ? t + 1 : (int64_t)p->topk * p->block;
  double *z = (double *)malloc((size_t)maxn * sizeof(double));
  const uint16_t **krow = (const uint16_t **)malloc((size_t)maxn * sizeof(*krow));
  const uint16_t **vrow = (const uint16_t **)malloc((size_t)maxn * sizeof(*vrow));
  if (!z || !krow || !vrow) {
    free(z); free(krow); free(vrow);
    return -1;
  }
  const int64_t lb = t / p->block;
  int rc = 0;
  for (int g = 0; g < p->G && rc == 0; ++g) {
    /* the token set of group g: selected blocks, tokens <= t */
    int n = 0;
    if (dense) {
      for (int64_t tok = 0; tok <= t; ++tok) {
        krow[n] = k + (size_t)tok * row + (size_t)g * p->D;
        vrow[n] = v + (size_t)tok * row + (size_t)g * p->D;
        ++n;
      }
    } else {
      const int32_t *s = sel_t + (size_t)g * p->topk;
      for (int j = 0; j < p->topk; ++j) {
        if (s[j] < 0) continue;
        if (s[j] > lb) { rc = -1; break; }
        for (int64_t tok = (int64_t)s[j] * p->block; tok < ((int64_t)s[j] + 1) * p->block; ++tok) {
          if (tok > t) continue;
          krow[n] = k + (size_t)tok * row + (size_t)g * p->D;
          vrow[n] = v + (size_t)tok * row + (size_t)g * p->D;
          ++n;
        }
      }
    }
    if (rc != 0) break;
    for (int hh = 0; hh < hpg; ++hh) {
      const int h = g * hpg + hh;
      const uint16_t *qh = q_t + (size_t)h * p->D;
      for (int i = 0; i < n; ++i) {
        double s = 0.0;
        for (int d = 0; d < p->D; ++d) s += bf16_to_double(qh[d]) * bf16_to_double(krow[i][d]);
        z[i] = s * p->scale;
      }
      softmax_combine(n, z, vrow, p->D, out_t + (size_t)h * p->D);
    }
  }
  free(z); free(krow); free(vrow);
  return rc;
}

int msa_ref_attend(const msa_ref_dims *p, int64_t t, const uint16_t *q_t, const uint16_t *k,
                   const uint16_t *v, const int32_t *sel_t, double *out_t) {
  if (!dims_ok(p) || t < 0 || !q_t || !k || !v || !sel_t || !out_t) return -1;
  return attend_tokens(p, t, q_t, k, v, sel_t, 0, out_t);
}

int msa_ref_dense(const msa_ref_dims *p, int64_t t, const uint16_t *q_t, const uint16_t *k,
                  const uint16_t *v, double *out_t) {
  if (!dims_ok(p) || t < 0 || !q_t || !k || !v || !out_t) return -1;
  return attend_tokens(p, t, q_t, k, v, NULL, 1, out_t);
}

/* Attention mass per block and head under the full causal softmax, then the
 * ideal selection under the MSA rule, and how much of the mass the given and
 * the ideal selections hold.  Double throughout. */
int msa_ref_quality(const msa_ref_dims *p, int64_t t, const uint16_t *q_t, const uint16_t *k,
                    const int32_t *sel_t, double *coverage, double *best_coverage,
                    int32_t *dense_sel, int32_t *hits, double *mass) {
  if (!dims_ok(p) || t < 0 || !q_t || !k || !sel_t || !coverage || !best_coverage ||
      !dense_sel || !hits)
    return -1;
  const int hpg = p->H / p->G;
  const size_t row = (size_t)p->G * p->D;
  const int64_t lb = t / p->block, nblk = lb + 1;
  double *z = (double *)malloc((size_t)(t + 1) * sizeof(double));
  double *A = (double *)malloc((size_t)hpg * nblk * sizeof(double)); /* [hh][b] */
  double *P = (double *)malloc((size_t)nblk * sizeof(double));
  cand_t *cand = (cand_t *)malloc((size_t)(lb > 0 ? lb : 1) * sizeof(cand_t));
  if (!z || !A || !P || !cand) {
    free(z); free(A); free(P); free(cand);
    return -1;
  }
  for (int g = 0; g < p->G; ++g) {
    for (int64_t b = 0; b < nblk; ++b) P[b] = 0.0;
    for (int hh = 0; hh < hpg; ++hh) {
      const uint16_t *qh = q_t + (size_t)(g * hpg + hh) * p->D;
      /* the full causal softmax of head h: every token 0..t */
      double m = -INFINITY;
      for (int64_t i = 0; i <= t; ++i) {
        const uint16_t *kr = k + (size_t)i * row + (size_t)g * p->D;
        double s = 0.0;
        for (int d = 0; d < p->D; ++d) s += bf16_to_double(qh[d]) * bf16_to_double(kr[d]);
        z[i] = s * p->scale;
        if (z[i] > m) m = z[i];
      }
      double Z = 0.0;
      for (int64_t i = 0; i <= t; ++i) {
        z[i] = exp(z[i] - m);
        Z += z[i];
      }
      double *Ah = A + (size_t)hh * nblk;
      for (int64_t b = 0; b < nblk; ++b) Ah[b] = 0.0;
      for (int64_t i = 0; i <= t; ++i) Ah[i / p->block] += z[i] / Z;
      for (int64_t b = 0; b < nblk; ++b) P[b] += Ah[b] / hpg;
    }
    if (mass)
      for (int64_t b = 0; b < nblk; ++b) mass[(size_t)g * nblk + b] = P[b];
    /* the ideal selection: local block forced, then the best candidates by
     * group-averaged mass (same ranking rule as the index branch) */
    for (int64_t b = 0; b < lb; ++b) {
      cand[b].score = P[b];
      cand[b].blk = (int32_t)b;
    }
    qsort(cand, (size_t)lb, sizeof(cand_t), cand_cmp);
    const int64_t nsel = lb + 1 < p->topk ? lb + 1 : p->topk;
    int32_t *ds = dense_sel + (size_t)g * p->topk;
    ds[0] = (int32_t)lb;
    for (int64_t i = 1; i < nsel; ++i) ds[i] = cand[i - 1].blk;
    qsort(ds, (size_t)nsel, sizeof(int32_t), int_cmp);
    for (int64_t i = nsel; i < p->topk; ++i) ds[i] = -1;
    /* the given selection as a set of distinct valid ids */
    const int32_t *s = sel_t + (size_t)g * p->topk;
    int32_t given[64];
    int ng = 0;
    for (int j = 0; j < p->topk && j < 64; ++j) {
      if (s[j] < 0 || s[j] > lb) continue;
      int dup = 0;
      for (int u = 0; u < ng; ++u) dup |= given[u] == s[j];
      if (!dup) given[ng++] = s[j];
    }
    int h = 0;
    for (int u = 0; u < ng; ++u)
      for (int64_t i = 0; i < nsel; ++i) h += given[u] == ds[i];
    hits[g] = h;
    for (int hh = 0; hh < hpg; ++hh) {
      const double *Ah = A + (size_t)hh * nblk;
      double c = 0.0, cb = 0.0;
      for (int u = 0; u < ng; ++u) c += Ah[given[u]];
      for (int64_t i = 0; i < nsel; ++i) cb += Ah[ds[i]];
      coverage[g * hpg + hh] = c;
      best_coverage[g * hpg + hh] = cb;
    }
  }
  free(z); free(A); free(P); free(cand);
  return 0;
}

/* The candidate blocks of one group: the distinct ids of s in [0, lb], in
 * slot order. */
static int candidates(const int32_t *s, int topk, int64_t lb, int32_t *out) {
  int n = 0;
  for (int j = 0; j < topk; ++j) {
    if (s[j] < 0 || s[j] > lb) continue;
    int dup = 0;
    for (int u = 0; u < n; ++u) dup |= out[u] == s[j];
    if (!dup) out[n++] = s[j];
  }
  return n;
}

int msa_ref_index_kl(const msa_ref_dims *p, int64_t t, const uint16_t *q_idx_t,
                     const uint16_t *k_idx, const uint16_t *q_t, const uint16_t *k,
                     const int32_t *sel_t, double *kl, double *dq_idx, double *dk_idx) {
  if (!dims_ok(p) || t < 0 || !q_idx_t || !k_idx || !q_t || !k || !sel_t || !kl || !dq_idx ||
      !dk_idx || p->topk > 64)
    return -1;
  const int hpg = p->H / p->G;
  const size_t row = (size_t)p->G * p->D;
  const int64_t lb = t / p->block;
  double *z = (double *)malloc((size_t)p->topk * p->block * sizeof(double));
  if (!z) return -1;
  for (int g = 0; g < p->G; ++g) {
    int32_t c[64];
    const int n = candidates(sel_t + (size_t)g * p->topk, p->topk, lb, c);
    double P[64], zi[64], Q[64];
    int64_t arg[64];
    for (int j = 0; j < n; ++j) P[j] = 0.0;
    /* P: the main branch's softmax over the selected tokens, mass per block,
     * averaged over the group's heads */
    for (int hh = 0; hh < hpg; ++hh) {
      const uint16_t *qh = q_t + (size_t)(g * hpg + hh) * p->D;
      double m = -INFINITY;
      int64_t ntok = 0;
      for (int j = 0; j < n; ++j)
        for (int64_t tok = (int64_t)c[j] * p->block; tok < ((int64_t)c[j] + 1) * p->block; ++tok) {
          if (tok > t) continue;
          const uint16_t *kr = k + (size_t)tok * row + (size_t)g * p->D;
          double s = 0.0;
          for (int d = 0; d < p->D; ++d) s += bf16_to_double(qh[d]) * bf16_to_double(kr[d]);
          z[ntok] = s * p->scale;
          if (z[ntok] > m) m = z[ntok];
          ++ntok;
        }
      double Z = 0.0;
      for (int64_t i = 0; i < ntok; ++i) Z += exp(z[i] - m);
      int64_t i = 0;
      for (int j = 0; j < n; ++j)
        for (int64_t tok = (int64_t)c[j] * p->block; tok < ((int64_t)c[j] + 1) * p->block; ++tok) {
          if (tok > t) continue;
          P[j] += exp(z[i++] - m) / Z / hpg;
        }
    }
    /* Q: softmax of the pooled index scores of the same blocks */
    const uint16_t *qi = q_idx_t + (size_t)g * p->Di;
    double zmax = -INFINITY;
    for (int j = 0; j < n; ++j) {
      zi[j] = -INFINITY;
      arg[j] = -1;
      for (int64_t tok = (int64_t)c[j] * p->block; tok < ((int64_t)c[j] + 1) * p->block; ++tok) {
        if (tok > t) continue;
        const uint16_t *kr = k_idx + (size_t)tok * p->Di;
        double s = 0.0;
        for (int d = 0; d < p->Di; ++d) s += bf16_to_double(qi[d]) * bf16_to_double(kr[d]);
        if (s > zi[j]) { /* strictly greater: the first maximal token wins */
          zi[j] = s;
          arg[j] = tok;
        }
      }
      if (zi[j] > zmax) zmax = zi[j];
    }
    double sq = 0.0;
    for (int j = 0; j < n; ++j) sq += exp(zi[j] - zmax);
    double loss = 0.0;
    for (int j = 0; j < n; ++j) {
      Q[j] = exp(zi[j] - zmax) / sq;
      if (P[j] > 0.0) loss += P[j] * (log(P[j]) - log(Q[j]));
    }
    kl[g] = loss;
    /* gradient through the pooled scores to the maximal tokens */
    double *dq = dq_idx + (size_t)g * p->Di;
    for (int d = 0; d < p->Di; ++d) dq[d] = 0.0;
    for (int j = 0; j < n; ++j) {
      const double dz = Q[j] - P[j];
      const uint16_t *kr = k_idx + (size_t)arg[j] * p->Di;
      double *dk = dk_idx + (size_t)arg[j] * p->Di;
      for (int d = 0; d < p->Di; ++d) {
        dq[d] += dz * bf16_to_double(kr[d]);
#pragma omp atomic
        dk[d] += dz * bf16_to_double(qi[d]);
      }
    }
  }
  free(z);
  return 0;
}

static int batch_ok(const msa_ref_dims *p, int B, int T, int max_blocks, const int32_t *q_start,
                    const int32_t *kv_len) {
  if (!dims_ok(p) || B < 0 || T < 0 || max_blocks < 0 || !q_start || !kv_len) return 0;
  for (int b = 0; b < B; ++b) {
    if (q_start[b] < 0 || (int64_t)q_start[b] + T > kv_len[b] ||
        (int64_t)kv_len[b] > (int64_t)max_blocks * p->block)
      return 0;
  }
  return 1;
}

int msa_ref_index_topk(const msa_ref_dims *p, int B, int T, int max_blocks, const uint16_t *q_idx,
                       const uint16_t *k_idx, const int32_t *q_start, const int32_t *kv_len,
                       int32_t *sel, int nthreads) {
  if (!batch_ok(p, B, T, max_blocks, q_start, kv_len) || !q_idx || !k_idx || !sel) return -1;
  const size_t cap = (size_t)max_blocks * p->block;
  int rc = 0;
  const int64_t n = (int64_t)B * T;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1)
  for (int64_t r = 0; r < n; ++r) {
    const int b = (int)(r / T), i = (int)(r % T);
    int e = msa_ref_select(p, (int64_t)q_start[b] + i, q_idx + (size_t)r * p->G * p->Di,
                           k_idx + (size_t)b * cap * p->Di, sel + (size_t)r * p->G * p->topk, NULL);
    if (e) {
#pragma omp atomic write
      rc = e;
    }
  }
  return rc;
}

static int batched_attn(const msa_ref_dims *p, int B, int T, int max_blocks, const uint16_t *q,
                        const uint16_t *k, const uint16_t *v, const int32_t *sel,
                        const int32_t *q_start, const int32_t *kv_len, double *out, int nthreads,
                        int dense) {
  if (!batch_ok(p, B, T, max_blocks, q_start, kv_len) || !q || !k || !v || !out) return -1;
  if (!dense && !sel) return -1;
  const size_t seq = (size_t)max_blocks * p->block * p->G * p->D;
  int rc = 0;
  const int64_t n = (int64_t)B * T;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1)
  for (int64_t r = 0; r < n; ++r) {
    const int b = (int)(r / T), i = (int)(r % T);
    const int64_t t = (int64_t)q_start[b] + i;
    const uint16_t *qt = q + (size_t)r * p->H * p->D;
    double *ot = out + (size_t)r * p->H * p->D;
    int e = dense ? msa_ref_dense(p, t, qt, k + (size_t)b * seq, v + (size_t)b * seq, ot)
                  : msa_ref_attend(p, t, qt, k + (size_t)b * seq, v + (size_t)b * seq,
                                   sel + (size_t)r * p->G * p->topk, ot);
    if (e) {
#pragma omp atomic write
      rc = e;
    }
  }
  return rc;
}

int msa_ref_sparse_attn(const msa_ref_dims *p, int B, int T, int max_blocks, const uint16_t *q,
                        const uint16_t *k, const uint16_t *v, const int32_t *sel,
                        const int32_t *q_start, const int32_t *kv_len, double *out, int nthreads) {
  return batched_attn(p, B, T, max_blocks, q, k, v, sel, q_start, kv_len, out, nthreads, 0);
}

int msa_ref_dense_attn(const msa_ref_dims *p, int B, int T, int max_blocks, const uint16_t *q,
                       const uint16_t *k, const uint16_t *v, const int32_t *q_start,
                       const int32_t *kv_len, double *out, int nthreads) {
  return batched_attn(p, B, T, max_blocks, q, k, v, NULL, q_start, kv_len, out, nthreads, 1);
}

int msa_ref_index_kl_batch(const msa_ref_dims *p, int B, int T, int max_blocks,
                           const uint16_t *q_idx, const uint16_t *k_idx, const uint16_t *q,
                           const uint16_t *k, const int32_t *sel, const int32_t *q_start,
                           const int32_t *kv_len, double *kl, double *dq_idx, double *dk_idx,
                           int nthreads) {
  if (!batch_ok(p, B, T, max_blocks, q_start, kv_len) || !q_idx || !k_idx || !q || !k || !sel ||
      !kl || !dq_idx || !dk_idx)
    return -1;
  const size_t cap = (size_t)max_blocks * p->block;
  const size_t seq = cap * p->G * p->D;
  int rc = 0;
  const int64_t n = (int64_t)B * T;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1)
  for (int64_t r = 0; r < n; ++r) {
    const int b = (int)(r / T), i = (int)(r % T);
    int e = msa_ref_index_kl(p, (int64_t)q_start[b] + i, q_idx + (size_t)r * p->G * p->Di,
                             k_idx + (size_t)b * cap * p->Di, q + (size_t)r * p->H * p->D,
                             k + (size_t)b * seq, sel + (size_t)r * p->G * p->topk,
                             kl + (size_t)r * p->G, dq_idx + (size_t)r * p->G * p->Di,
                             dk_idx + (size_t)b * cap * p->Di);
    if (e) {
#pragma omp atomic write
      rc = e;
    }
  }
  return rc;
}
