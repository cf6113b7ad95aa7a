/* MSA CPU oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, double-precision restatement of what the MiniMax Sparse
 * Attention (MSA) forward pass computes, written from the description in
 * "MiniMax 模型迭代与竞品分析：从 Text-01、M1、M2 到 M3", section 2
 * ("从 Lightning Attention 到 MSA"): the full-attention equation and the four
 * inference steps (global index scoring, 128-token max pooling, top-16 with
 * the local block forced in, exact softmax over the selected blocks).
 *
 * Only tests, the smoke check and the benchmark's CPU-baseline leg may load
 * this library.  It shares no code with the CUDA path.
 *
 * Tensors are bf16 bit patterns (uint16_t) in the library's layouts:
 *   q_idx [B][T][G][Di]     k_idx [B][cap][Di]      (cap = max_blocks*block)
 *   q     [B][T][H][D]      k, v  [B][max_blocks][block][G][D]
 *   sel   [B][T][G][topk]   ascending block ids, -1 padded
 *   out   [B][T][H][D]      double
 * Query i of sequence b sits at absolute position t = q_start[b] + i.
 */
#ifndef MSA_REF_H
#define MSA_REF_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int H;         /* query heads                                  */
  int G;         /* GQA groups = KV heads; heads of group g are  */
                 /* [g*H/G, (g+1)*H/G)                           */
  int D;         /* head dim of q, k, v                          */
  int Di;        /* index dim of q_idx, k_idx                    */
  int block;     /* tokens per KV block (128)                    */
  int topk;      /* blocks selected per (query, group) (16)      */
  double scale;  /* main-branch softmax scale (1/sqrt(D))        */
} msa_ref_dims;

/* Status: 0 ok, -1 bad argument. */

/* Index branch for one query at absolute position t of one sequence.
 * q_idx_t [G][Di]; k_idx [>= t+1][Di]; sel_t [G][topk] (output).
 * pooled (optional, may be NULL): [G][t/block] pooled scores of the
 * candidate blocks. */
int msa_ref_select(const msa_ref_dims *p, int64_t t, const uint16_t *q_idx_t,
                   const uint16_t *k_idx, int32_t *sel_t, double *pooled);

/* Main branch for one query: exact softmax attention of every head over the
 * tokens of its group's selected blocks that are <= t.
 * q_t [H][D]; k, v [nblocks][block][G][D]; sel_t [G][topk]; out_t [H][D]. */
int msa_ref_attend(const msa_ref_dims *p, int64_t t, const uint16_t *q_t,
                   const uint16_t *k, const uint16_t *v, const int32_t *sel_t,
                   double *out_t);

/* Dense causal GQA attention for one query over all tokens <= t (no
 * selection); the special case MSA must reduce to when t < topk*block. */
int msa_ref_dense(const msa_ref_dims *p, int64_t t, const uint16_t *q_t,
                  const uint16_t *k, const uint16_t *v, double *out_t);

/* Selection quality of one query (the evaluation the same section asks for:
 * how much of the attention the selected blocks recall).  For every head h
 * of every group g, with alpha_h the full causal softmax over all tokens
 * <= t (no selection) and A_h(b) = sum of alpha_h over the tokens of block b:
 *   coverage[h]      = sum of A_h(b) over the distinct valid ids b in sel_t[g]
 *   best_coverage[h] = sum of A_h(b) over b in dense_sel[g]
 *   dense_sel[g]     = the selection a perfect indexer would make under the
 *                      same rule: the local block lb plus the top
 *                      min(16, lb+1) - 1 blocks b < lb by the group-averaged
 *                      mass P_g(b) = mean over the group's heads of A_h(b)
 *                      (ties to the lower id), ascending, -1 padded
 *   hits[g]          = |sel_t[g] intersected with dense_sel[g]|
 * Selection recall is hits[g] / min(16, lb+1).  mass (optional, may be NULL):
 * [G][lb+1] receives P_g(b).  sel_t [G][topk]; q_t [H][D]; k as in attend. */
int msa_ref_quality(const msa_ref_dims *p, int64_t t, const uint16_t *q_t,
                    const uint16_t *k, const int32_t *sel_t, double *coverage,
                    double *best_coverage, int32_t *dense_sel, int32_t *hits,
                    double *mass);

/* Training signal of the index branch for one query ("MiniMax 模型迭代与竞品
 * 分析" section 2, the paragraph on how the indexer learns to select): over
 * the candidate blocks C = the distinct valid ids of sel_t[g],
 *   P_j  = mean over the group's heads of the main branch's softmax mass on
 *          block j (the sparse softmax over the selected tokens <= t);
 *          a target: no gradient flows into it
 *   z_j  = the block's pooled index score, max over its tokens <= t of
 *          <Q_idx[t,g], K_idx[tok]>, attained first at token a_j
 *   Q_j  = exp(z_j) / sum over C of exp(z_c)
 *   kl[g] = sum over C of P_j (ln P_j - ln Q_j)      (terms with P_j = 0 vanish)
 * and its gradient: dz_j = Q_j - P_j, so
 *   dq_idx[g][d]  = sum_j dz_j K_idx[a_j][d]              (written)
 *   dk_idx[a_j][d] += dz_j Q_idx[t,g][d]                  (accumulated)
 * q_idx_t [G][Di]; k_idx [>= t+1][Di]; q_t [H][D]; k as in attend; sel_t
 * [G][topk]; kl [G]; dq_idx [G][Di]; dk_idx [>= t+1][Di] (double). */
int msa_ref_index_kl(const msa_ref_dims *p, int64_t t, const uint16_t *q_idx_t,
                     const uint16_t *k_idx, const uint16_t *q_t, const uint16_t *k,
                     const int32_t *sel_t, double *kl, double *dq_idx, double *dk_idx);

/* Batched forms over the library layouts, OpenMP over queries when
 * nthreads > 1.  kv_len[b] bounds the causal context: q_start[b] + T <=
 * kv_len[b] <= max_blocks*block. */
int msa_ref_index_topk(const msa_ref_dims *p, int B, int T, int max_blocks,
                       const uint16_t *q_idx, const uint16_t *k_idx,
                       const int32_t *q_start, const int32_t *kv_len,
                       int32_t *sel, int nthreads);

int msa_ref_sparse_attn(const msa_ref_dims *p, int B, int T, int max_blocks,
                        const uint16_t *q, const uint16_t *k, const uint16_t *v,
                        const int32_t *sel, const int32_t *q_start,
                        const int32_t *kv_len, double *out, int nthreads);

/* msa_ref_index_kl for every query of a batch: kl [B][T][G], dq_idx
 * [B][T][G][Di] written, dk_idx [B][max_blocks*block][Di] accumulated. */
int msa_ref_index_kl_batch(const msa_ref_dims *p, int B, int T, int max_blocks,
                           const uint16_t *q_idx, const uint16_t *k_idx,
                           const uint16_t *q, const uint16_t *k, const int32_t *sel,
                           const int32_t *q_start, const int32_t *kv_len, double *kl,
                           double *dq_idx, double *dk_idx, int nthreads);

int msa_ref_dense_attn(const msa_ref_dims *p, int B, int T, int max_blocks,
                       const uint16_t *q, const uint16_t *k, const uint16_t *v,
                       const int32_t *q_start, const int32_t *kv_len,
                       double *out, int nthreads);

#ifdef __cplusplus
}
#endif
#endif
