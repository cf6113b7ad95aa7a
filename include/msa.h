/* msa.h -- C ABI of libmsa: the MiniMax Sparse Attention (MSA) forward pass on
 * one GB300 (sm_103a).
 *
 * What is computed ("MiniMax 模型迭代与竞品分析：从 Text-01、M1、M2 到 M3",
 * section 2 "从 Lightning Attention 到 MSA", inference steps 1-4):
 *   1. per GQA group g, a light index query Q_idx[t,g] is scored against the
 *      index key K_idx[i] that all groups share, for every causal token i;
 *   2. token scores are max-pooled into 128-token KV blocks;
 *   3. 16 blocks are selected per (query, group), the query's own (local)
 *      block lb = t/128 forced in as one of the 16;
 *   4. every query head of the group runs exact softmax attention
 *      (s = q.k * scale, softmax over the attended tokens, o = sum p v; the
 *      full-attention equation of the same section) over the tokens <= t of
 *      the selected blocks only, at most 16*128 = 2048 tokens.
 * The KV cache is block-major, block -> token -> head -> dim
 * ("前沿架构解码手记（三）：MiniMax M2.7 → M3", section 2.1 "KV-Block-Major").
 *
 * Readings fixed by this library where the pages are silent: the index score
 * is the raw dot product (no scale, no activation), ranked without exp; ties
 * between equal pooled scores go to the lower block id; with fewer than 16
 * causal blocks all lb+1 are selected; selected ids are written ascending
 * and padded with -1; one softmax spans all selected tokens of a head.
 *
 * Conventions for every entry point:
 *   - bf16 tensors are passed as uint16_t bit patterns in DEVICE memory that
 *     the caller owns; layouts are row-major, innermost index last:
 *       q_idx   [B][T][G][Di]           k_idx   [B][max_blocks*128][Di]
 *       q, out  [B][T][H][D]            k_cache, v_cache [B][max_blocks][128][G][D]
 *       sel     [B][T][G][16] int32     (device)
 *     Query head h belongs to group g = h / (H/G) and reads KV head g.
 *   - q_start and kv_len are HOST arrays of B int32: query i of sequence b
 *     sits at absolute position q_start[b] + i, and the causal context of
 *     sequence b is its first kv_len[b] tokens.  Required:
 *     0 <= q_start[b], q_start[b] + T <= kv_len[b] <= max_blocks*128.
 *     Prefill: q_start = 0, kv_len = T.  Chunked prefill: q_start = chunk
 *     start.  Decode: T = 1, q_start = kv_len - 1 (the new token's K, V and
 *     K_idx are already in the caches: msa_cache_append writes them).
 *   - ws is caller-owned device scratch of at least msa_workspace_bytes(p)
 *     bytes, 256-byte aligned.  The library never allocates memory and keeps
 *     no state between calls except a status word inside ws.
 *   - Work is enqueued asynchronously on `stream`; nothing synchronises.
 *     Inputs must stay valid until the stream reaches the call's end.  The
 *     calls enqueue only kernels and memsets, so a caller may capture them
 *     into a CUDA graph and replay it (a graph holds the pointers, sizes and
 *     positions of the captured call).
 *   - Every entry point returns MSA_OK or a negative msa_status.  Argument
 *     errors are found on the host before anything is enqueued.  A kernel
 *     whose bounded wait runs out records MSA_ERR_TIMEOUT in ws; read it with
 *     msa_workspace_status().
 *   - Supported shapes: block == 128, topk == 16, H % G == 0, D in {64, 128},
 *     Di in {32, 64}, 1 <= B <= MSA_MAX_BATCH, T >= 0 (T == 0 is a no-op),
 *     G <= 8, H/G <= 16, max_blocks <= 32768, and B*T*H and
 *     B*max_blocks*128 below 2^31 (tensor-copy row coordinates are 32-bit).
 *     Others return MSA_ERR_UNSUPPORTED.
 *   - Pointers must be 16-byte aligned (MSA_ERR_INVALID_ARG otherwise).
 */
#ifndef MSA_H
#define MSA_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MSA_BLOCK 128
#define MSA_TOPK 16
#define MSA_MAX_BATCH 256
#define MSA_NOALLOC_SCRATCH_BYTES (16u << 20)

typedef enum {
  MSA_OK = 0,
  MSA_ERR_INVALID_ARG = -1, /* null/misaligned pointer, inconsistent sizes    */
  MSA_ERR_UNSUPPORTED = -2, /* a shape outside the supported set              */
  MSA_ERR_WORKSPACE = -3,   /* ws too small                                   */
  MSA_ERR_CUDA = -4,        /* a CUDA launch or driver call failed            */
  MSA_ERR_TIMEOUT = -5      /* a kernel's bounded wait ran out (read from ws) */
} msa_status;

/* Which kernels run the prefill steps.  MSA_KERNELS_AUTO picks by shape: the
 * tensor-core (tcgen05) index scan and KV-outer attention for prefill-sized
 * T, the per-query streaming kernels for decode-sized T.  The two forced
 * values exist so that tests can exercise both families on any shape. */
typedef enum {
  MSA_KERNELS_AUTO = 0,
  MSA_KERNELS_STREAMING = 1,
  MSA_KERNELS_TENSORCORE = 2
} msa_kernels;

typedef struct {
  int B;          /* sequences in the call                                  */
  int T;          /* query tokens per sequence in the call                  */
  int H;          /* query heads                                            */
  int G;          /* GQA groups = KV heads                                  */
  int D;          /* head dim of q, k, v                                    */
  int Di;         /* index dim of q_idx, k_idx                              */
  int block;      /* tokens per KV block, must be MSA_BLOCK                 */
  int topk;       /* blocks per (query, group), must be MSA_TOPK            */
  int max_blocks; /* block capacity of each sequence's caches               */
  float scale;    /* main-branch softmax scale, normally 1/sqrt(D)          */
  int kernels;    /* an msa_kernels value                                   */
} msa_params;

/* Bytes of device scratch the entry points need for these params (the
 * maximum over msa_index_topk, msa_sparse_attn and msa_forward). */
size_t msa_workspace_bytes(const msa_params *p);

/* Steps 1-3.  Writes sel[B][T][G][16]: the selected block ids of each
 * (query, group), ascending, -1 padded; always min(16, lb+1) ids including
 * lb.  Index scores accumulate in fp32; they are exact when Q_idx and K_idx
 * products and sums fit fp32 exactly (e.g. values on a 2^-3 grid). */
int msa_index_topk(const msa_params *p, const uint16_t *q_idx, const uint16_t *k_idx,
                   const int32_t *q_start, const int32_t *kv_len, int32_t *sel,
                   void *ws, size_t ws_bytes, cudaStream_t stream);

/* Step 4 for a caller-given selection sel[B][T][G][16] (ids ascending or
 * not, -1 entries ignored, every id in [0, lb]).  Writes out[B][T][H][D]
 * bf16 (round to nearest even) from fp32 accumulation. */
int msa_sparse_attn(const msa_params *p, const uint16_t *q, const uint16_t *k_cache,
                    const uint16_t *v_cache, const int32_t *sel, const int32_t *q_start,
                    const int32_t *kv_len, uint16_t *out, void *ws, size_t ws_bytes,
                    cudaStream_t stream);

/* Steps 1-4.  sel_out may be NULL (the selection then lives in ws). */
int msa_forward(const msa_params *p, const uint16_t *q_idx, const uint16_t *k_idx,
                const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                const int32_t *q_start, const int32_t *kv_len, int32_t *sel_out,
                uint16_t *out, void *ws, size_t ws_bytes, cudaStream_t stream);

/* ---- Paged caches --------------------------------------------------------
 * "前沿架构解码手记（三）：MiniMax M2.7 → M3", section 2.1 ("KV-Block-Major
 * Prefill") keeps the KV cache block -> token -> head -> dim so that every
 * block a query selects is one contiguous run, and names this layout as what
 * lets paged serving engines run MSA unchanged.  Here the pages of such an
 * engine are exactly MSA's 128-token blocks: the K, V and K_idx of all
 * sequences live in pools of num_pool_blocks blocks,
 *     k_pool, v_pool  [num_pool_blocks][128][G][D]     bf16
 *     k_idx_pool      [num_pool_blocks][128][Di]       bf16
 * and block_table[B][max_blocks] (device int32) maps logical block kb of
 * sequence b (its tokens kb*128 .. kb*128+127) to a pool block.  Entries of
 * blocks a call never reaches are not read.  An entry that is read and lies
 * outside [0, num_pool_blocks) is not dereferenced: the kernels record
 * MSA_ERR_INVALID_ARG in ws (msa_workspace_status) and use zeros instead.
 * num_pool_blocks * 128 must stay below 2^31 - 128 (MSA_ERR_UNSUPPORTED). */

/* Appends p->T new tokens to every sequence's caches: the token of row i of
 * sequence b goes to position q_start[b] + i (host array), i.e. row
 * (q_start[b] + i) % 128 of logical block (q_start[b] + i) / 128.
 *   k_new, v_new [B][T][G][D] bf16, k_idx_new [B][T][Di] bf16 (device)
 * block_table NULL: the caches are per sequence (msa_forward's layout,
 * [B][max_blocks][128][...]) and num_pool_blocks is ignored; otherwise they
 * are the pools above.  Requires 0 <= q_start[b], q_start[b] + T <=
 * max_blocks * 128.  ws: at least 256 bytes of device scratch (256-byte
 * aligned) that receives the status word.  Only the rows written change. */
int msa_cache_append(const msa_params *p, const int32_t *block_table, int num_pool_blocks,
                     const uint16_t *k_new, const uint16_t *v_new, const uint16_t *k_idx_new,
                     const int32_t *q_start, uint16_t *k_cache, uint16_t *v_cache,
                     uint16_t *k_idx_cache, void *ws, size_t ws_bytes, cudaStream_t stream);

/* msa_forward over paged caches: the same steps, arguments and results, with
 * k_idx, k_cache and v_cache replaced by the pools and every cache block read
 * through block_table (both kernel families).  ws as for msa_forward
 * (msa_workspace_bytes(p)).  Decode appends the new token first
 * (msa_cache_append), then calls this with q_start = kv_len - 1. */
int msa_forward_paged(const msa_params *p, const int32_t *block_table, int num_pool_blocks,
                      const uint16_t *q_idx, const uint16_t *k_idx_pool, const uint16_t *q,
                      const uint16_t *k_pool, const uint16_t *v_pool, const int32_t *q_start,
                      const int32_t *kv_len, int32_t *sel_out, uint16_t *out, void *ws,
                      size_t ws_bytes, cudaStream_t stream);

/* msa_index_topk for callers that cannot allocate device memory.  The pages
 * have no counterpart: this is a deployment variant of steps 1-3, not part
 * of the method.
 *
 * Some callers cannot call cudaMalloc: a serving engine that gives all free
 * GPU memory to its KV-cache pool at start-up and forbids later allocations,
 * or a plugin host that passes the library nothing but its input and output
 * buffers.  Such callers cannot supply the workspace msa_index_topk takes.
 * This entry point takes none and allocates nothing (no cudaMalloc, no
 * cudaFree, no allocating library call): its scratch is a static device
 * array of MSA_NOALLOC_SCRATCH_BYTES bytes inside the library, which every
 * GPU that loads the library holds until the process exits.
 *   - Same arguments and results as msa_index_topk (sel is bit-identical),
 *     minus ws/ws_bytes, except that p->kernels is ignored: this entry point
 *     always runs the streaming (per-query) index kernels, whichever family
 *     p->kernels names.  The stream must belong to the current device.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current, and remembers it with
 *     the id of the current CUDA context; a call under another context of
 *     that device (after cudaDeviceReset, for example) looks it up again.
 *     Make the first call on a device (and the first after a reset) before
 *     any stream capture.
 *   - Returns MSA_ERR_WORKSPACE when the call would need more scratch than
 *     MSA_NOALLOC_SCRATCH_BYTES (B*T*ceil(max lb/64)*G*15*8 bytes, splits
 *     capped at 128), MSA_ERR_UNSUPPORTED when B*T > 65535.
 *   - Every call shares the one array and leaves its contents behind; each
 *     call writes every scratch entry it reads, so nothing needs clearing.
 *     Calls that overlap on the GPU (other streams, other host threads) race
 *     on the array: the caller must serialise them. */
int msa_index_topk_noalloc(const msa_params *p, const uint16_t *q_idx, const uint16_t *k_idx,
                           const int32_t *q_start, const int32_t *kv_len, int32_t *sel,
                           cudaStream_t stream);

/* Dense causal GQA attention over the same block-major caches: every query
 * head attends every token <= t of its group's KV head (the full-attention
 * equation of "MiniMax 模型迭代与竞品分析" section 2, without selection).
 * M3 keeps its first three layers dense (section 3 of the same page:
 * sparse_attention_freq starts with three zeros), so a model built on this
 * library runs those layers here, on the caches its MSA layers use.
 * Prefill-sized calls (the tensor-core choice of msa_sparse_attn) run one
 * query-outer tensor-core kernel: 128 queries of a head pair at a time over
 * every causal block, an online softmax with the output kept on chip.  Other
 * calls process the blocks in chunks of 16 through the streaming attention,
 * each chunk folded into fp32 running (output, max, sum) accumulators.  out
 * is bf16 (round to nearest even).  Arguments as for msa_sparse_attn without
 * sel; ws of at least msa_dense_workspace_bytes(p) bytes, 256-byte aligned
 * (the status word; for the streaming calls also B*T*H*(D+2) fp32
 * accumulators and the attention scratch). */
size_t msa_dense_workspace_bytes(const msa_params *p);
int msa_dense_attn(const msa_params *p, const uint16_t *q, const uint16_t *k_cache,
                   const uint16_t *v_cache, const int32_t *q_start, const int32_t *kv_len,
                   uint16_t *out, void *ws, size_t ws_bytes, cudaStream_t stream);

/* The index branch's training signal ("MiniMax 模型迭代与竞品分析" section 2,
 * the paragraph on how the indexer learns to select): over the candidate
 * blocks C of each (query, group) -- the distinct ids of sel in [0, lb] --
 *   P_j  the main branch's softmax mass on block j (the sparse softmax over
 *        the selected tokens <= t), averaged over the group's heads; the
 *        teacher, so no gradient flows into q or k_cache
 *   z_j  the block's pooled index score, max over its tokens <= t of
 *        <Q_idx, K_idx[tok]>, first attained at token a_j
 *   Q_j  exp(z_j) / sum over C of exp(z_c)      (the student)
 * Outputs (fp32, device, caller-owned):
 *   kl[B][T][G]          D_KL(P || Q) = sum_j P_j (ln P_j - ln Q_j)
 *   dq_idx[B][T][G][Di]  the gradient of the summed loss with respect to Q_idx:
 *                        sum_j (Q_j - P_j) K_idx[a_j]            (written)
 *   dk_idx[B][max_blocks*128][Di]  its gradient with respect to K_idx:
 *                        (Q_j - P_j) Q_idx added at row a_j with atomic adds
 *                        (accumulated: the caller zeroes it first)
 * Pooled scores accumulate in fp32, exact for inputs on a 2^-3 grid.  ws: at
 * least msa_index_kl_workspace_bytes(p) bytes, 256-byte aligned. */
size_t msa_index_kl_workspace_bytes(const msa_params *p);
int msa_index_kl(const msa_params *p, const uint16_t *q_idx, const uint16_t *k_idx,
                 const uint16_t *q, const uint16_t *k_cache, const int32_t *sel,
                 const int32_t *q_start, const int32_t *kv_len, float *kl, float *dq_idx,
                 float *dk_idx, void *ws, size_t ws_bytes, cudaStream_t stream);

/* Selection quality: how much of the attention a selection recalls, the
 * evaluation the same section asks for when it names the indexer's recall as
 * MSA's risk (a block the indexer misses cannot be read by the main branch).
 * For every (query, group) of the call, with A_h(b) the mass of block b (its
 * tokens <= t) under head h's FULL causal softmax over tokens 0..t:
 *   coverage[B][T][H]       sum of A_h(b) over the distinct ids of sel[b,t,g]
 *                           that lie in [0, lb] (others are ignored)
 *   dense_sel[B][T][G][16]  the ideal selection under the same rule: lb plus
 *                           the top min(16, lb+1)-1 blocks b < lb by the
 *                           group-averaged mass P(b) = mean over the group's
 *                           heads of A_h(b), ties to the lower id; ascending,
 *                           -1 padded
 *   best_coverage[B][T][H]  sum of A_h(b) over dense_sel
 *   hits[B][T][G]           |sel intersected with dense_sel|; selection recall
 *                           is hits / min(16, lb+1)
 * coverage and best_coverage are fp32 (scores of the bf16 inputs accumulate
 * in fp32); all four outputs are caller-owned device memory.  q, k_cache, sel,
 * q_start and kv_len are as in msa_sparse_attn.  ws: device scratch of at
 * least msa_quality_workspace_bytes(p) bytes, 256-byte aligned (it scales
 * with min(64, B*T) rows x G x max_blocks x (H/G + 1) x 8 bytes).  The cost
 * is that of dense attention scores over the whole context: meant for
 * sampled queries, not for every query of a long prefill. */
size_t msa_quality_workspace_bytes(const msa_params *p);
int msa_selection_quality(const msa_params *p, const uint16_t *q, const uint16_t *k_cache,
                          const int32_t *sel, const int32_t *q_start, const int32_t *kv_len,
                          float *coverage, float *best_coverage, int32_t *dense_sel,
                          int32_t *hits, void *ws, size_t ws_bytes, cudaStream_t stream);

/* Waits for `stream`, then returns the status the last call on ws left in
 * it: MSA_OK; MSA_ERR_TIMEOUT if a kernel's bounded wait ran out (its
 * outputs are then incomplete; this takes precedence over the next case);
 * MSA_ERR_INVALID_ARG if msa_sparse_attn met a selected id outside [0, lb]
 * or beyond max_blocks (that id was skipped, never read).  MSA_ERR_CUDA if
 * the read itself fails. */
int msa_workspace_status(const void *ws, cudaStream_t stream);

/* A static, human-readable name of a status code. */
const char *msa_status_string(int status);

/* Diagnostics: the number of kernels this library has enqueued since it was
 * loaded (all threads, all devices).  Benchmarks read it before and after a
 * timed region to count the launches inside it. */
uint64_t msa_kernel_launch_count(void);

/* Diagnostics, for tests of the failure path only (the pages have no
 * counterpart).  Every wait of a tensor-core kernel's pipeline (a stage
 * awaited from another warp: a copy landing, an MMA done, a buffer freed) is
 * bounded by 2 s of wall-clock time; on expiry the kernel records
 * MSA_ERR_TIMEOUT in ws, stops issuing work, waits for the copies and MMAs it
 * already issued (these waits keep the 2 s bound alone, so nothing lands in
 * shared memory after the CTA exits and tensor memory is always released)
 * and exits.  With polls > 0, each pipeline wait also gives up after `polls`
 * unsuccessful polls, so that a test can make the timeout happen on a correct
 * kernel; 0 (the default) restores the wall-clock bound alone.  Applies to
 * launches made after the call, from any thread; not for production use. */
void msa_debug_set_wait_polls(uint32_t polls);

#ifdef __cplusplus
}
#endif
#endif /* MSA_H */
