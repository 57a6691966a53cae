/*
 * msa.h -- C ABI of the GB300 (sm_103a) block-sparse GQA decode library.
 *
 * One decode step of indexer-selected block-sparse attention over a paged fp8
 * KV cache, as the vLLM MiniMax-M3 sparse attention pages and the
 * TensorRT-LLM PR #17171 "Custom decode kernels for MinimaxM3" describe it:
 *
 *   msa_score          each block's largest visible scaled q.k over the
 *                      query heads of its KV head              (stage 1)
 *   msa_topk           top-16 block selection                  (stage 2)
 *   msa_sparse_decode  split-K attention over the selected pages (stage 3)
 *   msa_combine        merge of the split-K partials            (stage 4)
 *   msa_sparse_decode_select  stages 2 and 3 in one kernel
 *   msa_dense_decode   attention over every visible block (dense layers)
 *   msa_sparse_prefill(_select)  the attend for prefill and chunked-prefill
 *                      batches: one query length per request (cu_seqlens_q)
 *   msa_score_kcache   stage 1 on a separate K-only (index-K) cache
 *   msa_*_q8           the same with an fp8 query and a per-tensor q_scale
 *   msa_decode_step    stages 1-4 of one step in one call
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor arguments are raw DEVICE pointers to memory the caller owns
 *    and keeps alive until the work enqueued on `stream` has finished.  The
 *    library allocates nothing and keeps no reference after returning.
 *  - Every call only enqueues work on `stream` (a cudaStream_t; NULL is the
 *    legacy default stream) and returns without waiting.  No call
 *    synchronises the host except msa_get_error.
 *  - Stream order: by default each call's work starts only after all work
 *    enqueued earlier on `stream` has completed, so its inputs may be written
 *    by any kernel or copy just before it.  Inside one call (and inside
 *    msa_decode_step) a library kernel may start while the library kernel
 *    before it finishes (programmatic dependent launch); it reads that
 *    kernel's outputs only after it has completed.  msa_set_input_overlap
 *    lets the first kernel of every call overlap the previous kernel too
 *    (see there).
 *  - Sizes: B requests, Q = decode_query_len query tokens per request,
 *    T = B*Q query tokens ordered request-major (token i = b*Q + j; the
 *    prefill entry points take T and cu_seqlens_q instead of Q),
 *    Hq query heads and Hkv KV heads with Hq = 16 * Hkv (query head h belongs
 *    to KV head g = h / 16), head size 128, page size 128 tokens, S = the
 *    block_table row stride (max logical blocks per request), num_blocks =
 *    physical pages in the cache.
 *  - Causal offset: query token j of request b sits at position
 *    pos = seq_lens[b] - Q + j and may see cache tokens 0..pos; its current
 *    block is cur = pos / 128.  A token with pos < 0 is a padding row.
 *  - Layouts (all contiguous, row-major):
 *      q           bf16  [T, Hq, 128]
 *      kv          fp8 e4m3 (OCP "fn") bytes [num_blocks, Hkv, 128, 256]:
 *                  per page and KV head, 128 token rows of 256 bytes, K in
 *                  bytes 0..127 and V in bytes 128..255 (the packed HND cache
 *                  of MiniMaxM3SparseBackend.get_kv_cache_shape)
 *      block_table int32 [B, S]; entry [b, n] = physical page of logical block n
 *      seq_lens    int32 [B]
 *      scores      fp32  [Hkv, T, S] (msa_score output)
 *      topk        int32 [T, Hkv, 16], -1 = unused slot
 *      out         bf16  [T, Hq, 128]
 *  - Return value: MSA_OK, or an MSA_E* code when the call was rejected on
 *    the host (nothing was enqueued) or a CUDA call failed.
 *  - Bad indices found on the device (see MSA_ERR_*) never trap: the bad
 *    entry is skipped and a bit is set in a per-device sticky error word that
 *    msa_get_error reads.
 */
#ifndef MSA_H
#define MSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, so callers need no CUDA header to use this one. */
typedef struct CUstream_st *msa_stream_t;

/* ---- status codes ------------------------------------------------------- */
#define MSA_OK 0
#define MSA_EINVAL 1  /* bad size, null or misaligned pointer: rejected on host */
#define MSA_ECUDA 3   /* a CUDA runtime call failed (no device, launch error)  */
#define MSA_ENOSPC 4  /* workspace smaller than msa_workspace_bytes()          */

/* ---- bits of the device error word (msa_get_error) ---------------------- */
#define MSA_ERR_TOPK_RANGE 0x01u  /* top-k entry not -1 and outside [0, cur]          */
#define MSA_ERR_TOPK_DUP 0x02u    /* a block listed twice for one (token, KV head)    */
#define MSA_ERR_PAGE_RANGE 0x04u  /* block_table entry outside [0, num_blocks)        */
#define MSA_ERR_SEQ_RANGE 0x08u   /* seq_lens[b] < 0 or ceil(seq_lens[b]/128) > S     */
#define MSA_ERR_SCORE_NAN 0x10u   /* msa_topk read a NaN score (ranked as -inf)       */
#define MSA_ERR_TIMEOUT 0x20u     /* a bounded wait for an async copy expired         */

/* ---- fixed geometry ----------------------------------------------------- */
#define MSA_HEAD_DIM 128
#define MSA_PAGE_SIZE 128
#define MSA_TOPK 16
#define MSA_GROUP 16      /* query heads per KV head */
#define MSA_MAX_QLEN 32

/*
 * msa_score -- stage 1, the block scorer.
 *
 * Defined by the scorer commit of TensorRT-LLM PR #17171 (each block's
 * largest q.k under the causal mask, stored head-major, then token, then
 * block): for every KV head g, query token i and logical block n < S,
 *
 *   scores[g, i, n] = max over query heads h of group g and over tokens t of
 *                     block n with 128*n + t <= pos(i) of
 *                     sm_scale * k_scale * sum_d q[i,h,d] * K8[page(b,n),g,t,d]
 *
 * where K8 is the fp8 key as stored (the cache's K half).  Blocks n > cur(i)
 * and every block of a padding row get -inf.  The whole [Hkv, T, S] buffer is
 * written.  sm_scale > 0 and k_scale > 0 (both finite) are required.
 * Numerics: the fp8 key tile is a tensor-core operand as stored; each (token,
 * KV head)'s query rows are scaled by a power of two (largest magnitude in
 * [2^7, 2^8)) and carried as the sum of two fp8 e4m3 parts, which is exact for
 * every element down to 2^-9 of the largest; products accumulate in fp32.
 * Errors: MSA_EINVAL for Q outside 1..32, Hq != 16*Hkv, S < 1, num_blocks < 1,
 * num_blocks*Hkv*128 >= 2^31, null or non-16-byte-aligned q/kv, null
 * block_table/seq_lens/scores.  Device: MSA_ERR_PAGE_RANGE (block scored
 * -inf), MSA_ERR_SEQ_RANGE (request treated as empty).
 */
int msa_score(const void *q, const void *kv, const int32_t *block_table,
              const int32_t *seq_lens, float *scores, int B, int Q, int Hq, int Hkv,
              int S, int64_t num_blocks, float sm_scale, float k_scale,
              msa_stream_t stream);

/*
 * msa_score_kcache -- msa_score reading the keys from a K-only cache: the
 * "index-K sub-pages" that the TensorRT-LLM dense-decode commit says the
 * MiniMax-M3 cache packs per sparse layer beside the K|V pages.  The pages
 * give that pool no layout; here it is read as fp8 e4m3 [num_blocks, Hkv, 128,
 * 128], each page-head the 16 KiB of one K half of a packed page (token row t
 * at byte offset ((page * Hkv + g) * 128 + t) * 128), addressed through the
 * same block_table and seq_lens, scaled by k_scale.  Everything else (the
 * operation, layouts, numerics and errors) is msa_score's, with k_cache in
 * place of kv; the scores are bit-identical to msa_score's on a packed cache
 * whose K halves hold the same bytes.  msa_score_kcache_q8 takes the fp8
 * query as msa_score_q8 does.
 */
int msa_score_kcache(const void *q, const void *k_cache, const int32_t *block_table,
                     const int32_t *seq_lens, float *scores, int B, int Q, int Hq, int Hkv, int S,
                     int64_t num_blocks, float sm_scale, float k_scale, msa_stream_t stream);
int msa_score_kcache_q8(const void *q8, float q_scale, const void *k_cache,
                        const int32_t *block_table, const int32_t *seq_lens, float *scores,
                        int B, int Q, int Hq, int Hkv, int S, int64_t num_blocks, float sm_scale,
                        float k_scale, msa_stream_t stream);

/*
 * msa_topk -- stage 2, the block selector.
 *
 * The selector of TensorRT-LLM PR #17171 reads the score buffer through
 * arbitrary strides; the kept-block list follows the vLLM test file's
 * _make_topk (ascending block ids, -1 padding).  For each (token i, KV head g)
 * with pos(i) >= 0:
 *   - if cur + 1 <= k every block 0..cur is kept;
 *   - else block cur is kept together with the k-1 best of 0..cur-1 in the
 *     order (score descending, block index ascending).
 * Kept ids are written ascending to topk[i, g, 0..], the rest is -1.  Padding
 * rows get all -1.  scores[g, i, n] is read at
 * scores + g*stride_h + i*stride_t + n*stride_n (element strides, any sign);
 * only n < cur is read.  The choice is exact (ties by index) for the given fp32
 * values; -0.0 ranks equal to +0.0.
 * Errors: MSA_EINVAL for k != 16, Q outside 1..32, Hkv < 1, S < 1, null or
 * misaligned pointers.  Device: MSA_ERR_SEQ_RANGE (row written as padding),
 * MSA_ERR_SCORE_NAN.
 */
int msa_topk(const float *scores, int64_t stride_h, int64_t stride_t, int64_t stride_n,
             const int32_t *seq_lens, int32_t *topk, int B, int Q, int Hkv, int S, int k,
             msa_stream_t stream);

/*
 * Bytes of workspace msa_sparse_decode needs for `num_splits` (0 if
 * num_splits <= 1): fp32 partial outputs [num_splits, T, Hq, 128] followed by
 * fp32 (m, l) pairs [num_splits, T, Hq, 2].  Returns 0 for invalid sizes.
 */
size_t msa_workspace_bytes(int B, int Q, int Hq, int num_splits);

/*
 * Split-K factor the library would pick for a decode step of B requests of Q
 * tokens on a GPU with `sm_count` SMs.  Q = 1: one CTA per (token, KV head),
 * split while those fill less than three quarters of two CTAs per SM.  Q >= 2
 * (the attend over the union of each 4-token tile's lists, one CTA per SM):
 * min(8, sm_count / units) CTAs per (request, tile, KV head) unit, 1 when the
 * units fill the SMs.  Depends on the shape only (never on seq_lens), so a
 * step captured in a CUDA graph keeps a fixed launch shape.  Returns >= 1.
 */
int msa_choose_splits(int B, int Q, int Hkv, int sm_count);

/*
 * msa_sparse_decode -- stage 3 (+ stage 4 when split), the sparse attend.
 *
 * The operation of minimax_m3_sparse_attn_decode and msa_cutlass_sparse_decode
 * on the vLLM pages: for each query row (i, h), g = h / 16, the key set is
 * every token t of every block n listed in topk[i, g, :] (entries -1 skipped)
 * with 128*n + t <= pos(i), and
 *
 *   out[i, h] = sum_t softmax_t(sm_scale * k_scale * q[i,h].K8_t) * v_scale * V8_t
 *
 * with no softcap, sink or output scale (o_scale = 1 on the vLLM page).  An
 * empty key set or a padding row gives exactly 0 (the TensorRT-LLM
 * flash-decoding commit zeroes padding rows instead of writing NaN).
 * Entries may be in any order.  num_splits = 0 lets the library choose
 * (msa_choose_splits); with an effective split count above 1 the partials go
 * to `workspace` and msa_combine is enqueued on `stream` by this call, so
 * `out` is complete when the stream reaches that point either way.
 * Numerics: the fp8 K and V tiles are tensor-core operands as stored; the
 * query, scaled per (token, KV head) by a power of two, is the exact sum of
 * two fp8 e4m3 parts; probabilities P <= 2^8.5 are the sum of two e4m3 parts
 * (about 8 significant bits); fp32 accumulation and softmax, output rounded
 * to bf16 (nearest even).
 * Errors: as msa_score, plus null/misaligned topk or out, v_scale not finite,
 * num_splits < 0 or > 16 (MSA_EINVAL), workspace_bytes too small (MSA_ENOSPC).
 * Device: MSA_ERR_TOPK_RANGE / MSA_ERR_TOPK_DUP / MSA_ERR_PAGE_RANGE (entry
 * skipped), MSA_ERR_SEQ_RANGE (request treated as empty).
 */
int msa_sparse_decode(const void *q, const void *kv, const int32_t *block_table,
                      const int32_t *seq_lens, const int32_t *topk, void *workspace,
                      size_t workspace_bytes, void *out, int B, int Q, int Hq, int Hkv,
                      int S, int64_t num_blocks, float sm_scale, float k_scale,
                      float v_scale, int num_splits, msa_stream_t stream);

/*
 * msa_sparse_decode_select -- stages 2 and 3 in one kernel: each (token, KV
 * head) row's blocks are selected exactly as msa_topk selects them, from
 * `scores` read through the element strides (stride_h, stride_t, stride_n),
 * written to `topk` [T, Hkv, 16], and attended as msa_sparse_decode attends a
 * given list (the split merge enqueued on `stream` when split).  Saves the
 * separate selector launch and the re-read of its output; the selection runs
 * in the attend kernel's prologue, overlapping the previous kernel's tail.
 * Rows of more than 512 candidate blocks are selected from shared memory
 * there, which is slower than msa_topk's register paths (up to 2048): for long
 * contexts msa_topk followed by msa_sparse_decode is the faster pair.
 * Arguments and errors: as msa_topk for the scores and as msa_sparse_decode
 * otherwise (`topk` is an output here).
 */
int msa_sparse_decode_select(const void *q, const void *kv, const int32_t *block_table,
                             const int32_t *seq_lens, const float *scores, int64_t stride_h,
                             int64_t stride_t, int64_t stride_n, int32_t *topk, void *workspace,
                             size_t workspace_bytes, void *out, int B, int Q, int Hq, int Hkv,
                             int S, int64_t num_blocks, float sm_scale, float k_scale,
                             float v_scale, int num_splits, msa_stream_t stream);

/*
 * Split count msa_dense_decode uses for a block-table stride of S blocks:
 * min(16, ceil(S / 16)), each split a range of ceil(S / splits) consecutive
 * blocks.  Returns 0 when S < 1 or a range would exceed 128 blocks (S > 2048,
 * contexts beyond 256k tokens), which msa_dense_decode rejects.  Size its
 * workspace with msa_workspace_bytes(B, Q, Hq, msa_dense_splits(S)).  For
 * Q >= 2 this is the most parts a row is cut into: when the (request,
 * 4-token tile, KV head) units are fewer than the SMs, each unit takes a
 * share of one CTA per SM in proportion to its visible blocks (computed on
 * the device from seq_lens), up to this many; with as many units as SMs,
 * one part each.
 */
int msa_dense_splits(int S);

/*
 * msa_dense_decode -- decode attention over every visible block: the dense
 * layers of the model (the TensorRT-LLM PR #17171 dense-decode commit: the
 * first layers attend the whole page table).  The same operation as
 * msa_sparse_decode with each row's list being all of its blocks 0 .. cur(i)
 * (keys 128 n + t <= pos(i)); no list is read.  Splits as msa_dense_splits;
 * with more than one the partials go to `workspace` (parts a row does not use
 * are marked empty) and the merge is enqueued on `stream`.  Numerics as
 * msa_sparse_decode.
 * Errors: as msa_sparse_decode (topk and num_splits aside), plus S > 2048
 * (MSA_EINVAL).  Device: MSA_ERR_PAGE_RANGE (page skipped), MSA_ERR_SEQ_RANGE.
 */
int msa_dense_decode(const void *q, const void *kv, const int32_t *block_table,
                     const int32_t *seq_lens, void *workspace, size_t workspace_bytes, void *out,
                     int B, int Q, int Hq, int Hkv, int S, int64_t num_blocks, float sm_scale,
                     float k_scale, float v_scale, msa_stream_t stream);

/*
 * fp8 query variants.  The vLLM CUTLASS decode (msa_cutlass_sparse_decode on
 * the vLLM pages) takes the query already quantised: query_fp8 with a
 * per-tensor q_scale_float.  These entry points take that form: `q8` is fp8
 * e4m3 (OCP "fn") [T, Hq, 128] whose value is q8 * q_scale, q_scale finite and
 * > 0; every other argument, the operation, and the errors are those of the
 * bf16 entry point of the same name.  The query tile is the fp8 rows as
 * stored, so the scorer issues half the tensor-core work of the bf16 path
 * (which carries each bf16 query exactly as two fp8 parts).
 */
int msa_score_q8(const void *q8, float q_scale, const void *kv, const int32_t *block_table,
                 const int32_t *seq_lens, float *scores, int B, int Q, int Hq, int Hkv, int S,
                 int64_t num_blocks, float sm_scale, float k_scale, msa_stream_t stream);
int msa_sparse_decode_q8(const void *q8, float q_scale, const void *kv,
                         const int32_t *block_table, const int32_t *seq_lens, const int32_t *topk,
                         void *workspace, size_t workspace_bytes, void *out, int B, int Q, int Hq,
                         int Hkv, int S, int64_t num_blocks, float sm_scale, float k_scale,
                         float v_scale, int num_splits, msa_stream_t stream);
int msa_sparse_decode_select_q8(const void *q8, float q_scale, const void *kv,
                                const int32_t *block_table, const int32_t *seq_lens,
                                const float *scores, int64_t stride_h, int64_t stride_t,
                                int64_t stride_n, int32_t *topk, void *workspace,
                                size_t workspace_bytes, void *out, int B, int Q, int Hq, int Hkv,
                                int S, int64_t num_blocks, float sm_scale, float k_scale,
                                float v_scale, int num_splits, msa_stream_t stream);
int msa_dense_decode_q8(const void *q8, float q_scale, const void *kv,
                        const int32_t *block_table, const int32_t *seq_lens, void *workspace,
                        size_t workspace_bytes, void *out, int B, int Q, int Hq, int Hkv, int S,
                        int64_t num_blocks, float sm_scale, float k_scale, float v_scale,
                        msa_stream_t stream);

/*
 * msa_sparse_prefill -- the sparse attend for prefill and chunked prefill:
 * minimax_m3_sparse_attn on the vLLM pages (MiniMaxM3SparseTritonImpl.forward,
 * the prefill part [nd:] of the batch, with MiniMaxM3SparsePrefillMetadata).
 * B requests with one query length each: request b owns query tokens
 * cu_seqlens_q[b] .. cu_seqlens_q[b + 1] - 1 of the T tokens of q, and they
 * are the last q_len_b = cu_seqlens_q[b + 1] - cu_seqlens_q[b] tokens of its
 * sequence: token j of request b sits at position
 *
 *   pos = context_len_b + j,  context_len_b = seq_lens[b] - q_len_b,
 *
 * so it sees pages 0 .. pos / 128, as the vLLM prefill test counts them.
 * Each token attends the blocks of its own list topk[i, g, :]
 * [T, Hkv, 16] with the causal bound 128*n + t <= pos; the operation, output
 * layout [T, Hq, 128], numerics and device errors are msa_sparse_decode's,
 * which this call equals when every request has the same query length.
 * cu_seqlens_q: int32 [B + 1] on the device, cu_seqlens_q[0] = 0, ascending,
 * cu_seqlens_q[B] = T (read by the kernel only, so it may be written by an
 * earlier kernel on `stream`).  Workspace for num_splits > 1:
 * msa_workspace_bytes(T, 1, Hq, splits); num_splits = 0 chooses
 * msa_choose_splits(T, 1, Hkv, sm_count) (one CTA per token).
 * Errors: as msa_sparse_decode, plus null or misaligned cu_seqlens_q, T < 0
 * or T > INT_MAX / 4, or exactly one of B and T zero (MSA_EINVAL); no query
 * length bound applies.  Device: a token in no request's range (e.g. past
 * cu_seqlens_q[B] < T) or of a request with q_len_b > seq_lens[b] sets
 * MSA_ERR_SEQ_RANGE and its rows are written as 0.  cu_seqlens_q is not
 * checked for order: if it is not ascending, a token is attended as a token
 * of some request whose range holds it, or flagged as above (every read
 * stays within cu_seqlens_q[0 .. B]).
 */
int msa_sparse_prefill(const void *q, const void *kv, const int32_t *block_table,
                       const int32_t *seq_lens, const int32_t *cu_seqlens_q,
                       const int32_t *topk, void *workspace, size_t workspace_bytes, void *out,
                       int B, int T, int Hq, int Hkv, int S, int64_t num_blocks, float sm_scale,
                       float k_scale, float v_scale, int num_splits, msa_stream_t stream);

/*
 * msa_sparse_prefill_select -- msa_sparse_prefill with each (token, KV head)
 * row's top-16 selected inside the kernel from `scores` [Hkv, T, >= S] (any
 * element strides), as msa_sparse_decode_select does for decode: the causal
 * top-k of each query row, with that token's own current block.  `topk`
 * [T, Hkv, 16] is written.  Arguments and errors as msa_sparse_prefill and
 * msa_sparse_decode_select.
 */
int msa_sparse_prefill_select(const void *q, const void *kv, const int32_t *block_table,
                              const int32_t *seq_lens, const int32_t *cu_seqlens_q,
                              const float *scores, int64_t stride_h, int64_t stride_t,
                              int64_t stride_n, int32_t *topk, void *workspace,
                              size_t workspace_bytes, void *out, int B, int T, int Hq, int Hkv,
                              int S, int64_t num_blocks, float sm_scale, float k_scale,
                              float v_scale, int num_splits, msa_stream_t stream);

/* fp8-query prefill (the vLLM prefill test feeds the attend query_fp8 with
 * q_scale): q8 and q_scale as the other _q8 entry points. */
int msa_sparse_prefill_q8(const void *q8, float q_scale, const void *kv,
                          const int32_t *block_table, const int32_t *seq_lens,
                          const int32_t *cu_seqlens_q, const int32_t *topk, void *workspace,
                          size_t workspace_bytes, void *out, int B, int T, int Hq, int Hkv, int S,
                          int64_t num_blocks, float sm_scale, float k_scale, float v_scale,
                          int num_splits, msa_stream_t stream);
int msa_sparse_prefill_select_q8(const void *q8, float q_scale, const void *kv,
                                 const int32_t *block_table, const int32_t *seq_lens,
                                 const int32_t *cu_seqlens_q, const float *scores,
                                 int64_t stride_h, int64_t stride_t, int64_t stride_n,
                                 int32_t *topk, void *workspace, size_t workspace_bytes,
                                 void *out, int B, int T, int Hq, int Hkv, int S,
                                 int64_t num_blocks, float sm_scale, float k_scale, float v_scale,
                                 int num_splits, msa_stream_t stream);

/*
 * msa_combine -- stage 4, merge of split-K partials ("fp32 split-K partials"
 * in the TensorRT-LLM flash-decoding commit).  For row r of T*Hq rows, part s
 * holds m_s (max logit in log2 units), l_s = sum 2^(z*log2(e) - m_s) and the
 * unnormalised o_s = sum 2^(z*log2(e) - m_s) * V (V already times v_scale):
 *
 *   out[r] = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s,  M = max_s m_s,
 *
 * parts with l_s = 0 ignored, and 0 when every part is empty.  `workspace`
 * uses the layout msa_workspace_bytes describes.  num_splits in 1..16.
 */
int msa_combine(const void *workspace, void *out, int T, int Hq, int num_splits,
                msa_stream_t stream);

/*
 * msa_sparse_decode_static -- msa_sparse_decode for callers that cannot
 * allocate device memory.  The vLLM and TensorRT-LLM pages have no counterpart
 * for it; it exists for callers that only hold the step's inputs and outputs:
 * a plugin or operator interface that gives the library no workspace, or a
 * runtime that forbids cudaMalloc on its hot path (an allocation can block on
 * the whole device or fail under memory pressure).
 *
 * Same arguments and result as msa_sparse_decode without the workspace pair.
 * The split-K partials go to one scratch array compiled into the library:
 * MSA_STATIC_SCRATCH_BYTES (4 MiB) of device memory that every GPU loading
 * the library holds until the process exits.  The call allocates nothing
 * (no cudaMalloc, cudaFree or allocating library routine).
 *  - A shape whose partials need more than MSA_STATIC_SCRATCH_BYTES
 *    (msa_workspace_bytes(B, Q, Hq, splits) > MSA_STATIC_SCRATCH_BYTES) is
 *    rejected with MSA_ENOSPC before anything is enqueued; pass a smaller
 *    num_splits (1 needs no scratch) or use msa_sparse_decode.
 *  - The first call on a device that needs the scratch looks up the array's
 *    device address (cudaGetSymbolAddress) with that device current; make
 *    that first call before any stream capture.
 *  - All calls share the one array, and it keeps the last call's contents.
 *    Nothing in it has to start at zero (each call writes every partial it
 *    reads back), but calls whose work overlaps on the GPU, e.g. on two
 *    streams at once, race on the array and give wrong results.
 */
#define MSA_STATIC_SCRATCH_BYTES (4u << 20)
int msa_sparse_decode_static(const void *q, const void *kv, const int32_t *block_table,
                             const int32_t *seq_lens, const int32_t *topk, void *out, int B,
                             int Q, int Hq, int Hkv, int S, int64_t num_blocks, float sm_scale,
                             float k_scale, float v_scale, int num_splits, msa_stream_t stream);

/*
 * msa_decode_step -- one whole decode step in one call: msa_score (or
 * msa_score_kcache on `index_k`), then the block selection and the attend,
 * as the TensorRT-LLM PR #17171 decode path chains its scorer, selector and
 * flash-decoding kernels on one stream.
 *   q_scale       0: q is bf16 [T, Hq, 128]; > 0: q is fp8 e4m3 whose value
 *                 is q * q_scale (as the _q8 entry points)
 *   index_k       NULL: the blocks are scored on kv's K halves with k_scale;
 *                 else on this K-only cache [num_blocks, Hkv, 128, 128]
 *                 (msa_score_kcache) with index_k_scale (finite, > 0)
 *   scores        fp32 [Hkv, T, S], written (msa_score's output)
 *   topk          int32 [T, Hkv, 16], written (msa_topk's output)
 *   workspace     as msa_sparse_decode (msa_workspace_bytes(B, Q, Hq, s)
 *                 bytes for the effective split count s > 1)
 *   out           bf16 [T, Hq, 128]
 * The result equals msa_score, msa_topk and msa_sparse_decode called in turn
 * on the same arguments.  Rows of at most 512 candidate blocks (S <= 512) are
 * selected inside the attend kernel (msa_sparse_decode_select), longer ones
 * by the selector kernel.  Every argument is checked before anything is
 * enqueued.  Errors: those of msa_score, msa_topk and msa_sparse_decode, plus
 * q_scale < 0 or not finite, or index_k given with a bad index_k_scale
 * (MSA_EINVAL).
 */
int msa_decode_step(const void *q, float q_scale, const void *kv, const void *index_k,
                    float index_k_scale, const int32_t *block_table, const int32_t *seq_lens,
                    float *scores, int32_t *topk, void *workspace, size_t workspace_bytes,
                    void *out, int B, int Q, int Hq, int Hkv, int S, int64_t num_blocks,
                    float sm_scale, float k_scale, float v_scale, int num_splits,
                    msa_stream_t stream);

/*
 * msa_set_union_tile -- how msa_sparse_decode(_select) (and msa_decode_step,
 * msa_sparse_decode_static) attend decode steps of Q >= 2 tokens per request.
 * Off (0, the default): one CTA per (token, KV head), each loading its own
 * token's listed pages.  On (non-zero): one CTA per (request, tile of 4
 * consecutive tokens, KV head, split) over the union of the tile's lists,
 * each union page loaded once and attended by the tokens that listed it (the
 * way the vLLM CUTLASS decode plan sizes a request's work by its query
 * length).  This pays off when a request's tokens list mostly the same
 * blocks; with lists that overlap little (e.g. 52 distinct pages for 64
 * listed ones) the one-CTA-per-token form is faster on a GB300.  Results
 * agree within the output tolerance (the accumulation order differs).  The
 * split count msa_choose_splits reports follows this setting.  Dense decode
 * (msa_dense_decode) always attends a tile's shared pages this way when
 * Q >= 2.  Process-wide; returns the previous setting (0 or 1).
 */
int msa_set_union_tile(int enable);

/*
 * msa_set_input_overlap -- whether the first kernel of each call may start
 * before the previous kernel on its stream has finished (programmatic
 * dependent launch), reading the call's inputs (q, kv, block_table, seq_lens,
 * a given topk, cu_seqlens_q, a merge workspace) early, to overlap that
 * kernel's tail.  Off (0) by default: each call then waits for all earlier
 * work on its stream, and its inputs may be written by any kernel just
 * before it.  Turn it on (non-zero) only when the kernel just before every
 * call on the stream is one of this library's, or one that writes none of
 * that call's inputs: a kernel that wrote them could otherwise be read
 * before its writes are visible.  Outputs are always ordered: no library
 * kernel writes a buffer before the previous kernel has finished.
 * Process-wide; returns the previous setting (0 or 1).
 */
int msa_set_input_overlap(int enable);

/*
 * msa_test_wait_timeout -- for tests of the failure path.  Every wait inside
 * the library's kernels is bounded (2 s): when a phase does not complete in
 * time, the kernel sets MSA_ERR_TIMEOUT in the error word, waits (bounded)
 * for the copies it has in flight, frees its tensor memory and returns, so
 * the context stays usable.  This call enqueues one small kernel that takes
 * that exit on purpose: it allocates tensor memory, starts a bulk copy, and
 * waits limit_ns on an mbarrier that nothing completes.  Afterwards
 * msa_get_error reports MSA_ERR_TIMEOUT and later calls work as usual.
 * limit_ns in [1000, 2e9]; MSA_EINVAL otherwise.
 */
int msa_test_wait_timeout(unsigned long long limit_ns, msa_stream_t stream);

/*
 * Read the current device's sticky error word (an OR of MSA_ERR_* bits set by
 * any earlier call on any stream) into *flags, and reset it when `clear` is
 * non-zero.  Synchronises the device first.  Returns MSA_OK or MSA_ECUDA.
 */
int msa_get_error(unsigned int *flags, int clear);

/* Human-readable text for a status code. */
const char *msa_strerror(int status);

/* Library ABI version (major * 100 + minor). */
int msa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MSA_H */
