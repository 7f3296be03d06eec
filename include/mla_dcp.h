/*
 * mla_dcp.h -- C ABI of the GB300 (sm_103a) absorbed-MLA decode attention
 * library under decode context parallelism (DCP).
 *
 * Operations and their sources (page title, then section):
 *   - "vllm.v1.attention.backends.mla.flashattn_mla", FlashAttnMLAImpl.
 *     _forward_decode: the absorbed MLA decode.  The query is split into
 *     q_nope (kv_lora_rank = 512) and q_pe (qk_rope_head_dim = 64); one cache
 *     row is kv_c (first 512) followed by k_pe (64); the kernel is called
 *     with q=q_pe, k=k_pe, v=kv_c, q_v=q_nope, causal, a paged block_table,
 *     per-request seq_lens, cu_seqlens_q = query_start_loc, softmax_scale,
 *     and returns the softmax LSE laid out [tokens, heads] for DCP.
 *   - "[Attention] add DCP support for FLASH_ATTN_MLA backend", review
 *     thread: tokens are interleaved over the DCP ranks (token p on rank
 *     p mod D) and every query row has its own seqlen_k on each rank (the
 *     "DCP Rank 0/1" mask tables).
 *   - "[Attention][DCP] Support DCP with query length > 1 (MTP) with FA3",
 *     Purpose: q_len > 1 and mixed prefill/decode batches; the kernel only
 *     needs the cp world size and rank.
 *   - "[Attention] DCP sparse MLA output-merge optimizations", summary: the
 *     LSE-weighted merge of the per-rank results, the W_UV projection that
 *     commutes with it, per-row valid counts, sparse MLA.
 *
 * Conventions for every call:
 *   - Pointers marked "device" point to device memory of the current CUDA
 *     device; the caller owns every buffer.  The library allocates nothing:
 *     scratch comes from the caller's workspace.
 *   - All work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  No call synchronises the host or reads device memory from the
 *     host, so every call is asynchronous and returns before the GPU is done.
 *   - bf16 is IEEE bfloat16 stored in 16 bits; lse is float32 natural-log
 *     sum-exp of the scaled scores (softmax_scale included).
 *   - Return value: MLA_OK, or an error code with a message retrievable by
 *     mla_last_error() (thread-local).  Argument errors are detected on the
 *     host before anything is launched.  Data-dependent conditions the host
 *     cannot see without a sync (a page id out of range, q_len > seq_len)
 *     are checked by the kernels, which record the first failure in the
 *     workspace status word and skip the offending access; read it with
 *     mla_workspace_status().
 *   - An FP8 E4M3 latent cache is served by the dense _fp8 calls (the
 *     backend's constructor rejects one; this library adds it); the other
 *     calls, like the backend, return MLA_ERR_UNSUPPORTED for it, as for other
 *     head dims.
 */
#ifndef MLA_DCP_H
#define MLA_DCP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MLA_KV_LORA_RANK 512
#define MLA_ROPE_DIM 64
#define MLA_KV_ROW (MLA_KV_LORA_RANK + MLA_ROPE_DIM)
#define MLA_V_HEAD_DIM 128

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,   /* shape, pointer, alignment, rank >= world ... */
  MLA_ERR_UNSUPPORTED = 2,   /* FP8 cache, page size or head dims not served */
  MLA_ERR_CUDA = 3,          /* a CUDA runtime/driver call or launch failed */
  MLA_ERR_WORKSPACE = 4,     /* workspace NULL or smaller than required */
  MLA_ERR_DEVICE_CHECK = 5   /* (mla_workspace_status) a kernel check fired */
} mla_status;

typedef enum { MLA_DTYPE_BF16 = 0, MLA_DTYPE_F32 = 1, MLA_DTYPE_FP8_E4M3 = 2 } mla_dtype;

/* Message of the last failing call on this thread ("" if none). */
const char *mla_last_error(void);

/* ------------------------------------------------------------------------
 * mla_dcp_decode -- dense absorbed-MLA paged decode attention of DCP shard
 * `dcp_rank` of `dcp_world` ("flashattn_mla" _forward_decode with the DCP
 * mask of the FLASH_ATTN_MLA DCP review thread and the MTP page's cp world
 * size / rank).
 *
 * For request b (0 <= b < num_requests) with global length L = seq_lens[b]
 * and query tokens t in [query_start_loc[b], query_start_loc[b+1]) (q_len of
 * them), query token i sits at global position P = L - q_len + i.  This
 * shard holds the tokens p with p mod D == r at local slots j = p div D,
 * local slot j of request b being row (j mod page_size) of page
 * block_table[b * block_table_stride + j / page_size] of kv_cache.  Row
 * (t, h) sees local slot j iff j*D + r <= P, i.e. the first
 * n = floor((P - r)/D) + 1 slots (0 if P < r).  With
 *   s_j = scale * (q_nope[t,h,:] . kv_c_j + q_pe[t,h,:] . k_pe_j)
 * it writes lse[t,h] = log(sum_j exp(s_j)) and
 * out[t,h,:] = sum_j exp(s_j - lse) kv_c_j; a row that sees no key gets
 * lse = -inf and out = 0.  row_counts[t] = n.
 *
 *  q_nope   device bf16, row (t,h) at q_nope + (t*H + h)*q_nope_row_stride
 *           elements, 512 contiguous elements; stride >= 512, a multiple of 8.
 *  q_pe     device bf16, same with q_pe_row_stride (>= 64, multiple of 8).
 *           (q_nope = q, q_pe = q + 512 with both strides 576 serves a fused
 *           [T, H, 576] query.)
 *  kv_cache device bf16 [num_blocks, page_size, 576], contiguous, 16-byte
 *           aligned: this shard's cache slice.
 *  page_size  8, 16, 32, or a multiple of 64.
 *  block_table device int32 [num_requests, block_table_stride]: shard-local
 *           page ids; only the first ceil(local_len/page_size) entries of a
 *           row are read.
 *  seq_lens device int32 [num_requests]: GLOBAL lengths, new tokens
 *           included (q_len <= seq_len).
 *  query_start_loc device int32 [num_requests + 1], nondecreasing, [0] = 0,
 *           [num_requests] = num_tokens.
 *  max_query_len  upper bound of the q_lens; 0 is treated as 1 (the
 *           backend's capture-time clamp).
 *  max_seq_len    upper bound of seq_lens (sizes the split plan).
 *  out      device [num_tokens, num_heads, 512] of out_dtype (BF16 or F32).
 *  lse      device float32 [num_tokens, num_heads].
 *  row_counts device int32 [num_tokens], or NULL.
 *  scale    softmax scale, finite and > 0 (1/sqrt(192) for 128 + 64 q-k dims); the
 *           kernels take a row's largest score from the unscaled dot
 *           products, which needs a positive scale.
 *  num_splits  0 = automatic split-KV plan, else an upper bound on the KV
 *           chunks per request (fix it for CUDA-graph capture).
 *  workspace   device scratch of at least mla_dcp_decode_workspace_size()
 *           bytes, 256-byte aligned; contents need not be initialised.  Its
 *           size is bounded by the GPU's SM count (two slots of up to 64
 *           partial rows per SM), not by the batch.
 *  Stream order: every kernel of this library writes nothing before all
 *  earlier work on the stream has finished, but this call starts reading its
 *  inputs (q_nope, q_pe, kv_cache, block_table, seq_lens, query_start_loc)
 *  while the previous kernel on the stream finishes when that kernel is one
 *  of this library's.  So these inputs must not be outputs of the
 *  immediately preceding call of this library on the same stream.
 *  Launches: three kernels on `stream` (prep, decode, and the LSE merge of
 *  the KV chunks of row groups the decode split over several CTAs).
 *  Errors: INVALID_ARG (NULL/misaligned pointers, sizes < 0, dcp_rank not in
 *  [0, dcp_world), num_heads not in [1, 128], num_tokens * num_heads >=
 *  2^31, scale not finite and positive), UNSUPPORTED (page size),
 *  WORKSPACE, CUDA.  num_tokens == 0 is a
 *  successful no-op.
 * ---------------------------------------------------------------------- */
size_t mla_dcp_decode_workspace_size(int32_t num_requests, int32_t num_tokens, int32_t num_heads,
                                     int32_t max_query_len, int32_t max_seq_len, int32_t dcp_world,
                                     int32_t num_splits);

int mla_dcp_decode(const void *q_nope, int64_t q_nope_row_stride, const void *q_pe, int64_t q_pe_row_stride,
                   const void *kv_cache, int64_t num_blocks, int32_t page_size, int32_t kv_cache_dtype,
                   const int32_t *block_table, int32_t block_table_stride, const int32_t *seq_lens,
                   const int32_t *query_start_loc, int32_t num_requests, int32_t num_tokens, int32_t num_heads,
                   int32_t max_query_len, int32_t max_seq_len, int32_t dcp_world, int32_t dcp_rank, float scale,
                   void *out, int32_t out_dtype, float *lse, int32_t *row_counts, int32_t num_splits,
                   void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------
 * mla_dcp_decode_fp8 / mla_dcp_decode_fused_fp8 -- mla_dcp_decode and
 * mla_dcp_decode_fused over an FP8 latent cache.  "vllm.v1.attention.
 * backends.mla.flashattn_mla" (FlashAttnMLAImpl.__init__, _forward_decode)
 * rejects an FP8 KV cache; these calls serve the plainest such cache: every
 * value of a row (kv_c and k_pe) is one OCP FP8 E4M3 code (1 sign, 4 exponent
 * bits of bias 7, 3 mantissa bits; subnormals; no infinities; S.1111.111 is
 * NaN and must not occur) and the whole cache shares one dequantisation
 * scale, value = kv_scale * decode(code).  Scores and outputs are those of
 * mla_dcp_decode(_fused) on the dequantised values.
 *
 *  kv_cache / kv_caches  device uint8 [num_blocks, page_size, 576] of E4M3
 *            codes (576 bytes per row), 16-byte aligned; page layout and block
 *            tables as the bf16 calls.
 *  kv_scale  finite and > 0.
 *  workspace at least mla_dcp_decode_workspace_size() (resp.
 *            mla_dcp_decode_fused_workspace_size()) bytes: those sizes cover
 *            the bf16 and the FP8 calls.
 *  Other arguments, launches, stream order and errors as the bf16 calls
 *  (INVALID_ARG also for a bad kv_scale).
 * ---------------------------------------------------------------------- */
int mla_dcp_decode_fp8(const void *q_nope, int64_t q_nope_row_stride, const void *q_pe, int64_t q_pe_row_stride,
                       const void *kv_cache, int64_t num_blocks, int32_t page_size, float kv_scale,
                       const int32_t *block_table, int32_t block_table_stride, const int32_t *seq_lens,
                       const int32_t *query_start_loc, int32_t num_requests, int32_t num_tokens, int32_t num_heads,
                       int32_t max_query_len, int32_t max_seq_len, int32_t dcp_world, int32_t dcp_rank, float scale,
                       void *out, int32_t out_dtype, float *lse, int32_t *row_counts, int32_t num_splits,
                       void *workspace, size_t workspace_bytes, void *stream);

int mla_dcp_decode_fused_fp8(const void *q_nope, int64_t q_nope_row_stride, const void *q_pe,
                             int64_t q_pe_row_stride, const void *const *kv_caches, const int64_t *num_blocks,
                             int32_t page_size, float kv_scale, const int32_t *const *block_tables,
                             int32_t block_table_stride, const int32_t *seq_lens, const int32_t *query_start_loc,
                             int32_t num_requests, int32_t num_tokens, int32_t num_heads, int32_t max_query_len,
                             int32_t max_seq_len, int32_t dcp_world, float scale, void *out, int32_t out_dtype,
                             float *lse, int32_t num_splits, void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------
 * mla_sparse_dcp_decode -- the same attention over per-token top-k key lists
 * ("[Attention] DCP sparse MLA output-merge optimizations": sparse MLA with
 * per-row valid counts), restricted to DCP shard r of D.
 *
 * Query token t (of request b, global position P) uses the entries
 * topk_indices[t * topk + e] for e < topk_valid[t]; an entry is a global
 * token position of request b and is used iff 0 <= idx <= P (-1 pads).
 * Shard r keeps the used entries with idx mod D == r (local slot idx div D,
 * read through block_table as above).  Every kept entry is one key: with the
 * same s_j as the dense call, lse/out are the softmax over the kept keys of
 * that token (all heads share the list); local_counts[t] = number kept;
 * no key kept gives lse = -inf, out = 0.
 *
 *  topk_indices device int32 [num_tokens, topk], topk in [1, 65536].
 *  topk_valid   device int32 [num_tokens].
 *  local_counts device int32 [num_tokens] (required: it is the merge's
 *               per-row valid count).
 *  Other arguments as in mla_dcp_decode.  workspace >=
 *  mla_sparse_dcp_decode_workspace_size() bytes (per token, 8 bytes per
 *  list entry for the resolved cache-row addresses, plus a part bounded by
 *  the SM count).
 *  Launches: three kernels on `stream` (the key lists: each kept entry
 *  resolved to its cache row and counted, rows of tokens that keep none
 *  written; the decode over balanced ranges of (token, head group) key
 *  tiles; the LSE merge of the pairs it split).  The first waits for all
 *  earlier work on the stream before it reads anything.
 * ---------------------------------------------------------------------- */
size_t mla_sparse_dcp_decode_workspace_size(int32_t num_tokens, int32_t num_heads, int32_t topk,
                                            int32_t dcp_world);

int mla_sparse_dcp_decode(const void *q_nope, int64_t q_nope_row_stride, const void *q_pe, int64_t q_pe_row_stride,
                          const void *kv_cache, int64_t num_blocks, int32_t page_size, int32_t kv_cache_dtype,
                          const int32_t *block_table, int32_t block_table_stride, const int32_t *seq_lens,
                          const int32_t *query_start_loc, int32_t num_requests, int32_t num_tokens,
                          int32_t num_heads, const int32_t *topk_indices, int32_t topk, const int32_t *topk_valid,
                          int32_t dcp_world, int32_t dcp_rank, float scale, void *out, int32_t out_dtype,
                          float *lse, int32_t *local_counts, void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------
 * dcp_lse_merge -- LSE-weighted merge of the D shard results, optionally
 * fused with the per-head W_UV up-projection ("[Attention] DCP sparse MLA
 * output-merge optimizations", summary: _dcp_lse_merge /
 * _dcp_merge_and_v_up_proj; the projection commutes with the merge).
 *
 * For token t, head h, over the shards r that take part (valid_counts[r*T+t]
 * > 0 when valid_counts is given, else lses[(r*T+t)*H+h] > -inf):
 *   LSE = log(sum_r exp(lse_r)),  o = sum_r exp(lse_r - LSE) * partial_r
 *   out[t,h,:] = o            (w_uv == NULL, width 512)
 *   out[t,h,:] = o . W_UV[h]  (w_uv != NULL, width 128)
 * A row no shard takes part in gets out = 0 and LSE = -inf; the partials and
 * lses of shards that do not take part are not read (they may hold
 * anything, NaN included).
 *
 *  partials  device [dcp_world, num_tokens, num_heads, 512] of
 *            partial_dtype (BF16 or F32), 16-byte aligned.
 *  lses      device float32 [dcp_world, num_tokens, num_heads].
 *  valid_counts device int32 [dcp_world, num_tokens] or NULL.
 *  w_uv      device bf16 [num_heads, 512, 128] or NULL, 16-byte aligned.
 *  out       device [num_tokens, num_heads, 128 or 512] of out_dtype (BF16
 *            or F32).
 *  lse_out   device float32 [num_tokens, num_heads] or NULL.
 *  Errors: INVALID_ARG, CUDA.  num_tokens == 0 is a successful no-op.
 * ---------------------------------------------------------------------- */
int dcp_lse_merge(const void *partials, int32_t partial_dtype, const float *lses, const int32_t *valid_counts,
                  const void *w_uv, int32_t dcp_world, int32_t num_tokens, int32_t num_heads, void *out,
                  int32_t out_dtype, float *lse_out, void *stream);

/* ------------------------------------------------------------------------
 * mla_dcp_decode_fused -- every DCP shard of one decode step in one launch,
 * with the LSE merge built in, for one GPU that holds all D shard slices.
 * The pages define the D shard attentions ("[Attention] add DCP support for
 * FLASH_ATTN_MLA backend", the per-rank mask tables) and their LSE merge
 * ("[Attention] DCP sparse MLA output-merge optimizations"); a softmax that
 * continues over shard r's keys after shard r-1's computes exactly that
 * merge.  Each (request, row group) streams shard 0's visible
 * keys, then shard 1's, ..., each through its own cache slice, block table
 * and DCP mask (key j of shard r is seen by the query at position P iff
 * j*D + r <= P), so the D partial outputs never reach memory.
 *
 *  kv_caches    host array of D device pointers, shard r's cache slice
 *               [num_blocks[r], page_size, 576] bf16 (as mla_dcp_decode's
 *               kv_cache for rank r).
 *  num_blocks   host array of D page counts.
 *  block_tables host array of D device pointers, shard r's block table
 *               [num_requests, block_table_stride] int32 (shard-local ids).
 *  dcp_world    D, 1..8.
 *  out, lse     the merged result: out [num_tokens, num_heads, 512] of
 *               out_dtype (BF16 or F32), lse float32 [num_tokens, num_heads]
 *               = log of the sum of exp(scores) over every shard's visible
 *               keys.  (For the W_UV projection, pass F32 out to
 *               dcp_lse_merge with dcp_world 1.)
 *  workspace    device scratch of at least mla_dcp_decode_fused_workspace_size()
 *               bytes, 256-byte aligned.
 *  Other arguments, errors and the stream-order rule as mla_dcp_decode.
 * ---------------------------------------------------------------------- */
size_t mla_dcp_decode_fused_workspace_size(int32_t num_requests, int32_t num_tokens, int32_t num_heads,
                                           int32_t max_query_len, int32_t max_seq_len, int32_t num_splits);

int mla_dcp_decode_fused(const void *q_nope, int64_t q_nope_row_stride, const void *q_pe, int64_t q_pe_row_stride,
                         const void *const *kv_caches, const int64_t *num_blocks, int32_t page_size,
                         int32_t kv_cache_dtype, const int32_t *const *block_tables, int32_t block_table_stride,
                         const int32_t *seq_lens, const int32_t *query_start_loc, int32_t num_requests,
                         int32_t num_tokens, int32_t num_heads, int32_t max_query_len, int32_t max_seq_len,
                         int32_t dcp_world, float scale, void *out, int32_t out_dtype, float *lse,
                         int32_t num_splits, void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------
 * mla_sparse_dcp_decode_fused -- the sparse decode of every DCP shard of one
 * step in one call, with the merge built in, for one GPU that holds all D
 * shard slices (the sparse counterpart of mla_dcp_decode_fused).  Token t's
 * result merged over the D shards ("[Attention] DCP sparse MLA output-merge
 * optimizations": LSE merge with per-row valid counts) is the softmax over
 * the union of the shards' kept entries, i.e. over every used entry of its
 * list, each read from its own shard (idx mod D) at local slot idx div D
 * through that shard's block table.  One key-list kernel resolves every
 * entry to its cache row, then one decode launch runs each (token, head
 * group) over the whole list.
 *
 *  kv_caches, num_blocks, block_tables  host arrays of D entries, as in
 *               mla_dcp_decode_fused.
 *  topk_indices, topk, topk_valid  as in mla_sparse_dcp_decode.
 *  dcp_world    D, 1..8.
 *  out, lse     the merged result (as mla_dcp_decode_fused); no used entry
 *               gives lse = -inf, out = 0.
 *  kept_counts  device int32 [num_tokens] (the number of used entries over
 *               all shards), or NULL.
 *  workspace    >= mla_sparse_dcp_decode_workspace_size() bytes.
 *  Errors as mla_sparse_dcp_decode; INVALID_ARG if dcp_world > 8.
 * ---------------------------------------------------------------------- */
int mla_sparse_dcp_decode_fused(const void *q_nope, int64_t q_nope_row_stride, const void *q_pe,
                                int64_t q_pe_row_stride, const void *const *kv_caches, const int64_t *num_blocks,
                                int32_t page_size, int32_t kv_cache_dtype, const int32_t *const *block_tables,
                                int32_t block_table_stride, const int32_t *seq_lens, const int32_t *query_start_loc,
                                int32_t num_requests, int32_t num_tokens, int32_t num_heads,
                                const int32_t *topk_indices, int32_t topk, const int32_t *topk_valid,
                                int32_t dcp_world, float scale, void *out, int32_t out_dtype, float *lse,
                                int32_t *kept_counts, void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------
 * mla_dcp_decode_two_stage -- the two-stage decomposition of a DCP decode
 * step with q_len >= 1, for one GPU that holds all D shard slices: the
 * alternative to a custom mask offered in the review thread of
 * "[Attention] add DCP support for FLASH_ATTN_MLA backend" (context keys with
 * the causal mask off, the query's own keys with it on, results merged).
 * For request b with L keys and q_len queries:
 *   stage 1  every query row over the context positions [0, L - q_len), no
 *            mask: a shard-fused dense decode whose sequence lengths are the
 *            context lengths (derived on the device);
 *   stage 2  query i over the new positions L - q_len .. L - q_len + i: the
 *            shard-fused sparse decode over per-token position lists built on
 *            the device (list width max_query_len);
 *   merge    the two (out, lse) results by LSE (dcp_lse_merge with the two
 *            stages as its two partials).
 * The result equals mla_dcp_decode_fused's (the causal DCP attention over
 * all L keys), up to rounding; a row's stage-1 result is empty (lse -inf)
 * when its request has no context.  Launches: the prep kernel, stage 1's
 * three, stage 2's two, a status fold and the merge; no host copy.
 *
 *  Arguments as mla_dcp_decode_fused (kv_cache_dtype BF16 only); num_splits
 *  is not taken.
 *  max_query_len  >= every request's q_len (the list width), 1..65536 when
 *               num_tokens > 0.
 *  workspace    device scratch of at least
 *               mla_dcp_decode_two_stage_workspace_size() bytes, 256-byte
 *               aligned; its status word (mla_workspace_status) reports the
 *               first failing check of either stage.
 *  Errors as mla_dcp_decode_fused.
 * ---------------------------------------------------------------------- */
size_t mla_dcp_decode_two_stage_workspace_size(int32_t num_requests, int32_t num_tokens, int32_t num_heads,
                                               int32_t max_query_len, int32_t max_seq_len);

int mla_dcp_decode_two_stage(const void *q_nope, int64_t q_nope_row_stride, const void *q_pe,
                             int64_t q_pe_row_stride, const void *const *kv_caches, const int64_t *num_blocks,
                             int32_t page_size, int32_t kv_cache_dtype, const int32_t *const *block_tables,
                             int32_t block_table_stride, const int32_t *seq_lens, const int32_t *query_start_loc,
                             int32_t num_requests, int32_t num_tokens, int32_t num_heads, int32_t max_query_len,
                             int32_t max_seq_len, int32_t dcp_world, float scale, void *out, int32_t out_dtype,
                             float *lse, void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------
 * mla_workspace_status -- synchronises `stream`, then reads the status word
 * the kernels keep in a decode workspace: MLA_OK, or MLA_ERR_DEVICE_CHECK
 * with *detail set to the first failing check's code: 1 = a page id (or its
 * block-table column) out of range, 2 = q_len > seq_len or a bad
 * query_start_loc, 3 = a pipeline wait gave up, 4 = a split-table entry
 * out of range (an internal inconsistency).  This is the one call that
 * blocks the host.
 *
 * A decode CTA whose wait gives up stops issuing work, waits (with a bound
 * of its own) for every copy and MMA it already issued, frees its tensor
 * memory and exits, so the call completes and the context stays usable; its
 * outputs are then unspecified.  The workspace's third 32-bit word then
 * holds the site of the first wait that gave up (a diagnostic number).
 * ---------------------------------------------------------------------- */
int mla_workspace_status(const void *workspace, void *stream, int32_t *detail);

/* ------------------------------------------------------------------------
 * mla_dcp_decode_static_scratch -- mla_dcp_decode for callers that cannot
 * allocate device memory.  No counterpart on the pages; it exists for users
 * of this library, not for the method.
 *
 * Some callers cannot call cudaMalloc (or anything that allocates) when they
 * run a decode step: code working inside a device-memory budget fixed at
 * start-up, engines whose only allocator is their own pre-reserved pool, or
 * latency-critical paths where allocation is forbidden.  They cannot provide
 * the workspace mla_dcp_decode asks for.  This variant takes the same
 * arguments minus the workspace and uses a fixed array of
 * MLA_STATIC_SCRATCH_BYTES in the library's device memory instead.
 *
 *  - The array exists on every GPU that loads the library and stays
 *    allocated until the process exits.
 *  - The first call on a device looks up the array's device address, with
 *    that device current, and keeps it for the device's current CUDA context
 *    (a context created later, e.g. after cudaDeviceReset, gets a fresh
 *    lookup).  Make that first call before any stream capture on the device.
 *  - Arguments are checked first (errors as mla_dcp_decode); only a valid
 *    problem can be refused for its size.
 *  - Problems whose scratch (mla_dcp_decode_workspace_size) exceeds the
 *    array are refused with MLA_ERR_WORKSPACE before anything runs.  The
 *    dense workspace is bounded by the GPU's SM count: 2 partial slots of
 *    16, 32 or 64 rows of 2 KB per SM (the rows per work unit grow with
 *    max_query_len x num_heads: up to 16, 32, then 64) plus small tables.
 *    On a 152-SM GB300, problems of up to 32 rows per request fit; those
 *    with more (about 40 MB) are refused.
 *  - Every call shares the one array: calls that may overlap on the GPU
 *    (unordered streams) race on it.  Calls on one stream are fine.  The
 *    array keeps the last call's contents; what must start at zero (the
 *    status word) is cleared by each call.
 *  - mla_workspace_status() cannot reach this array; device checks of this
 *    variant are not reported.
 *  - It allocates nothing and calls no allocating routine.
 * ---------------------------------------------------------------------- */
#define MLA_STATIC_SCRATCH_BYTES (24u * 1024u * 1024u)

int mla_dcp_decode_static_scratch(const void *q_nope, int64_t q_nope_row_stride, const void *q_pe,
                                  int64_t q_pe_row_stride, const void *kv_cache, int64_t num_blocks, int32_t page_size,
                                  int32_t kv_cache_dtype, const int32_t *block_table, int32_t block_table_stride,
                                  const int32_t *seq_lens, const int32_t *query_start_loc, int32_t num_requests,
                                  int32_t num_tokens, int32_t num_heads, int32_t max_query_len, int32_t max_seq_len,
                                  int32_t dcp_world, int32_t dcp_rank, float scale, void *out, int32_t out_dtype,
                                  float *lse, int32_t *row_counts, int32_t num_splits, void *stream);

/* ------------------------------------------------------------------------
 * mla_kernel_launch_count -- number of kernels this library has launched in
 * this process so far (all threads; memsets excluded).  Lets a caller state
 * how many of the library's kernels ran inside a timed region.
 * ---------------------------------------------------------------------- */
int64_t mla_kernel_launch_count(void);

/* ------------------------------------------------------------------------
 * mla_debug_set_wait_budget_ns -- test hook: the budget, in ns, of every
 * pipeline wait inside the decode kernels launched after this call by any
 * thread of the process (0 restores the default, 2 s).  With a budget too
 * short for the pipeline, waits give up and the call reports check 3 through
 * mla_workspace_status; nothing else changes.  Not for production use.
 * ---------------------------------------------------------------------- */
void mla_debug_set_wait_budget_ns(uint64_t ns);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DCP_H */
