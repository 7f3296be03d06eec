// api.cu -- the C ABI (include/mla_dcp.h): argument checks, planning, launches.
#include <stdarg.h>
#include <stdio.h>

#include <atomic>
#include <cmath>
#include <string>

#include "common.cuh"
#include "decode_kernels.h"
#include "pdl_launch.h"
#include "plan.h"

namespace {

thread_local std::string g_last_error;
std::atomic<int64_t> g_launches{0};
std::atomic<uint64_t> g_wait_budget_ns{0};  // 0: the kernels' default (2 s)

void count_launch(int n = 1) { g_launches.fetch_add(n, std::memory_order_relaxed); }

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int ok() {
  g_last_error.clear();
  return MLA_OK;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(MLA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int current_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 152;
  }
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return 152;
  }
  return n;
}

bool page_size_supported(int32_t ps) { return ps == 8 || ps == 16 || ps == 32 || (ps >= 64 && ps % 64 == 0); }

// Checks shared by the dense and sparse decode calls.
int check_decode_common(const void* q_nope, int64_t q_nope_row_stride, const void* q_pe, int64_t q_pe_row_stride,
                        const void* kv_cache, int64_t num_blocks, int32_t page_size, int32_t kv_cache_dtype,
                        const int32_t* block_table, int32_t block_table_stride, const int32_t* seq_lens,
                        const int32_t* query_start_loc, int32_t num_requests, int32_t num_tokens, int32_t num_heads,
                        int32_t dcp_world, int32_t dcp_rank, float scale, void* out, int32_t out_dtype, float* lse,
                        void* workspace, bool fp8_call = false) {
  if (fp8_call ? kv_cache_dtype != MLA_DTYPE_FP8_E4M3 : kv_cache_dtype != MLA_DTYPE_BF16)
    return fail(MLA_ERR_UNSUPPORTED,
                fp8_call ? "kv_cache_dtype %d: the _fp8 calls take an FP8 E4M3 cache"
                         : "kv_cache_dtype %d: this call takes a bf16 latent cache (an FP8 E4M3 cache goes through "
                           "mla_dcp_decode_fp8 / mla_dcp_decode_fused_fp8)",
                kv_cache_dtype);
  if (num_tokens < 0 || num_requests < 1 || num_heads < 1 || num_heads > mla::kMaxHeads)
    return fail(MLA_ERR_INVALID_ARG, "bad sizes: num_requests=%d num_tokens=%d num_heads=%d (heads in [1,%d])",
                num_requests, num_tokens, num_heads, mla::kMaxHeads);
  if (dcp_world < 1 || dcp_world > 64 || dcp_rank < 0 || dcp_rank >= dcp_world)
    return fail(MLA_ERR_INVALID_ARG, "dcp_rank %d not in [0, dcp_world=%d) or dcp_world not in [1, 64]", dcp_rank,
                dcp_world);
  if (num_blocks < 1 || kv_cache == nullptr)
    return fail(MLA_ERR_INVALID_ARG, "empty KV cache (num_blocks=%lld)", (long long)num_blocks);
  if (!page_size_supported(page_size))
    return fail(MLA_ERR_UNSUPPORTED, "page_size %d: supported are 8, 16, 32 and multiples of 64", page_size);
  if (block_table_stride < 1) return fail(MLA_ERR_INVALID_ARG, "block_table_stride %d < 1", block_table_stride);
  if (!q_nope || !q_pe || !block_table || !seq_lens || !query_start_loc || !out || !lse)
    return fail(MLA_ERR_INVALID_ARG, "a required pointer is NULL");
  if (q_nope_row_stride < mla::kNope || q_nope_row_stride % 8 || q_pe_row_stride < mla::kRope ||
      q_pe_row_stride % 8)
    return fail(MLA_ERR_INVALID_ARG, "query row strides %lld/%lld: need >= 512/64 and multiples of 8",
                (long long)q_nope_row_stride, (long long)q_pe_row_stride);
  if (!aligned(q_nope, 16) || !aligned(q_pe, 16) || !aligned(kv_cache, 16) || !aligned(out, 16) ||
      !aligned(lse, 4) || !aligned(block_table, 4))
    return fail(MLA_ERR_INVALID_ARG, "misaligned pointer (q/cache/out need 16-byte alignment)");
  if (out_dtype != MLA_DTYPE_BF16 && out_dtype != MLA_DTYPE_F32)
    return fail(MLA_ERR_INVALID_ARG, "out_dtype %d: BF16 or F32", out_dtype);
  if (!std::isfinite(scale) || !(scale > 0.f))
    return fail(MLA_ERR_INVALID_ARG, "scale %g: a finite positive softmax scale is required", scale);
  if (workspace == nullptr || !aligned(workspace, 256))
    return fail(MLA_ERR_WORKSPACE, "workspace NULL or not 256-byte aligned");
  return MLA_OK;
}

}  // namespace

namespace mla {
// Lets other translation units of the library report through mla_last_error.
int set_last_error(int code, const char* msg) { return fail(code, "%s", msg); }

// Every host-side check of an mla_dcp_decode call except those on the
// workspace: MLA_OK, or the error the call would return (message set).
int check_dense_decode_args(const void* q_nope, int64_t q_nope_row_stride, const void* q_pe, int64_t q_pe_row_stride,
                            const void* kv_cache, int64_t num_blocks, int32_t page_size, int32_t kv_cache_dtype,
                            const int32_t* block_table, int32_t block_table_stride, const int32_t* seq_lens,
                            const int32_t* query_start_loc, int32_t num_requests, int32_t num_tokens,
                            int32_t num_heads, int32_t max_query_len, int32_t max_seq_len, int32_t dcp_world,
                            int32_t dcp_rank, float scale, void* out, int32_t out_dtype, float* lse,
                            int32_t num_splits) {
  static __align__(256) const uint8_t placeholder[1] = {0};  // stands for a workspace; never read
  int rc = check_decode_common(q_nope, q_nope_row_stride, q_pe, q_pe_row_stride, kv_cache, num_blocks, page_size,
                               kv_cache_dtype, block_table, block_table_stride, seq_lens, query_start_loc,
                               num_requests, num_tokens, num_heads, dcp_world, dcp_rank, scale, out, out_dtype, lse,
                               const_cast<uint8_t*>(placeholder));
  if (rc != MLA_OK) return rc;
  (void)max_query_len;
  if (max_seq_len < 0 || num_splits < 0 || num_splits > 1024)
    return fail(MLA_ERR_INVALID_ARG, "max_seq_len %d / num_splits %d out of range", max_seq_len, num_splits);
  if ((int64_t)num_tokens * num_heads > 0x7fffffff)
    return fail(MLA_ERR_INVALID_ARG, "num_tokens * num_heads = %lld exceeds 2^31 - 1",
                (long long)num_tokens * num_heads);
  return MLA_OK;
}
}  // namespace mla

extern "C" {

const char* mla_last_error(void) { return g_last_error.c_str(); }

// The larger of the bf16 and FP8 plans' workspaces (their unit sizes, and so
// their grids and partial slots, can differ), so one size serves both calls.
static size_t dense_workspace_bytes(int32_t num_requests, int32_t num_tokens, int32_t num_heads,
                                    int32_t max_query_len, int32_t max_seq_len, int32_t D, int32_t num_splits) {
  const int sms = current_sm_count();
  const size_t a = mla::make_decode_plan(num_requests, num_tokens, num_heads, max_query_len, max_seq_len, D,
                                         num_splits, sms, false).total;
  const size_t b = mla::make_decode_plan(num_requests, num_tokens, num_heads, max_query_len, max_seq_len, D,
                                         num_splits, sms, true).total;
  return a > b ? a : b;
}

size_t mla_dcp_decode_workspace_size(int32_t num_requests, int32_t num_tokens, int32_t num_heads,
                                     int32_t max_query_len, int32_t max_seq_len, int32_t dcp_world,
                                     int32_t num_splits) {
  if (dcp_world < 1) dcp_world = 1;
  return dense_workspace_bytes(num_requests, num_tokens, num_heads, max_query_len, max_seq_len, dcp_world,
                               num_splits);
}

}  // extern "C"

namespace {

// The LSE merge of the chunks of the row groups a decode launch of `grid`
// CTAs split (entries of its split table), right after it on the stream.
cudaError_t launch_split_merge(const mla::DecodeArgs& da, int rows_per_group, int grid, int64_t num_rows,
                               cudaStream_t st) {
  mla::SplitMergeArgs sa{};
  sa.cta_stride = da.gang > 1 ? da.gang : 1;
  sa.split_desc = da.split_desc;
  sa.part_lse = da.part_lse;
  sa.part_o = da.part_o;
  sa.rows_per_group = rows_per_group;
  sa.grid = grid;
  sa.num_rows = num_rows;
  sa.out = da.out;
  sa.out_f32 = da.out_f32;
  sa.lse = da.lse;
  sa.hdr = da.hdr;
  const int blocks = grid * (rows_per_group / mla::kSplitMergeRows);
  return mla::launch_pdl(mla::split_merge_kernel, dim3(blocks), dim3(128), 0, st, sa);
}

// The dense decode over nshard consecutive shards from rank shard0 (one
// shard: mla_dcp_decode; all D: mla_dcp_decode_fused).  Arguments checked.
int dense_decode(const void* q_nope, int64_t q_nope_row_stride, const void* q_pe, int64_t q_pe_row_stride,
                 int nshard, int shard0, const void* const* kv_caches, const int64_t* num_blocks, int32_t page_size,
                 const int32_t* const* block_tables, int32_t block_table_stride, const int32_t* seq_lens,
                 const int32_t* query_start_loc, int32_t num_requests, int32_t num_tokens, int32_t num_heads,
                 int32_t max_query_len, int32_t max_seq_len, int32_t dcp_world, float scale, void* out,
                 int32_t out_dtype, float* lse, int32_t* row_counts, int32_t num_splits, void* workspace,
                 size_t workspace_bytes, void* stream, bool kv_fp8 = false, float kv_scale = 1.f,
                 bool causal = true) {
  if (max_seq_len < 0 || num_splits < 0 || num_splits > 1024)
    return fail(MLA_ERR_INVALID_ARG, "max_seq_len %d / num_splits %d out of range", max_seq_len, num_splits);
  if (num_tokens == 0) return ok();
  if ((int64_t)num_tokens * num_heads > 0x7fffffff)
    return fail(MLA_ERR_INVALID_ARG, "num_tokens * num_heads = %lld exceeds 2^31 - 1",
                (long long)num_tokens * num_heads);
  const mla::DecodePlan plan = mla::make_decode_plan(num_requests, num_tokens, num_heads, max_query_len, max_seq_len,
                                                     dcp_world / nshard, num_splits, current_sm_count(), kv_fp8);
  if (workspace_bytes < plan.total)
    return fail(MLA_ERR_WORKSPACE, "workspace %zu bytes < %zu required", workspace_bytes, plan.total);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  mla::WorkspaceHeader* hdr = reinterpret_cast<mla::WorkspaceHeader*>(ws);

  cudaError_t e;
  mla::PrepArgs pa{};
  pa.seq_lens = seq_lens;
  pa.query_start_loc = query_start_loc;
  pa.num_requests = num_requests;
  pa.num_tokens = num_tokens;
  pa.num_heads = num_heads;
  pa.dcp_world = dcp_world;
  pa.shard0 = shard0;
  pa.nshard = nshard;
  pa.rows_per_group = plan.rows_per_group;
  pa.noncausal = causal ? 0 : 1;
  pa.hdr = hdr;
  pa.row_counts = row_counts;
  pa.out = out;
  pa.out_f32 = out_dtype == MLA_DTYPE_F32;
  pa.lse = lse;
  {
    int blocks = (num_requests + 255) / 256;
    if (blocks > 64) blocks = 64;
    if ((e = mla::launch_pdl(mla::prep_kernel, dim3(blocks), dim3(256), 0, st, pa)) != cudaSuccess)
      return cuda_fail(e, "prep_kernel launch");
  }
  count_launch();

  mla::DecodeArgs da{};
  da.q_nope = static_cast<const __nv_bfloat16*>(q_nope);
  da.q_nope_stride = q_nope_row_stride;
  da.q_pe = static_cast<const __nv_bfloat16*>(q_pe);
  da.q_pe_stride = q_pe_row_stride;
  da.kv = static_cast<const __nv_bfloat16*>(kv_caches[0]);
  da.page_size = page_size;
  da.bt_stride = block_table_stride;
  da.nshard = nshard;
  da.shard0 = shard0;
  for (int k = 0; k < nshard; ++k) {
    da.kvs[k] = static_cast<const __nv_bfloat16*>(kv_caches[k]);
    da.bts[k] = block_tables[k];
    da.nblocks[k] = num_blocks[k];
  }
  da.num_heads = num_heads;
  da.dcp_world = dcp_world;
  da.scale = scale;
  da.kv_fp8 = kv_fp8 ? 1 : 0;
  da.kv_scale = kv_fp8 ? kv_scale : 1.f;
  da.out = out;
  da.out_f32 = out_dtype == MLA_DTYPE_F32;
  da.lse = lse;
  da.hdr = hdr;
  da.seq_lens = seq_lens;
  da.query_start_loc = query_start_loc;
  da.num_requests = num_requests;
  da.unit_penalty = plan.unit_penalty;
  da.gang = plan.gang;
  da.wait_ns = g_wait_budget_ns.load(std::memory_order_relaxed);
  da.noncausal = causal ? 0 : 1;
  da.split_desc = reinterpret_cast<int4*>(ws + plan.off_desc);
  da.part_lse = reinterpret_cast<float*>(ws + plan.off_plse);
  da.part_o = reinterpret_cast<float*>(ws + plan.off_po);
  da.num_tokens = num_tokens;
  if ((e = mla::launch_decode_tc(da, plan.rows_per_group, false, plan.grid, plan.grid, st)) != cudaSuccess)
    return cuda_fail(e, "decode launch");
  count_launch();

  if ((e = launch_split_merge(da, plan.rows_per_group, plan.grid, (int64_t)num_tokens * num_heads, st)) !=
      cudaSuccess)
    return cuda_fail(e, "split_merge_kernel launch");
  count_launch();
  return ok();
}

// The sparse decode over nshard consecutive shards from rank shard0 (one
// shard: mla_sparse_dcp_decode; all D: mla_sparse_dcp_decode_fused).
// Arguments other than the list inputs checked by the caller.
int sparse_decode(const void* q_nope, int64_t q_nope_row_stride, const void* q_pe, int64_t q_pe_row_stride,
                  int nshard, int shard0, const void* const* kv_caches, const int64_t* num_blocks, int32_t page_size,
                  const int32_t* const* block_tables, int32_t block_table_stride, const int32_t* seq_lens,
                  const int32_t* query_start_loc, int32_t num_requests, int32_t num_tokens, int32_t num_heads,
                  const int32_t* topk_indices, int32_t topk, const int32_t* topk_valid, int32_t dcp_world,
                  float scale, void* out, int32_t out_dtype, float* lse, int32_t* counts_out, void* workspace,
                  size_t workspace_bytes, void* stream) {
  if (!topk_indices || !topk_valid) return fail(MLA_ERR_INVALID_ARG, "topk_indices and topk_valid are required");
  if (topk < 1 || topk > 65536) return fail(MLA_ERR_INVALID_ARG, "topk %d not in [1, 65536]", topk);
  if (num_tokens == 0) return ok();
  if ((int64_t)num_tokens * num_heads > 0x7fffffff)
    return fail(MLA_ERR_INVALID_ARG, "num_tokens * num_heads = %lld exceeds 2^31 - 1",
                (long long)num_tokens * num_heads);
  const mla::SparsePlan plan = mla::make_sparse_plan(num_tokens, num_heads, topk, current_sm_count());
  if (workspace_bytes < plan.total)
    return fail(MLA_ERR_WORKSPACE, "workspace %zu bytes < %zu required", workspace_bytes, plan.total);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  mla::WorkspaceHeader* hdr = reinterpret_cast<mla::WorkspaceHeader*>(ws);
  cudaError_t e = cudaMemsetAsync(hdr, 0, 16, st);
  if (e != cudaSuccess) return cuda_fail(e, "workspace header reset");

  mla::SparseListArgs la{};
  la.topk = topk_indices;
  la.topk_valid = topk_valid;
  la.seq_lens = seq_lens;
  la.query_start_loc = query_start_loc;
  la.num_requests = num_requests;
  la.num_tokens = num_tokens;
  la.topk_k = topk;
  la.dcp_world = dcp_world;
  la.shard0 = shard0;
  la.nshard = nshard;
  for (int k = 0; k < nshard; ++k) {
    la.kvs[k] = kv_caches[k];
    la.bts[k] = block_tables[k];
    la.nblocks[k] = num_blocks[k];
  }
  la.page_size = page_size;
  la.bt_stride = block_table_stride;
  la.key_rows = reinterpret_cast<int64_t*>(ws + plan.off_lists);
  la.counts = counts_out ? counts_out : reinterpret_cast<int32_t*>(ws + plan.off_cnt);
  la.hdr = hdr;
  la.num_heads = num_heads;
  la.out = out;
  la.out_f32 = out_dtype == MLA_DTYPE_F32;
  la.lse = lse;
  if ((e = mla::launch_sparse_lists(la, st)) != cudaSuccess) return cuda_fail(e, "sparse list launch");
  count_launch();

  mla::DecodeArgs da{};
  da.q_nope = static_cast<const __nv_bfloat16*>(q_nope);
  da.q_nope_stride = q_nope_row_stride;
  da.q_pe = static_cast<const __nv_bfloat16*>(q_pe);
  da.q_pe_stride = q_pe_row_stride;
  da.kv = static_cast<const __nv_bfloat16*>(kv_caches[0]);
  da.page_size = page_size;
  da.nshard = 1;  // the key lists hold row addresses: the decode reads no shard table
  da.shard0 = shard0;
  da.kvs[0] = static_cast<const __nv_bfloat16*>(kv_caches[0]);
  da.bts[0] = block_tables[0];
  da.nblocks[0] = num_blocks[0];
  da.bt_stride = block_table_stride;
  da.num_heads = num_heads;
  da.dcp_world = dcp_world;
  da.scale = scale;
  da.kv_fp8 = 0;
  da.kv_scale = 1.f;
  da.out = out;
  da.out_f32 = out_dtype == MLA_DTYPE_F32;
  da.lse = lse;
  da.hdr = hdr;
  da.key_rows = la.key_rows;
  da.list_count = la.counts;
  da.list_stride = topk;
  da.num_tokens = num_tokens;
  da.unit_penalty = mla::kUnitPenalty;
  da.gang = 1;
  da.wait_ns = g_wait_budget_ns.load(std::memory_order_relaxed);
  da.split_desc = reinterpret_cast<int4*>(ws + plan.off_desc);
  da.part_lse = reinterpret_cast<float*>(ws + plan.off_plse);
  da.part_o = reinterpret_cast<float*>(ws + plan.off_po);
  if ((e = mla::launch_decode_tc(da, plan.rows_per_group, true, plan.grid, plan.grid, st)) != cudaSuccess)
    return cuda_fail(e, "sparse decode launch");
  count_launch();
  if ((e = launch_split_merge(da, plan.rows_per_group, plan.grid, (int64_t)num_tokens * num_heads, st)) !=
      cudaSuccess)
    return cuda_fail(e, "split_merge_kernel launch");
  count_launch();
  return ok();
}

}  // namespace

extern "C" {

int mla_dcp_decode(const void* q_nope, int64_t q_nope_row_stride, const void* q_pe, int64_t q_pe_row_stride,
                   const void* kv_cache, int64_t num_blocks, int32_t page_size, int32_t kv_cache_dtype,
                   const int32_t* block_table, int32_t block_table_stride, const int32_t* seq_lens,
                   const int32_t* query_start_loc, int32_t num_requests, int32_t num_tokens, int32_t num_heads,
                   int32_t max_query_len, int32_t max_seq_len, int32_t dcp_world, int32_t dcp_rank, float scale,
                   void* out, int32_t out_dtype, float* lse, int32_t* row_counts, int32_t num_splits,
                   void* workspace, size_t workspace_bytes, void* stream) {
  int rc = check_decode_common(q_nope, q_nope_row_stride, q_pe, q_pe_row_stride, kv_cache, num_blocks, page_size,
                               kv_cache_dtype, block_table, block_table_stride, seq_lens, query_start_loc,
                               num_requests, num_tokens, num_heads, dcp_world, dcp_rank, scale, out, out_dtype, lse,
                               workspace);
  if (rc != MLA_OK) return rc;
  const void* kvs[1] = {kv_cache};
  const int64_t nbs[1] = {num_blocks};
  const int32_t* bts[1] = {block_table};
  return dense_decode(q_nope, q_nope_row_stride, q_pe, q_pe_row_stride, 1, dcp_rank, kvs, nbs, page_size, bts,
                      block_table_stride, seq_lens, query_start_loc, num_requests, num_tokens, num_heads,
                      max_query_len, max_seq_len, dcp_world, scale, out, out_dtype, lse, row_counts, num_splits,
                      workspace, workspace_bytes, stream);
}

size_t mla_dcp_decode_fused_workspace_size(int32_t num_requests, int32_t num_tokens, int32_t num_heads,
                                           int32_t max_query_len, int32_t max_seq_len, int32_t num_splits) {
  return dense_workspace_bytes(num_requests, num_tokens, num_heads, max_query_len, max_seq_len, 1, num_splits);
}

int mla_dcp_decode_fused(const void* q_nope, int64_t q_nope_row_stride, const void* q_pe, int64_t q_pe_row_stride,
                         const void* const* kv_caches, const int64_t* num_blocks, int32_t page_size,
                         int32_t kv_cache_dtype, const int32_t* const* block_tables, int32_t block_table_stride,
                         const int32_t* seq_lens, const int32_t* query_start_loc, int32_t num_requests,
                         int32_t num_tokens, int32_t num_heads, int32_t max_query_len, int32_t max_seq_len,
                         int32_t dcp_world, float scale, void* out, int32_t out_dtype, float* lse, int32_t num_splits,
                         void* workspace, size_t workspace_bytes, void* stream) {
  if (dcp_world < 1 || dcp_world > mla::kMaxShards)
    return fail(MLA_ERR_INVALID_ARG, "dcp_world %d not in [1, %d] for the fused call", dcp_world, mla::kMaxShards);
  if (kv_caches == nullptr || num_blocks == nullptr || block_tables == nullptr)
    return fail(MLA_ERR_INVALID_ARG, "kv_caches / num_blocks / block_tables arrays are NULL");
  for (int r = 0; r < dcp_world; ++r) {
    int rc = check_decode_common(q_nope, q_nope_row_stride, q_pe, q_pe_row_stride, kv_caches[r], num_blocks[r],
                                 page_size, kv_cache_dtype, block_tables[r], block_table_stride, seq_lens,
                                 query_start_loc, num_requests, num_tokens, num_heads, dcp_world, r, scale, out,
                                 out_dtype, lse, workspace);
    if (rc != MLA_OK) return rc;
  }
  return dense_decode(q_nope, q_nope_row_stride, q_pe, q_pe_row_stride, dcp_world, 0, kv_caches, num_blocks,
                      page_size, block_tables, block_table_stride, seq_lens, query_start_loc, num_requests,
                      num_tokens, num_heads, max_query_len, max_seq_len, dcp_world, scale, out, out_dtype, lse,
                      nullptr, num_splits, workspace, workspace_bytes, stream);
}

int mla_dcp_decode_fp8(const void* q_nope, int64_t q_nope_row_stride, const void* q_pe, int64_t q_pe_row_stride,
                       const void* kv_cache, int64_t num_blocks, int32_t page_size, float kv_scale,
                       const int32_t* block_table, int32_t block_table_stride, const int32_t* seq_lens,
                       const int32_t* query_start_loc, int32_t num_requests, int32_t num_tokens, int32_t num_heads,
                       int32_t max_query_len, int32_t max_seq_len, int32_t dcp_world, int32_t dcp_rank, float scale,
                       void* out, int32_t out_dtype, float* lse, int32_t* row_counts, int32_t num_splits,
                       void* workspace, size_t workspace_bytes, void* stream) {
  if (!std::isfinite(kv_scale) || !(kv_scale > 0.f))
    return fail(MLA_ERR_INVALID_ARG, "kv_scale %g: a finite positive dequantisation scale is required", kv_scale);
  int rc = check_decode_common(q_nope, q_nope_row_stride, q_pe, q_pe_row_stride, kv_cache, num_blocks, page_size,
                               MLA_DTYPE_FP8_E4M3, block_table, block_table_stride, seq_lens, query_start_loc,
                               num_requests, num_tokens, num_heads, dcp_world, dcp_rank, scale, out, out_dtype, lse,
                               workspace, true);
  if (rc != MLA_OK) return rc;
  const void* kvs[1] = {kv_cache};
  const int64_t nbs[1] = {num_blocks};
  const int32_t* bts[1] = {block_table};
  return dense_decode(q_nope, q_nope_row_stride, q_pe, q_pe_row_stride, 1, dcp_rank, kvs, nbs, page_size, bts,
                      block_table_stride, seq_lens, query_start_loc, num_requests, num_tokens, num_heads,
                      max_query_len, max_seq_len, dcp_world, scale, out, out_dtype, lse, row_counts, num_splits,
                      workspace, workspace_bytes, stream, true, kv_scale);
}

int mla_dcp_decode_fused_fp8(const void* q_nope, int64_t q_nope_row_stride, const void* q_pe,
                             int64_t q_pe_row_stride, const void* const* kv_caches, const int64_t* num_blocks,
                             int32_t page_size, float kv_scale, const int32_t* const* block_tables,
                             int32_t block_table_stride, const int32_t* seq_lens, const int32_t* query_start_loc,
                             int32_t num_requests, int32_t num_tokens, int32_t num_heads, int32_t max_query_len,
                             int32_t max_seq_len, int32_t dcp_world, float scale, void* out, int32_t out_dtype,
                             float* lse, int32_t num_splits, void* workspace, size_t workspace_bytes, void* stream) {
  if (dcp_world < 1 || dcp_world > mla::kMaxShards)
    return fail(MLA_ERR_INVALID_ARG, "dcp_world %d not in [1, %d] for the fused call", dcp_world, mla::kMaxShards);
  if (kv_caches == nullptr || num_blocks == nullptr || block_tables == nullptr)
    return fail(MLA_ERR_INVALID_ARG, "kv_caches / num_blocks / block_tables arrays are NULL");
  if (!std::isfinite(kv_scale) || !(kv_scale > 0.f))
    return fail(MLA_ERR_INVALID_ARG, "kv_scale %g: a finite positive dequantisation scale is required", kv_scale);
  for (int r = 0; r < dcp_world; ++r) {
    int rc = check_decode_common(q_nope, q_nope_row_stride, q_pe, q_pe_row_stride, kv_caches[r], num_blocks[r],
                                 page_size, MLA_DTYPE_FP8_E4M3, block_tables[r], block_table_stride, seq_lens,
                                 query_start_loc, num_requests, num_tokens, num_heads, dcp_world, r, scale, out,
                                 out_dtype, lse, workspace, true);
    if (rc != MLA_OK) return rc;
  }
  return dense_decode(q_nope, q_nope_row_stride, q_pe, q_pe_row_stride, dcp_world, 0, kv_caches, num_blocks,
                      page_size, block_tables, block_table_stride, seq_lens, query_start_loc, num_requests,
                      num_tokens, num_heads, max_query_len, max_seq_len, dcp_world, scale, out, out_dtype, lse,
                      nullptr, num_splits, workspace, workspace_bytes, stream, true, kv_scale);
}

size_t mla_sparse_dcp_decode_workspace_size(int32_t num_tokens, int32_t num_heads, int32_t topk, int32_t dcp_world) {
  (void)dcp_world;
  return mla::make_sparse_plan(num_tokens, num_heads, topk, current_sm_count()).total;
}

int mla_sparse_dcp_decode(const void* q_nope, int64_t q_nope_row_stride, const void* q_pe, int64_t q_pe_row_stride,
                          const void* kv_cache, int64_t num_blocks, int32_t page_size, int32_t kv_cache_dtype,
                          const int32_t* block_table, int32_t block_table_stride, const int32_t* seq_lens,
                          const int32_t* query_start_loc, int32_t num_requests, int32_t num_tokens,
                          int32_t num_heads, const int32_t* topk_indices, int32_t topk, const int32_t* topk_valid,
                          int32_t dcp_world, int32_t dcp_rank, float scale, void* out, int32_t out_dtype,
                          float* lse, int32_t* local_counts, void* workspace, size_t workspace_bytes,
                          void* stream) {
  int rc = check_decode_common(q_nope, q_nope_row_stride, q_pe, q_pe_row_stride, kv_cache, num_blocks, page_size,
                               kv_cache_dtype, block_table, block_table_stride, seq_lens, query_start_loc,
                               num_requests, num_tokens, num_heads, dcp_world, dcp_rank, scale, out, out_dtype, lse,
                               workspace);
  if (rc != MLA_OK) return rc;
  if (!local_counts) return fail(MLA_ERR_INVALID_ARG, "local_counts is required");
  return sparse_decode(q_nope, q_nope_row_stride, q_pe, q_pe_row_stride, 1, dcp_rank, &kv_cache, &num_blocks,
                       page_size, &block_table, block_table_stride, seq_lens, query_start_loc, num_requests,
                       num_tokens, num_heads, topk_indices, topk, topk_valid, dcp_world, scale, out, out_dtype, lse,
                       local_counts, workspace, workspace_bytes, stream);
}

int mla_sparse_dcp_decode_fused(const void* q_nope, int64_t q_nope_row_stride, const void* q_pe,
                                int64_t q_pe_row_stride, const void* const* kv_caches, const int64_t* num_blocks,
                                int32_t page_size, int32_t kv_cache_dtype, const int32_t* const* block_tables,
                                int32_t block_table_stride, const int32_t* seq_lens, const int32_t* query_start_loc,
                                int32_t num_requests, int32_t num_tokens, int32_t num_heads,
                                const int32_t* topk_indices, int32_t topk, const int32_t* topk_valid,
                                int32_t dcp_world, float scale, void* out, int32_t out_dtype, float* lse,
                                int32_t* kept_counts, void* workspace, size_t workspace_bytes, void* stream) {
  if (dcp_world < 1 || dcp_world > mla::kMaxShards)
    return fail(MLA_ERR_INVALID_ARG, "dcp_world %d not in [1, %d] for the fused call", dcp_world, mla::kMaxShards);
  if (!kv_caches || !num_blocks || !block_tables)
    return fail(MLA_ERR_INVALID_ARG, "kv_caches, num_blocks and block_tables are required");
  for (int r = 0; r < dcp_world; ++r) {
    int rc = check_decode_common(q_nope, q_nope_row_stride, q_pe, q_pe_row_stride, kv_caches[r], num_blocks[r],
                                 page_size, kv_cache_dtype, block_tables[r], block_table_stride, seq_lens,
                                 query_start_loc, num_requests, num_tokens, num_heads, dcp_world, r, scale, out,
                                 out_dtype, lse, workspace);
    if (rc != MLA_OK) return rc;
  }
  return sparse_decode(q_nope, q_nope_row_stride, q_pe, q_pe_row_stride, dcp_world, 0, kv_caches, num_blocks,
                       page_size, block_tables, block_table_stride, seq_lens, query_start_loc, num_requests,
                       num_tokens, num_heads, topk_indices, topk, topk_valid, dcp_world, scale, out, out_dtype, lse,
                       kept_counts, workspace, workspace_bytes, stream);
}

}  // extern "C"

namespace {

// Where the two-stage call keeps its pieces inside its workspace (byte
// offsets, 256-byte aligned): the first stage's dense workspace at 0 (its
// status word is the call's), the second stage's sparse workspace, the two
// stages' fp32 results and LSEs (the merge's two partials), and the device
// inputs the prep kernel derives.
struct TwoStageLayout {
  size_t sparse, parts, lses, lists, valid, ctx, total;
};

TwoStageLayout two_stage_layout(int32_t num_requests, int32_t num_tokens, int32_t num_heads, int32_t max_query_len,
                                int32_t max_seq_len) {
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t T = num_tokens > 0 ? (size_t)num_tokens : 0, H = num_heads > 0 ? (size_t)num_heads : 0;
  const size_t B = num_requests > 0 ? (size_t)num_requests : 0;
  const size_t W = max_query_len > 0 ? (size_t)max_query_len : 1;
  TwoStageLayout L;
  L.sparse = al(dense_workspace_bytes(num_requests, num_tokens, num_heads, max_query_len, max_seq_len, 1, 0));
  L.parts = L.sparse + al(mla::make_sparse_plan(num_tokens, num_heads, (int32_t)W, current_sm_count()).total);
  L.lses = L.parts + al(2 * T * H * mla::kNope * sizeof(float));
  L.lists = L.lses + al(2 * T * H * sizeof(float));
  L.valid = L.lists + al(T * W * sizeof(int32_t));
  L.ctx = L.valid + al(T * sizeof(int32_t));
  L.total = L.ctx + al(B * sizeof(int32_t));
  return L;
}

}  // namespace

extern "C" {

size_t mla_dcp_decode_two_stage_workspace_size(int32_t num_requests, int32_t num_tokens, int32_t num_heads,
                                               int32_t max_query_len, int32_t max_seq_len) {
  return two_stage_layout(num_requests, num_tokens, num_heads, max_query_len, max_seq_len).total;
}

int mla_dcp_decode_two_stage(const void* q_nope, int64_t q_nope_row_stride, const void* q_pe, int64_t q_pe_row_stride,
                             const void* const* kv_caches, const int64_t* num_blocks, int32_t page_size,
                             int32_t kv_cache_dtype, const int32_t* const* block_tables, int32_t block_table_stride,
                             const int32_t* seq_lens, const int32_t* query_start_loc, int32_t num_requests,
                             int32_t num_tokens, int32_t num_heads, int32_t max_query_len, int32_t max_seq_len,
                             int32_t dcp_world, float scale, void* out, int32_t out_dtype, float* lse,
                             void* workspace, size_t workspace_bytes, void* stream) {
  if (dcp_world < 1 || dcp_world > mla::kMaxShards)
    return fail(MLA_ERR_INVALID_ARG, "dcp_world %d not in [1, %d] for the two-stage call", dcp_world,
                mla::kMaxShards);
  if (kv_caches == nullptr || num_blocks == nullptr || block_tables == nullptr)
    return fail(MLA_ERR_INVALID_ARG, "kv_caches / num_blocks / block_tables arrays are NULL");
  for (int r = 0; r < dcp_world; ++r) {
    int rc = check_decode_common(q_nope, q_nope_row_stride, q_pe, q_pe_row_stride, kv_caches[r], num_blocks[r],
                                 page_size, kv_cache_dtype, block_tables[r], block_table_stride, seq_lens,
                                 query_start_loc, num_requests, num_tokens, num_heads, dcp_world, r, scale, out,
                                 out_dtype, lse, workspace);
    if (rc != MLA_OK) return rc;
  }
  if (max_seq_len < 0) return fail(MLA_ERR_INVALID_ARG, "max_seq_len %d < 0", max_seq_len);
  if (num_tokens == 0) return ok();
  if (max_query_len < 1 || max_query_len > 65536)
    return fail(MLA_ERR_INVALID_ARG, "max_query_len %d not in [1, 65536]", max_query_len);
  const TwoStageLayout L = two_stage_layout(num_requests, num_tokens, num_heads, max_query_len, max_seq_len);
  if (workspace_bytes < L.total)
    return fail(MLA_ERR_WORKSPACE, "workspace %zu bytes < %zu required", workspace_bytes, L.total);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* parts = reinterpret_cast<float*>(ws + L.parts);
  float* lses = reinterpret_cast<float*>(ws + L.lses);
  const int64_t rows = (int64_t)num_tokens * num_heads;

  mla::TwoStageArgs ta{};
  ta.seq_lens = seq_lens;
  ta.query_start_loc = query_start_loc;
  ta.num_requests = num_requests;
  ta.num_tokens = num_tokens;
  ta.list_stride = max_query_len;
  ta.ctx_lens = reinterpret_cast<int32_t*>(ws + L.ctx);
  ta.new_keys = reinterpret_cast<int32_t*>(ws + L.lists);
  ta.new_valid = reinterpret_cast<int32_t*>(ws + L.valid);
  cudaError_t e = mla::launch_two_stage_prep(ta, st);
  if (e != cudaSuccess) return cuda_fail(e, "two-stage prep launch");
  count_launch();
  // stage 1: every query row over its request's whole context, no mask
  int rc = dense_decode(q_nope, q_nope_row_stride, q_pe, q_pe_row_stride, dcp_world, 0, kv_caches, num_blocks,
                        page_size, block_tables, block_table_stride, ta.ctx_lens, query_start_loc, num_requests,
                        num_tokens, num_heads, max_query_len, max_seq_len, dcp_world, scale, parts, MLA_DTYPE_F32,
                        lses, nullptr, 0, ws, L.sparse, stream, false, 1.f, /*causal=*/false);
  if (rc != MLA_OK) return rc;
  // stage 2: every query row over the new keys up to its own position
  rc = sparse_decode(q_nope, q_nope_row_stride, q_pe, q_pe_row_stride, dcp_world, 0, kv_caches, num_blocks,
                     page_size, block_tables, block_table_stride, seq_lens, query_start_loc, num_requests, num_tokens,
                     num_heads, ta.new_keys, max_query_len, ta.new_valid, dcp_world, scale, parts + rows * mla::kNope,
                     MLA_DTYPE_F32, lses + rows, nullptr, ws + L.sparse, L.parts - L.sparse, stream);
  if (rc != MLA_OK) return rc;
  e = mla::launch_fold_status(reinterpret_cast<mla::WorkspaceHeader*>(ws),
                              reinterpret_cast<const mla::WorkspaceHeader*>(ws + L.sparse), st);
  if (e != cudaSuccess) return cuda_fail(e, "status fold launch");
  count_launch();
  // the two stages' results merged by LSE (a row without context keys has
  // lse -inf and output 0 from stage 1: weight 0)
  mla::MergeArgs ma{};
  ma.partials = parts;
  ma.partial_f32 = 1;
  ma.lses = lses;
  ma.valid_counts = nullptr;
  ma.w_uv = nullptr;
  ma.dcp_world = 2;
  ma.num_tokens = num_tokens;
  ma.num_heads = num_heads;
  ma.out = out;
  ma.out_f32 = out_dtype == MLA_DTYPE_F32;
  ma.lse_out = lse;
  ma.num_sms = current_sm_count();
  e = mla::launch_merge(ma, st);
  if (e != cudaSuccess) return cuda_fail(e, "merge launch");
  count_launch();
  return ok();
}

int dcp_lse_merge(const void* partials, int32_t partial_dtype, const float* lses, const int32_t* valid_counts,
                  const void* w_uv, int32_t dcp_world, int32_t num_tokens, int32_t num_heads, void* out,
                  int32_t out_dtype, float* lse_out, void* stream) {
  if (dcp_world < 1 || dcp_world > 64) return fail(MLA_ERR_INVALID_ARG, "dcp_world %d not in [1, 64]", dcp_world);
  if (num_tokens < 0 || num_heads < 1 || num_heads > mla::kMaxHeads)
    return fail(MLA_ERR_INVALID_ARG, "bad sizes: num_tokens=%d num_heads=%d", num_tokens, num_heads);
  if (!partials || !lses || !out) return fail(MLA_ERR_INVALID_ARG, "partials, lses and out are required");
  if (partial_dtype != MLA_DTYPE_BF16 && partial_dtype != MLA_DTYPE_F32)
    return fail(MLA_ERR_INVALID_ARG, "partial_dtype %d: BF16 or F32", partial_dtype);
  if (out_dtype != MLA_DTYPE_BF16 && out_dtype != MLA_DTYPE_F32)
    return fail(MLA_ERR_INVALID_ARG, "out_dtype %d: BF16 or F32", out_dtype);
  if (!aligned(partials, 16) || !aligned(out, 16) || !aligned(lses, 4) || (w_uv && !aligned(w_uv, 16)))
    return fail(MLA_ERR_INVALID_ARG, "misaligned pointer (partials/out/w_uv need 16-byte alignment)");
  if (num_tokens == 0) return ok();
  mla::MergeArgs ma{};
  ma.partials = partials;
  ma.partial_f32 = partial_dtype == MLA_DTYPE_F32;
  ma.lses = lses;
  ma.valid_counts = valid_counts;
  ma.w_uv = static_cast<const __nv_bfloat16*>(w_uv);
  ma.dcp_world = dcp_world;
  ma.num_tokens = num_tokens;
  ma.num_heads = num_heads;
  ma.out = out;
  ma.out_f32 = out_dtype == MLA_DTYPE_F32;
  ma.lse_out = lse_out;
  ma.num_sms = current_sm_count();
  cudaError_t e = mla::launch_merge(ma, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "merge launch");
  count_launch();
  return ok();
}

int64_t mla_kernel_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

void mla_debug_set_wait_budget_ns(uint64_t ns) { g_wait_budget_ns.store(ns, std::memory_order_relaxed); }

int mla_workspace_status(const void* workspace, void* stream, int32_t* detail) {
  if (!workspace) return fail(MLA_ERR_INVALID_ARG, "workspace is NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  int32_t h[2] = {0, 0};
  e = cudaMemcpy(h, workspace, sizeof h, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  if (detail) *detail = h[1];
  if (h[0] != 0) return fail(MLA_ERR_DEVICE_CHECK, "device check %d fired", h[1]);
  return ok();
}

}  // extern "C"
