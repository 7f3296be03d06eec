// decode_kernels.h -- launchers of the decode, sparse-list and merge kernels.
#pragma once

#include <cuda_runtime.h>

#include "decode_args.h"

namespace mla {

// Tensor-core decode: min(max_units, num_sms) persistent CTAs over the
// scheduler's balanced key-tile ranges (dense; max_units must then equal the
// grid the scheduler planned for) or over the T * groups (token, head group)
// units (sparse).
cudaError_t launch_decode_tc(const DecodeArgs& a, int rows_per_group, bool sparse, int max_units, int num_sms,
                             cudaStream_t stream);

// The sparse decode's key lists: for every token, the cache-row addresses
// of the entries it keeps on shards shard0 .. shard0 + nshard - 1 (one
// shard's call, or all D when fused), resolved through that shard's block
// table once here instead of once per head group in the decode.
struct SparseListArgs {
  const int32_t* topk;        // [T, K]
  const int32_t* topk_valid;  // [T]
  const int32_t* seq_lens;
  const int32_t* query_start_loc;
  int32_t num_requests, num_tokens, topk_k, dcp_world;
  int32_t shard0, nshard;
  const void* kvs[kMaxShards];      // shard caches [num_blocks, page_size, 576] bf16
  const int32_t* bts[kMaxShards];   // shard block tables [B, bt_stride]
  int64_t nblocks[kMaxShards];
  int32_t page_size, bt_stride;
  int64_t* key_rows;  // [T, K] out: device addresses of the kept entries' cache rows, in list order
  int32_t* counts;    // [T] out: entries kept
  WorkspaceHeader* hdr;
  // the final rows (o = 0, lse = -inf) of tokens that keep no entry (the
  // decode has no unit for them)
  int32_t num_heads;
  void* out;  // [T, H, 512]
  int32_t out_f32;
  float* lse;  // [T, H]
};
cudaError_t launch_sparse_lists(const SparseListArgs& a, cudaStream_t stream);

struct MergeArgs {
  const void* partials;  // [D, T, H, 512]
  int32_t partial_f32;
  const float* lses;             // [D, T, H]
  const int32_t* valid_counts;   // [D, T] or NULL
  const __nv_bfloat16* w_uv;     // [H, 512, 128] or NULL
  int32_t dcp_world, num_tokens, num_heads;
  void* out;
  int32_t out_f32;
  float* lse_out;  // or NULL
  int32_t num_sms;  // SMs of the device (grid sizing)
};
cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream);
// W_UV-fused merge on tensor cores (CTAs per head, each over blocks of 32 tokens).
cudaError_t launch_merge_wuv_tc(const MergeArgs& a, cudaStream_t stream);

// Device inputs of the two-stage decomposition: ctx_lens[b] = L_b - q_len_b,
// new_keys[t][j] = the j-th new-key position of token t (-1 past its own
// position), new_valid[t] = its count.
struct TwoStageArgs {
  const int32_t* seq_lens;
  const int32_t* query_start_loc;
  int32_t num_requests, num_tokens;
  int32_t list_stride;  // >= the largest q_len
  int32_t* ctx_lens;    // [num_requests]
  int32_t* new_keys;    // [num_tokens, list_stride]
  int32_t* new_valid;   // [num_tokens]
};
cudaError_t launch_two_stage_prep(const TwoStageArgs& a, cudaStream_t stream);
// main->status takes other's first failure when main has none.
cudaError_t launch_fold_status(WorkspaceHeader* main, const WorkspaceHeader* other, cudaStream_t stream);

}  // namespace mla
