// decode_args.h -- argument block shared by the dense and sparse decode kernels.
#pragma once

#include "common.cuh"

namespace mla {

struct DecodeArgs {
  const __nv_bfloat16* q_nope;
  int64_t q_nope_stride;  // elements between consecutive (token, head) rows
  const __nv_bfloat16* q_pe;
  int64_t q_pe_stride;
  const __nv_bfloat16* kv;  // [num_blocks, page_size, 576]
  int64_t num_blocks;
  int32_t page_size;
  const int32_t* block_table;
  int32_t bt_stride;
  int32_t num_heads, dcp_world, dcp_rank;
  float scale;
  void* out;  // [T, H, 512]
  int32_t out_f32;
  float* lse;  // [T, H]
  WorkspaceHeader* hdr;
  // dense
  const ReqInfo* req;
  const PairInfo* pairs;
  int32_t* pair_done;  // finished KV chunks per pair (the last finisher merges)
  const int32_t* cta_pair0;  // pair holding the first item of each CTA's range
  float* part_lse;
  float* part_o;
  // sparse
  const int32_t* lists;       // [T, list_stride] shard-local slots
  const int32_t* list_count;  // [T]
  const int32_t* tok_req;     // [T] owning request
  int32_t list_stride;
  int32_t num_tokens;
  int32_t groups_per_token;
};

}  // namespace mla
