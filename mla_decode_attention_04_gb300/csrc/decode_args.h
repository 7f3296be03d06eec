// decode_args.h -- argument block shared by the dense and sparse decode kernels.
#pragma once

#include "common.cuh"

namespace mla {

struct DecodeArgs {
  const __nv_bfloat16* q_nope;
  int64_t q_nope_stride;  // elements between consecutive (token, head) rows
  const __nv_bfloat16* q_pe;
  int64_t q_pe_stride;
  const __nv_bfloat16* kv;  // shard 0's cache (sparse: the source of zero-length copies)
  int32_t page_size;
  int32_t bt_stride;
  // dense: the call covers shards shard0 .. shard0 + nshard - 1 (one shard,
  // or all D when fused); shard k's cache pages and block table
  int32_t nshard, shard0;
  const __nv_bfloat16* kvs[kMaxShards];
  const int32_t* bts[kMaxShards];
  int64_t nblocks[kMaxShards];
  int32_t num_heads, dcp_world;
  float scale;
  // 1: the caches hold FP8 E4M3 codes (576 bytes per row), value =
  // kv_scale * decode(code); 0: bf16 (kv_scale 1)
  int32_t kv_fp8;
  float kv_scale;
  // budget of each pipeline wait in ns (2 s unless a test shortens it);
  // waits for copies already in flight when a role gave up have their own
  uint64_t wait_ns;
  // 1: every row sees every key of its request (seq_lens then hold the
  // context lengths: the first pass of the two-stage decomposition)
  int32_t noncausal;
  void* out;  // [T, H, 512]
  int32_t out_f32;
  float* lse;  // [T, H]
  WorkspaceHeader* hdr;
  // the requests (dense: every CTA derives the split plan from them)
  const int32_t* seq_lens;
  const int32_t* query_start_loc;
  int32_t num_requests;
  int32_t unit_penalty;
  // CTAs per gang (1: no gangs).  With gangs of S CTAs, gang j takes a range
  // of the requests' key tiles and its CTA g runs row group g of each
  // request over that range, so the S row groups read each tile at about
  // the same time (one HBM read serves them all through L2).
  int32_t gang;
  int4* split_desc;  // [grid] the split pair whose first chunk CTA c holds: {chunks, first row, rows, 0}
  float* part_lse;   // [2 grid NR]
  float* part_o;     // [2 grid NR, 512]
  // sparse (the split plan's sources are the tokens)
  const int64_t* key_rows;    // [T, list_stride] cache-row addresses of each token's keys
  const int32_t* list_count;  // [T]
  int32_t list_stride;
  int32_t num_tokens;
};

}  // namespace mla
