// plan.h -- host-side split plan, workspace layout and kernel argument blocks.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace mla {

struct SchedArgs {
  const int32_t* seq_lens;
  const int32_t* query_start_loc;
  int32_t num_requests, num_tokens, num_heads, dcp_world, dcp_rank;
  int32_t rows_per_group, max_splits, target_tiles, max_tiles, max_partial_rows;
  WorkspaceHeader* hdr;
  ReqInfo* req;
  Tile* tiles;
  int32_t* tok2req;
  int32_t* row_counts;  // may be NULL
};

struct CombineArgs {
  const ReqInfo* req;
  const int32_t* tok2req;
  const float* part_lse;
  const float* part_o;
  int32_t num_tokens, num_heads;
  void* out;
  int32_t out_f32;
  float* lse;
};

// Where everything lives inside a dense-decode workspace (byte offsets).
struct DecodePlan {
  int32_t rows_per_group;   // rows (token, head) per tile: 16 or 32
  int32_t max_splits;       // KV chunks per request at most
  int32_t target_tiles;     // scheduler aims at this many tiles
  int32_t max_tiles;        // capacity of the tile list
  int64_t max_partial_rows; // capacity of the split partials
  size_t off_req, off_tok, off_tiles, off_plse, off_po, total;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline DecodePlan make_decode_plan(int32_t B, int32_t T, int32_t H, int32_t max_query_len, int32_t max_seq_len,
                                   int32_t D, int32_t num_splits, int32_t num_sms) {
  DecodePlan p{};
  if (max_query_len < 1) max_query_len = 1;
  p.rows_per_group = (int64_t)max_query_len * H <= 16 ? 16 : 32;
  const int64_t NR = p.rows_per_group;
  p.target_tiles = 2 * (num_sms > 0 ? num_sms : 148);
  const int64_t max_local = (max_seq_len + D - 1) / (D > 0 ? D : 1);
  const int64_t max_key_tiles = (max_local + kKeyTile - 1) / kKeyTile;
  const int64_t groups_lb = ((int64_t)T * H + NR - 1) / NR;
  int64_t ms;
  if (num_splits > 0) {
    ms = num_splits;
  } else {
    ms = (p.target_tiles + (groups_lb > 0 ? groups_lb : 1) - 1) / (groups_lb > 0 ? groups_lb : 1);
    if (ms > 64) ms = 64;
  }
  if (ms > max_key_tiles) ms = max_key_tiles;
  if (ms < 1) ms = 1;
  p.max_splits = (int32_t)ms;
  p.max_tiles = (int32_t)((groups_lb + B) * ms);
  p.max_partial_rows = ms > 1 ? ms * (int64_t)T * H : 0;
  size_t off = sizeof(WorkspaceHeader);
  p.off_req = off;
  off = align_up(off + sizeof(ReqInfo) * (size_t)(B > 0 ? B : 1), 256);
  p.off_tok = off;
  off = align_up(off + sizeof(int32_t) * (size_t)(T > 0 ? T : 1), 256);
  p.off_tiles = off;
  off = align_up(off + sizeof(Tile) * (size_t)(p.max_tiles > 0 ? p.max_tiles : 1), 256);
  p.off_plse = off;
  off = align_up(off + sizeof(float) * (size_t)p.max_partial_rows, 256);
  p.off_po = off;
  off = align_up(off + sizeof(float) * kNope * (size_t)p.max_partial_rows, 256);
  p.total = off;
  return p;
}

// Sparse decode workspace: header, then the per-token shard-local key lists.
struct SparsePlan {
  int32_t rows_per_group;
  size_t off_tok, off_lists, total;
};

inline SparsePlan make_sparse_plan(int32_t T, int32_t H, int32_t topk) {
  SparsePlan p{};
  p.rows_per_group = H <= 16 ? 16 : 32;
  const size_t nt = (size_t)(T > 0 ? T : 1);
  p.off_tok = sizeof(WorkspaceHeader);
  p.off_lists = align_up(p.off_tok + sizeof(int32_t) * nt, 256);
  p.total = align_up(p.off_lists + sizeof(int32_t) * nt * (size_t)(topk > 0 ? topk : 1), 256);
  return p;
}

__global__ void schedule_kernel(SchedArgs a);
__global__ void combine_kernel(CombineArgs a);

}  // namespace mla
