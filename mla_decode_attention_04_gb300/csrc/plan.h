// plan.h -- host-side workspace layout of the decode calls and the argument
// block of the dense prep kernel.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace mla {

struct PrepArgs {
  const int32_t* seq_lens;
  const int32_t* query_start_loc;
  int32_t num_requests, num_tokens, num_heads, dcp_world;
  int32_t shard0, nshard;  // the shards the decode covers (one, or all D when fused)
  int32_t rows_per_group;
  int32_t noncausal;  // every row sees every key of its request
  WorkspaceHeader* hdr;
  int32_t* row_counts;  // may be NULL
  // rows of requests without local keys get their final result here
  void* out;
  int32_t out_f32;
  float* lse;
};

// Where everything lives inside a dense-decode workspace (byte offsets).
// Split partials are addressed by decode CTA (chunk_slot): CTA c owns rows
// [2 c NR, 2 c NR + NR) for the chunk its first unit continues and
// [(2 c + 1) NR, (2 c + 2) NR) for the chunk its last unit starts; entry c
// of the split table describes the pair whose first chunk CTA c holds.
struct DecodePlan {
  int32_t rows_per_group;  // rows (token, head) per work unit: 16, 32 or 64
  int32_t grid;            // decode CTAs
  int32_t unit_penalty;    // balancing cost of a unit start, in 64-key tiles
  int32_t gang;            // CTAs per gang (1: none); grid is a multiple of it
  size_t off_desc, off_plse, off_po, total;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Rows (token, head) per decode work unit for a request (or token) of up to
// `rows` rows: the fewest of 16, 32, 64 that hold them (64 at most; more
// rows form several units, each of which streams the keys).  Bigger units
// read each key tile for more rows.
inline int32_t rows_per_unit(int64_t rows) { return rows <= 16 ? 16 : rows <= 32 ? 32 : 64; }

inline DecodePlan make_decode_plan(int32_t B, int32_t T, int32_t H, int32_t max_query_len, int32_t max_seq_len,
                                   int32_t D, int32_t num_splits, int32_t num_sms, bool kv_fp8 = false) {
  DecodePlan p{};
  if (max_query_len < 1) max_query_len = 1;  // the backend's capture-time clamp
  if (D < 1) D = 1;
  p.rows_per_group = rows_per_unit((int64_t)max_query_len * H);
  // an FP8 cache adds four converter warps, whose registers the 64-row
  // softmax cannot spare: units of up to 32 rows
  if (kv_fp8 && p.rows_per_group > 32) p.rows_per_group = 32;
  p.unit_penalty = kUnitPenalty;
  const int64_t NR = p.rows_per_group;
  const int64_t max_local = (max_seq_len + D - 1) / D;
  const int64_t max_key_tiles = (max_local + kKeyTile - 1) / kKeyTile;
  const int64_t groups_ub = ((int64_t)T * H + NR - 1) / NR + B;  // >= sum_b ceil(q_len_b H / NR)
  const int64_t items_ub = groups_ub * max_key_tiles;
  const int64_t sms = num_sms > 0 ? num_sms : 148;
  // Gangs: when a request has 2 to 8 row groups, the grid runs in gangs of
  // that many CTAs (one per row group) over shared tile ranges, so the row
  // groups' reads of a key tile come close together and L2 serves all but
  // the first.  Without gangs the groups of a request stream the same tiles
  // at different times, each from HBM.
  const int64_t groups_max = ((int64_t)max_query_len * H + NR - 1) / NR;
  p.gang = (groups_max >= 2 && groups_max <= 8 && groups_max * 2 <= sms) ? (int32_t)groups_max : 1;
  const int64_t S = p.gang;
  int64_t g = sms / S;  // gangs (or CTAs)
  // num_splits > 0 caps the grid at num_splits CTAs per row group (gangs:
  // per request); with balanced ranges a row group of average size is then
  // cut into about num_splits KV chunks
  if (num_splits > 0) {
    const int64_t units_lb = S > 1 ? ((int64_t)T + max_query_len - 1) / max_query_len : ((int64_t)T * H + NR - 1) / NR;
    const int64_t cap = (int64_t)num_splits * (units_lb > 0 ? units_lb : 1);
    if (g > cap) g = cap;
  }
  if (g > items_ub) g = items_ub;
  if (g < 1) g = 1;
  p.grid = (int32_t)(g * S);
  size_t off = sizeof(WorkspaceHeader);
  p.off_desc = off;
  off = align_up(off + 16 * (size_t)p.grid, 256);
  p.off_plse = off;
  off = align_up(off + sizeof(float) * 2 * (size_t)p.grid * NR, 256);
  p.off_po = off;
  off = align_up(off + sizeof(float) * kNope * 2 * (size_t)p.grid * NR, 256);
  p.total = off;
  return p;
}

// Sparse decode workspace: header, per-token key counts (used when the
// caller does not ask for them), per-token lists of
// cache-row addresses, and the split table and partials of the (token, head
// group) pairs the balanced plan cuts over CTAs (as in DecodePlan).
struct SparsePlan {
  int32_t rows_per_group;
  int32_t grid;  // decode CTAs
  size_t off_cnt, off_lists, off_desc, off_plse, off_po, total;
};

inline SparsePlan make_sparse_plan(int32_t T, int32_t H, int32_t topk, int32_t num_sms) {
  SparsePlan p{};
  p.rows_per_group = rows_per_unit(H);
  const size_t NR = (size_t)p.rows_per_group;
  p.grid = num_sms > 0 ? num_sms : 148;
  const size_t nt = (size_t)(T > 0 ? T : 1);
  p.off_cnt = sizeof(WorkspaceHeader);
  p.off_lists = align_up(p.off_cnt + sizeof(int32_t) * nt, 256);
  p.off_desc = align_up(p.off_lists + sizeof(int64_t) * nt * (size_t)(topk > 0 ? topk : 1), 256);
  p.off_plse = align_up(p.off_desc + 16 * (size_t)p.grid, 256);
  p.off_po = align_up(p.off_plse + sizeof(float) * 2 * (size_t)p.grid * NR, 256);
  p.total = align_up(p.off_po + sizeof(float) * kNope * 2 * (size_t)p.grid * NR, 256);
  return p;
}

__global__ void prep_kernel(PrepArgs a);

// The split-merge kernel: the LSE merge of the chunks of every row group the
// decode cut over several CTAs (entry c of the split table: {chunks, first
// global (token, head) row, rows, 0}; chunk k's partial rows at
// chunk_slot(c, k, NR, cta_stride)).  Block (c, s) merges rows [4 s, 4 s + 4) of entry c.
struct SplitMergeArgs {
  const int4* split_desc;  // [grid]
  const float* part_lse;   // [2 grid NR]
  const float* part_o;     // [2 grid NR, 512]
  int32_t rows_per_group, grid;
  int32_t cta_stride;      // CTAs between a pair's consecutive chunks (the gang size, or 1)
  int64_t num_rows;        // T * H
  void* out;               // [T, H, 512]
  int32_t out_f32;
  float* lse;              // [T, H]
  WorkspaceHeader* hdr;
};
constexpr int kSplitMergeRows = 4;  // rows per split-merge block

__global__ void split_merge_kernel(SplitMergeArgs a);

}  // namespace mla
