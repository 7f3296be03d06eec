// sparse_lists.cu -- per-token key lists of the sparse decode.
//
// Sparse MLA ("[Attention] DCP sparse MLA output-merge optimizations": per-row
// index lists with valid counts) under DCP: shard r of D keeps, in list
// order, the entries e < valid[t] whose global position idx satisfies
// 0 <= idx <= P (P = the token's own position) and idx mod D == r; its local
// slot is idx div D.  The count kept is the merge's per-row valid count.  A
// call covers shards shard0 .. shard0 + nshard - 1: one shard, or all D for
// the shard-fused call, whose list is then every kept entry of the token and
// whose attention over it is the merged result.  Each kept entry is resolved
// here, once, to the address of its cache row (page = the shard's block
// table at column slot div page_size).  One warp per token; order is kept
// with a ballot.
#include "common.cuh"
#include "decode_kernels.h"
#include "pdl_launch.h"

namespace mla {

__global__ void __launch_bounds__(256) sparse_lists_kernel(SparseListArgs a) {
  grid_dep_sync();
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= a.num_tokens) return;
  // owning request: the largest b with query_start_loc[b] <= t
  int lo = 0, hi = a.num_requests - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a.query_start_loc[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int b = lo;
  const int q0 = a.query_start_loc[b], q1 = a.query_start_loc[b + 1];
  const int L = a.seq_lens[b];
  const int q_len = q1 - q0;
  int valid = a.topk_valid[t];
  valid = valid < 0 ? 0 : (valid > a.topk_k ? a.topk_k : valid);
  int P = L - q_len + (t - q0);
  if (q_len <= 0 || q_len > L || t >= q1) {
    if (lane == 0) record_check(a.hdr, kCheckBadQueryLayout);
    valid = 0;
  }
  const int D = a.dcp_world, ps = a.page_size;
  const int32_t* src = a.topk + (int64_t)t * a.topk_k;
  int64_t* dst = a.key_rows + (int64_t)t * a.topk_k;
  int count = 0;
  bool bad = false;
  for (int e0 = 0; e0 < valid; e0 += 32) {
    const int e = e0 + lane;
    const int idx = e < valid ? src[e] : -1;
    const int k = idx >= 0 ? idx % D - a.shard0 : -1;  // shard index within the call
    bool keep = idx >= 0 && idx <= P && k >= 0 && k < a.nshard;
    int64_t row = 0;
    if (keep) {
      const int j = idx / D, col = j / ps;
      const int32_t* bt = pick_shard(a.bts, k);
      const int page = col < a.bt_stride ? bt[(int64_t)b * a.bt_stride + col] : -1;
      if (page < 0 || page >= pick_shard(a.nblocks, k)) {
        bad = true;  // the entry is dropped; the call reports check 1
        keep = false;
      } else {
        row = (int64_t)reinterpret_cast<uintptr_t>(pick_shard(a.kvs, k)) +
              ((int64_t)page * ps + j % ps) * (int64_t)(kRow * 2);
      }
    }
    const unsigned m = __ballot_sync(0xffffffffu, keep);
    if (keep) dst[count + __popc(m & ((1u << lane) - 1u))] = row;
    count += __popc(m);
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) record_check(a.hdr, kCheckPageOutOfRange);
  if (lane == 0) {
    a.counts[t] = count;
    a.tok_req[t] = b;
  }
}

cudaError_t launch_sparse_lists(const SparseListArgs& a, cudaStream_t stream) {
  if (a.num_tokens <= 0) return cudaSuccess;
  const int warps = 8;
  const int grid = (a.num_tokens + warps - 1) / warps;
  return launch_pdl(sparse_lists_kernel, dim3(grid), dim3(warps * 32), 0, stream, a);
}

}  // namespace mla
