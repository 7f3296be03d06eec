// sparse_lists.cu -- per-token shard-local key lists of the sparse decode.
//
// Sparse MLA ("[Attention] DCP sparse MLA output-merge optimizations": per-row
// index lists with valid counts) under DCP: shard r of D keeps, in list
// order, the entries e < valid[t] whose global position idx satisfies
// 0 <= idx <= P (P = the token's own position) and idx mod D == r, and
// stores their local slots idx div D.  The count kept is the merge's
// per-row valid count.  One warp per token; order is kept with a ballot.
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
  const int D = a.dcp_world, r = a.dcp_rank;
  const int32_t* src = a.topk + (int64_t)t * a.topk_k;
  int32_t* dst = a.lists + (int64_t)t * a.topk_k;
  int count = 0;
  for (int e0 = 0; e0 < valid; e0 += 32) {
    const int e = e0 + lane;
    const int idx = e < valid ? src[e] : -1;
    const bool keep = idx >= 0 && idx <= P && idx % D == r;
    const unsigned m = __ballot_sync(0xffffffffu, keep);
    if (keep) dst[count + __popc(m & ((1u << lane) - 1u))] = idx / D;
    count += __popc(m);
  }
  if (lane == 0) {
    a.local_counts[t] = count;
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
