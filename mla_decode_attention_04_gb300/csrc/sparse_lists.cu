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
// table at column slot div page_size).
#include "common.cuh"
#include "decode_kernels.h"
#include "pdl_launch.h"

namespace mla {

// One block of 256 threads per token.  A pass covers 2048 entries: warp w
// takes entries [256 w, 256 w + 256) of the pass in 8 rounds of 32; all
// list entries of a thread are loaded first, then all their block-table
// entries, so each pass costs two memory latencies whatever the list length.
// Kept entries are compacted in list order (ballot within a warp, then the
// warps' counts in order).
constexpr int kListThreads = 256;
constexpr int kListRounds = 8;
constexpr int kListPass = kListThreads * kListRounds;  // entries per pass

__global__ void __launch_bounds__(kListThreads) sparse_lists_kernel(SparseListArgs a) {
  grid_dep_sync();
  __shared__ int s_warp[kListThreads / 32];
  __shared__ int s_bad;
  const int t = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) s_bad = 0;
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
  const int P = L - q_len + (t - q0);
  if (q_len <= 0 || q_len > L || t >= q1) {
    if (tid == 0) record_check(a.hdr, kCheckBadQueryLayout);
    valid = 0;
  }
  const int D = a.dcp_world, ps = a.page_size;
  const int32_t* src = a.topk + (int64_t)t * a.topk_k;
  int64_t* dst = a.key_rows + (int64_t)t * a.topk_k;
  __syncthreads();
  int count = 0;  // entries kept by earlier passes (the same in every thread)
  for (int base = 0; base < valid; base += kListPass) {
    int idx[kListRounds], k[kListRounds], page[kListRounds];
#pragma unroll
    for (int r = 0; r < kListRounds; ++r) {
      const int e = base + warp * (32 * kListRounds) + r * 32 + lane;
      idx[r] = e < valid ? src[e] : -1;
    }
#pragma unroll
    for (int r = 0; r < kListRounds; ++r) {
      k[r] = idx[r] >= 0 ? idx[r] % D - a.shard0 : -1;  // shard index within the call
      const bool used = idx[r] >= 0 && idx[r] <= P && k[r] >= 0 && k[r] < a.nshard;
      page[r] = -2;  // not used
      if (used) {
        const int col = (idx[r] / D) / ps;
        page[r] = col < a.bt_stride ? pick_shard(a.bts, k[r])[(int64_t)b * a.bt_stride + col] : -1;
      }
    }
    int64_t row[kListRounds];
    int pos[kListRounds];
    int wcount = 0;
#pragma unroll
    for (int r = 0; r < kListRounds; ++r) {
      bool keep = page[r] != -2;
      row[r] = 0;
      if (keep) {
        if (page[r] < 0 || page[r] >= pick_shard(a.nblocks, k[r])) {
          s_bad = 1;  // the entry is dropped; the call reports check 1
          keep = false;
        } else {
          const int j = idx[r] / D;
          row[r] = (int64_t)reinterpret_cast<uintptr_t>(pick_shard(a.kvs, k[r])) +
                   ((int64_t)page[r] * ps + j % ps) * (int64_t)(kRow * 2);
        }
      }
      const unsigned m = __ballot_sync(0xffffffffu, keep);
      pos[r] = keep ? wcount + __popc(m & ((1u << lane) - 1u)) : -1;
      wcount += __popc(m);
    }
    if (lane == 0) s_warp[warp] = wcount;
    __syncthreads();
    int before = 0, total = 0;
#pragma unroll
    for (int w = 0; w < kListThreads / 32; ++w) {
      const int c = s_warp[w];
      if (w < warp) before += c;
      total += c;
    }
#pragma unroll
    for (int r = 0; r < kListRounds; ++r)
      if (pos[r] >= 0) dst[count + before + pos[r]] = row[r];
    count += total;
    __syncthreads();  // s_warp is reused by the next pass
  }
  if (tid == 0) {
    if (s_bad) record_check(a.hdr, kCheckPageOutOfRange);
    a.counts[t] = count;
  }
  if (count == 0) {
    // no key: the token's final rows (the decode has no unit for them)
    for (int h = warp; h < a.num_heads; h += kListThreads / 32) {
      const int64_t grow = (int64_t)t * a.num_heads + h;
      if (lane == 0) a.lse[grow] = -INFINITY;
      if (a.out_f32) {
        float4* o = reinterpret_cast<float4*>(static_cast<float*>(a.out) + grow * kNope);
        for (int q = lane; q < kNope / 4; q += 32) o[q] = make_float4(0.f, 0.f, 0.f, 0.f);
      } else {
        uint4* o = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + grow * kNope);
        for (int q = lane; q < kNope / 8; q += 32) o[q] = make_uint4(0, 0, 0, 0);
      }
    }
  }
}

cudaError_t launch_sparse_lists(const SparseListArgs& a, cudaStream_t stream) {
  if (a.num_tokens <= 0) return cudaSuccess;
  return launch_pdl(sparse_lists_kernel, dim3(a.num_tokens), dim3(kListThreads), 0, stream, a);
}

}  // namespace mla
