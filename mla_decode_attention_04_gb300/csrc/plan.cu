// plan.cu -- balanced split-KV scheduler of the dense decode.
//
// The scheduler runs on the device (one CTA) so that turning seq_lens /
// query_start_loc into work needs no host synchronisation: the review of
// "[Attention][DCP] Support DCP with query length > 1 (MTP) with FA3" rejects
// a CPU sync for the DCP local token counts, and
// "vllm.v1.attention.backends.mla.flashattn_mla" (metadata builder,
// _schedule_decode / num_splits) plans the KV splits ahead of the kernel.
//
// Every request's rows (q_len * H, token-major) are cut into row groups of NR;
// each (request, row group) pair owns the 64-key tiles of the request's
// shard-local keys.  All pairs' tiles form one list of W work items which the
// G decode CTAs divide into equal contiguous ranges, so every CTA streams the
// same number of KV tiles whatever the length mix; a pair cut by range
// boundaries is computed in several KV chunks whose results are merged by
// LSE (the same merge as the DCP merge, over chunks) by the decode CTA that
// finishes the pair's last chunk.  Rows of requests without local keys get
// their final result (out 0, lse -inf) here.
#include "common.cuh"
#include "plan.h"

namespace mla {

namespace {

// Exclusive block-wide scan of one int per thread (blockDim.x == 1024).
__device__ long long block_exclusive_scan(long long v, long long* warp_sums, long long* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    long long w = warp_sums[lane];
    long long s = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      long long y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    warp_sums[lane] = s - w;
    if (lane == 31) *total = s;
  }
  __syncthreads();
  long long r = warp_sums[warp] + x - v;
  __syncthreads();
  return r;
}

struct ReqPlan {
  int q0, q_len, L, Lr, groups, nt;
  bool ok;
};

__device__ ReqPlan plan_request(const SchedArgs& a, int b) {
  ReqPlan p{};
  const int q0 = a.query_start_loc[b], q1 = a.query_start_loc[b + 1], L = a.seq_lens[b];
  p.ok = !(q1 - q0 < 0 || q1 - q0 > L || q0 < 0 || q1 > a.num_tokens);
  p.q0 = q0 < 0 ? 0 : q0;
  p.q_len = p.ok ? q1 - q0 : 0;
  p.L = L;
  p.Lr = local_len(L, a.dcp_world, a.dcp_rank);
  p.groups = (p.q_len * a.num_heads + a.rows_per_group - 1) / a.rows_per_group;
  p.nt = (p.Lr + kKeyTile - 1) / kKeyTile;
  return p;
}

}  // namespace

__global__ void __launch_bounds__(1024) schedule_kernel(SchedArgs a) {
  __shared__ long long warp_sums[32];
  __shared__ long long s_total;
  __shared__ int s_overflow;
  grid_dep_sync();
  WorkspaceHeader* hdr = a.hdr;
  const int H = a.num_heads, NR = a.rows_per_group;
  if (threadIdx.x == 0) {
    s_overflow = 0;
    hdr->status = 0;  // this call's checks start clean (no kernel of it has run yet)
    hdr->detail = 0;
  }
  for (int t = threadIdx.x; t < a.num_tokens; t += blockDim.x) a.tok2req[t] = -1;
  __syncthreads();

  // pass 1: pair and item prefix sums over requests
  long long pair_carry = 0, item_carry = 0;
  for (int base = 0; base < a.num_requests; base += blockDim.x) {
    const int b = base + threadIdx.x;
    ReqPlan p{};
    if (b < a.num_requests) p = plan_request(a, b);
    const long long pair_off = block_exclusive_scan(p.groups, warp_sums, &s_total) + pair_carry;
    const long long pair_tot = s_total;
    const long long vlen = p.nt > 0 ? (long long)p.nt + a.unit_penalty : 0;  // list items of one pair
    const long long item_off = block_exclusive_scan((long long)p.groups * vlen, warp_sums, &s_total) + item_carry;
    const long long item_tot = s_total;
    if (b < a.num_requests) {
      if (!p.ok) record_check(hdr, kCheckBadQueryLayout);
      ReqInfo ri{};
      ri.q0 = p.q0;
      ri.q_len = p.q_len;
      ri.seq_len = p.L;
      ri.local_len = p.Lr;
      ri.rows = p.q_len * H;
      ri.pair_base = (int)pair_off;
      a.req[b] = ri;
      if (pair_off + p.groups > a.max_pairs) {
        s_overflow = 1;
      } else {
        // provisional pair entries (split plan filled in pass 2)
        for (int g = 0; g < p.groups; ++g) {
          PairInfo pi{};
          pi.item0 = item_off + (long long)g * vlen + (p.nt > 0 ? a.unit_penalty : 0);
          pi.b = b;
          pi.row0 = g * NR;
          pi.nrows = min(NR, ri.rows - g * NR);
          pi.nt = p.nt;
          pi.nsplit = 1;
          pi.pbase = 0;
          pi.q0 = ri.q0;
          pi.q_len = ri.q_len;
          pi.seq_len = ri.seq_len;
          pi.local_len = ri.local_len;
          a.pairs[pair_off + g] = pi;
          a.pair_done[pair_off + g] = 0;
        }
      }
      if (p.nt == 0 && p.q_len > 0) {
        // no local key: the rows' final result (no decode unit covers them)
        for (int r = 0; r < ri.rows; ++r) {
          const int64_t grow = (int64_t)p.q0 * H + r;
          a.lse[grow] = -INFINITY;
          if (a.out_f32) {
            float4* o = reinterpret_cast<float4*>(static_cast<float*>(a.out) + grow * kNope);
            for (int k = 0; k < kNope / 4; ++k) o[k] = make_float4(0.f, 0.f, 0.f, 0.f);
          } else {
            uint4* o = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + grow * kNope);
            for (int k = 0; k < kNope / 8; ++k) o[k] = make_uint4(0, 0, 0, 0);
          }
        }
      }
      for (int i = 0; i < p.q_len; ++i) {
        const int t = p.q0 + i;
        a.tok2req[t] = b;
        if (a.row_counts) {
          const int P = p.L - p.q_len + i;
          a.row_counts[t] = min(visible_keys(P, a.dcp_world, a.dcp_rank), p.Lr);
        }
      }
    }
    pair_carry += pair_tot;
    item_carry += item_tot;
  }
  __syncthreads();
  // balance over min(grid, W) ranges so that no range is empty: then every
  // range boundary inside a pair starts a real chunk and the chunk index of
  // a unit is its owner minus the owner of the pair's first item
  const long long W = item_carry, G = (long long)a.grid < W ? (long long)a.grid : (W > 0 ? W : 1);

  // pass 2: chunks per pair (how many CTA ranges cut it) and partial slots
  long long part_carry = 0;
  for (int base = 0; base < a.num_requests; base += blockDim.x) {
    const int b = base + threadIdx.x;
    long long parts = 0;
    int pb = 0, groups = 0;
    if (b < a.num_requests && !s_overflow) {
      pb = a.req[b].pair_base;
      const ReqPlan p = plan_request(a, b);
      groups = p.groups;
      for (int g = 0; g < groups; ++g) {
        PairInfo& pi = a.pairs[pb + g];
        int ns = 1;
        if (pi.nt > 0 && W > 0) {
          ns = (int)(item_owner(pi.item0 + pi.nt - 1, W, G) - item_owner(pi.item0, W, G) + 1);
          // CTA c's range starts at item floor(c W / G): the CTAs whose range
          // starts inside the pair's list items [item0 - penalty, item0 + nt)
          // begin with this pair
          const long long v0 = pi.item0 - a.unit_penalty;
          const long long c_lo = (v0 * G + W - 1) / W, c_hi = ((pi.item0 + pi.nt) * G + W - 1) / W;
          for (long long c = c_lo; c < c_hi; ++c) a.cta_pair0[c] = pb + g;
        }
        pi.nsplit = ns;
        if (ns > 1) parts += (long long)ns * NR;
      }
    }
    long long part_off = block_exclusive_scan(parts, warp_sums, &s_total) + part_carry;
    const long long part_tot = s_total;
    if (b < a.num_requests && !s_overflow) {
      if (part_off + parts > a.max_partial_rows) {
        s_overflow = 1;
      } else {
        for (int g = 0; g < groups; ++g) {
          PairInfo& pi = a.pairs[pb + g];
          if (pi.nsplit > 1) {
            pi.pbase = (int)part_off;
            part_off += (long long)pi.nsplit * NR;
          }
        }
      }
    }
    part_carry += part_tot;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (s_overflow) record_check(hdr, kCheckTileOverflow);
    // on overflow (the host bounds make it impossible) no decode work runs
    hdr->num_pairs = s_overflow ? 0 : (int)pair_carry;
    hdr->total_items = s_overflow ? 0 : W;
  }
}

}  // namespace mla
