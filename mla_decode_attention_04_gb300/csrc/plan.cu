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

// Exclusive block-wide scans of two values per thread (blockDim.x == 1024)
// with one set of barriers; totals in tot[0..1].
__device__ void block_exclusive_scan2(long long v0, long long v1, longlong2* warp_sums, long long* tot,
                                      long long& r0, long long& r1) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long x0 = v0, x1 = v1;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y0 = __shfl_up_sync(0xffffffffu, x0, o), y1 = __shfl_up_sync(0xffffffffu, x1, o);
    if (lane >= o) x0 += y0, x1 += y1;
  }
  if (lane == 31) warp_sums[warp] = make_longlong2(x0, x1);
  __syncthreads();
  if (warp == 0) {
    const longlong2 w = warp_sums[lane];
    long long s0 = w.x, s1 = w.y;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y0 = __shfl_up_sync(0xffffffffu, s0, o), y1 = __shfl_up_sync(0xffffffffu, s1, o);
      if (lane >= o) s0 += y0, s1 += y1;
    }
    warp_sums[lane] = make_longlong2(s0 - w.x, s1 - w.y);
    if (lane == 31) tot[0] = s0, tot[1] = s1;
  }
  __syncthreads();
  const longlong2 base = warp_sums[warp];
  r0 = base.x + x0 - v0;
  r1 = base.y + x1 - v1;
  __syncthreads();
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
  __shared__ longlong2 warp_sums[32];
  __shared__ long long s_tot[2];
  __shared__ int s_overflow;
  grid_dep_sync();
  WorkspaceHeader* hdr = a.hdr;
  const int H = a.num_heads, NR = a.rows_per_group;
  const long long pen = a.unit_penalty;
  if (threadIdx.x == 0) {
    s_overflow = 0;
    hdr->status = 0;  // this call's checks start clean (no kernel of it has run yet)
    hdr->detail = 0;
  }
  for (int t = threadIdx.x; t < a.num_tokens; t += blockDim.x) a.tok2req[t] = -1;
  __syncthreads();
  // with at most one request per thread (every workload the decode targets)
  // pass 2 takes pass 1's values from registers instead of re-reading them
  const bool single = a.num_requests <= (int)blockDim.x;

  // pass 1: pair and item prefix sums over requests
  long long pair_carry = 0, item_carry = 0;
  ReqPlan p1{};
  long long pair_off1 = 0, item_off1 = 0;
  for (int base = 0; base < a.num_requests; base += blockDim.x) {
    const int b = base + threadIdx.x;
    ReqPlan p{};
    if (b < a.num_requests) p = plan_request(a, b);
    const long long vlen = p.nt > 0 ? (long long)p.nt + pen : 0;  // list items of one pair
    long long pair_off, item_off;
    block_exclusive_scan2(p.groups, (long long)p.groups * vlen, warp_sums, s_tot, pair_off, item_off);
    pair_off += pair_carry;
    item_off += item_carry;
    const long long pair_tot = s_tot[0], item_tot = s_tot[1];
    if (b < a.num_requests) {
      if (!p.ok) record_check(hdr, kCheckBadQueryLayout);
      ReqInfo ri{};
      ri.q0 = p.q0;
      ri.q_len = p.q_len;
      ri.seq_len = p.L;
      ri.local_len = p.Lr;
      ri.rows = p.q_len * H;
      ri.pair_base = (int)pair_off;
      ri.item_base = item_off;
      a.req[b] = ri;
      if (pair_off + p.groups > a.max_pairs) {
        s_overflow = 1;
      } else {
        for (int g = 0; g < p.groups; ++g) a.pair_done[pair_off + g] = 0;
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
    p1 = p;
    pair_off1 = pair_off;
    item_off1 = item_off;
    pair_carry += pair_tot;
    item_carry += item_tot;
  }
  __syncthreads();
  // balance over min(grid, W) ranges so that no range is empty: then every
  // range boundary inside a pair starts a real chunk and the chunk index of
  // a unit is its owner minus the owner of the pair's first item
  const long long W = item_carry, G = (long long)a.grid < W ? (long long)a.grid : (W > 0 ? W : 1);
  // Range ownership: CTA c's range is [floor(c W / G), floor((c + 1) W / G)).
  // Integer division is a long dependent sequence on the GPU and these run
  // several times per pair on few threads, so each quotient is a float
  // estimate (t * (1 / W)) corrected with exact integer products.
  const float rW = W > 0 ? 1.0f / (float)W : 0.f;
  auto quot_floor = [&](long long t) -> long long {  // floor(t / W), t >= 0
    long long q = (long long)((float)t * rW);
    while (q > 0 && q * W > t) --q;
    while ((q + 1) * W <= t) ++q;
    return q;
  };
  // largest c with c W < (i + 1) G, i.e. ceil((i + 1) G / W) - 1
  auto owner = [&](long long i) -> long long { return quot_floor((i + 1) * G - 1); };
  // smallest c with c W >= v G, i.e. ceil(v G / W)
  auto first_start_at_or_after = [&](long long v) -> long long { return v > 0 ? quot_floor(v * G - 1) + 1 : 0; };

  // pass 2: chunks per pair (how many CTA ranges cut it), partial slots, and
  // the final pair records
  long long part_carry = 0;
  for (int base = 0; base < a.num_requests; base += blockDim.x) {
    const int b = base + threadIdx.x;
    const bool mine = b < a.num_requests && !s_overflow;
    ReqPlan p{};
    long long pb = 0, ib = 0;
    if (mine) {
      if (single) {
        p = p1;
        pb = pair_off1;
        ib = item_off1;
      } else {
        p = plan_request(a, b);
        const ReqInfo ri = a.req[b];
        pb = ri.pair_base;
        ib = ri.item_base;
      }
    }
    const long long vlen = p.nt > 0 ? (long long)p.nt + pen : 0;
    const int rows = p.q_len * H;
    // chunks of pair g: CTA c's range starts at item floor(c W / G)
    auto nsplit_of = [&](long long item0) -> int {
      return (p.nt > 0 && W > 0) ? (int)(owner(item0 + p.nt - 1) - owner(item0) + 1) : 1;
    };
    long long parts = 0;
    if (mine) {
      for (int g = 0; g < p.groups; ++g) {
        const long long item0 = ib + g * vlen + (p.nt > 0 ? pen : 0);
        const int ns = nsplit_of(item0);
        if (ns > 1) parts += (long long)ns * NR;
        if (p.nt > 0 && W > 0) {
          // the CTAs whose range starts inside the pair's list items
          // [item0 - penalty, item0 + nt) begin with this pair
          const long long c_lo = first_start_at_or_after(item0 - pen), c_hi = first_start_at_or_after(item0 + p.nt);
          for (long long c = c_lo; c < c_hi; ++c) a.cta_pair0[c] = (int)(pb + g);
        }
      }
    }
    long long part_off, unused;
    block_exclusive_scan2(parts, 0, warp_sums, s_tot, part_off, unused);
    part_off += part_carry;
    const long long part_tot = s_tot[0];
    if (mine) {
      if (part_off + parts > a.max_partial_rows) {
        s_overflow = 1;
      } else {
        for (int g = 0; g < p.groups; ++g) {
          PairInfo pi{};
          pi.item0 = ib + g * vlen + (p.nt > 0 ? pen : 0);
          pi.b = b;
          pi.row0 = g * NR;
          pi.nrows = min(NR, rows - g * NR);
          pi.nt = p.nt;
          pi.cta0 = (p.nt > 0 && W > 0) ? (int)owner(pi.item0) : 0;
          pi.nsplit = (p.nt > 0 && W > 0) ? (int)(owner(pi.item0 + p.nt - 1) - pi.cta0 + 1) : 1;
          pi.pbase = 0;
          if (pi.nsplit > 1) {
            pi.pbase = (int)part_off;
            part_off += (long long)pi.nsplit * NR;
          }
          pi.q0 = p.q0;
          pi.q_len = p.q_len;
          pi.seq_len = p.L;
          pi.local_len = p.Lr;
          a.pairs[pb + g] = pi;
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
