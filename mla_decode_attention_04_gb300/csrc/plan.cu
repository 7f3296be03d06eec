// plan.cu -- the dense decode's prep kernel.
//
// The split-KV plan itself is derived inside the decode kernel: every decode
// CTA scans the requests' key-tile counts (seq_lens and query_start_loc only,
// so turning them into work needs no host synchronisation, as the review of
// "[Attention][DCP] Support DCP with query length > 1 (MTP) with FA3" asks)
// and takes its equal share of the flattened tile list, the way
// "vllm.v1.attention.backends.mla.flashattn_mla" (metadata builder,
// _schedule_decode / num_splits) plans KV splits ahead of the kernel.  What
// cannot be derived per CTA is done here, once per call: the status word is
// reset, malformed query ranges are
// recorded, per-token key counts are written, and rows of requests without
// local keys get their final result (o = 0, lse = -inf).
//
// The decode launches as soon as this kernel starts, plans and streams, and
// waits for this kernel's completion before its first global write (outputs,
// split partials and table, the status word).
#include "common.cuh"
#include "plan.h"

namespace mla {

__global__ void __launch_bounds__(256) prep_kernel(PrepArgs a) {
  // The decode may launch at once: it reads only its inputs before it waits
  // for this kernel.  This kernel writes nothing before the kernels ahead of
  // it in the stream (the previous call's readers of these outputs) finish.
  grid_dep_launch();
  grid_dep_wait();
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    a.hdr->status = 0;  // this call's checks start clean
    a.hdr->detail = 0;
    a.hdr->where = 0;
  }
  const int H = a.num_heads;
  const int nthreads = gridDim.x * blockDim.x, tid = blockIdx.x * blockDim.x + threadIdx.x;
  for (int b = tid; b < a.num_requests; b += nthreads) {
    const ReqFacts f = request_facts(a.seq_lens, a.query_start_loc, b, a.num_tokens, H, a.dcp_world, a.shard0,
                                     a.nshard, a.rows_per_group, !a.noncausal);
    if (!f.ok) record_check(a.hdr, kCheckBadQueryLayout);
    if (f.nt == 0 && f.q_len > 0) {
      // no local key: the rows' final result (no decode unit covers them)
      for (int r = 0; r < f.q_len * H; ++r) {
        const int64_t grow = (int64_t)f.q0 * H + r;
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
    if (a.row_counts) {  // one-shard calls only
      for (int i = 0; i < f.q_len; ++i) {
        const int P = a.noncausal ? f.seq_len - 1 : f.seq_len - f.q_len + i;
        a.row_counts[f.q0 + i] = min(visible_keys(P, a.dcp_world, a.shard0), f.local_len);
      }
    }
  }
}

}  // namespace mla
