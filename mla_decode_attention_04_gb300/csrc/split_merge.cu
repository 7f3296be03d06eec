// split_merge.cu -- LSE merge of the KV chunks of split row groups.
//
// The dense decode cuts a (request, row group) whose key tiles exceed one
// CTA's share into chunks on consecutive CTAs; each chunk leaves its rows
// normalised over its own keys, together with their LSE.  The rows' result
// is the LSE-weighted merge of the chunks, the same combination that joins
// the DCP shards ("[Attention] DCP sparse MLA output-merge optimizations",
// summary):  lse = log sum_k exp(lse_k),  o = sum_k exp(lse_k - lse) o_k.
// It runs as a kernel of its own right after the decode (programmatic
// launch: its blocks become resident early and wait on the device for the
// decode to complete), so no decode CTA waits for another one or carries a
// merge at its end, and the split plan can balance key tiles alone.
#include "common.cuh"
#include "plan.h"

namespace mla {

namespace {

// folds chunk rows (l, v) into the running (m, z, acc) of the same rows
__device__ __forceinline__ void fold_chunk(float& m, float& z, float4& acc, float l, const float4& v) {
  if (l == -INFINITY) return;  // a chunk in which the row sees no key adds nothing
  if (l > m) {
    const float r = m > -INFINITY ? __expf(m - l) : 0.f;
    acc = make_float4(r * acc.x + v.x, r * acc.y + v.y, r * acc.z + v.z, r * acc.w + v.w);
    z = r * z + 1.f;
    m = l;
  } else {
    const float w = __expf(l - m);
    acc = make_float4(acc.x + w * v.x, acc.y + w * v.y, acc.z + w * v.z, acc.w + w * v.w);
    z += w;
  }
}

}  // namespace

__global__ void __launch_bounds__(128) split_merge_kernel(SplitMergeArgs a) {
  grid_dep_launch();
  grid_dep_wait();  // the decode's partials and table are complete and visible
  constexpr int R = kSplitMergeRows;
  constexpr int kAhead = 2;  // chunks whose loads go out with the table entry's (a pair has 2, mostly)
  const int NR = a.rows_per_group;
  const int slices = NR / R;
  const int c = blockIdx.x / slices, n0 = (blockIdx.x % slices) * R;
  const int d0 = threadIdx.x * 4;  // latent dims [d0, d0 + 4) of each of the block's rows
  // The first kAhead chunks' rows are loaded before the entry is known (their
  // slots exist whenever c + k < grid; rows of chunks the entry does not have
  // are never used), so the entry and the data cost one memory latency.
  float l[kAhead][R];
  float4 v[kAhead][R];
#pragma unroll
  for (int k = 0; k < kAhead; ++k) {
    const bool exists = c + k * a.cta_stride < a.grid;
    const int64_t slot = chunk_slot(c, k, NR, a.cta_stride) + n0;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      l[k][r] = exists ? __ldcg(a.part_lse + slot + r) : -INFINITY;
      v[k][r] = exists ? __ldcg(reinterpret_cast<const float4*>(a.part_o + (slot + r) * kNope + d0))
                       : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  const int4 d = a.split_desc[c];
  const int nsplit = d.x, nrows = d.z;
  const int64_t g0 = d.y;
  if (nsplit < 2 || n0 >= nrows) return;  // no split row group starts at CTA c (or no rows here)
  if ((int64_t)c + (int64_t)(nsplit - 1) * a.cta_stride >= a.grid || nrows > NR || g0 < 0 ||
      g0 + nrows > a.num_rows) {
    if (threadIdx.x == 0 && n0 == 0) record_check(a.hdr, kCheckBadSplitEntry);
    return;
  }
  float m[R], z[R];
  float4 acc[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    m[r] = -INFINITY;
    z[r] = 0.f;
    acc[r] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int k = 0; k < kAhead; ++k)
#pragma unroll
    for (int r = 0; r < R; ++r)
      if (k < nsplit && n0 + r < nrows) fold_chunk(m[r], z[r], acc[r], l[k][r], v[k][r]);
  // longer splits: the rest, kAhead chunks per pass (all loads of a pass in flight)
#pragma unroll 1
  for (int sp = kAhead; sp < nsplit; sp += kAhead) {
#pragma unroll
    for (int k = 0; k < kAhead; ++k) {
      const bool use = sp + k < nsplit;
      const int64_t slot = chunk_slot(c, sp + k, NR, a.cta_stride) + n0;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        l[k][r] = use && n0 + r < nrows ? __ldcg(a.part_lse + slot + r) : -INFINITY;
        v[k][r] = use && n0 + r < nrows ? __ldcg(reinterpret_cast<const float4*>(a.part_o + (slot + r) * kNope + d0))
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int k = 0; k < kAhead; ++k)
#pragma unroll
      for (int r = 0; r < R; ++r) fold_chunk(m[r], z[r], acc[r], l[k][r], v[k][r]);
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (n0 + r >= nrows) break;
    const int64_t g = g0 + n0 + r;
    const float inv = z[r] > 0.f ? 1.f / z[r] : 0.f;
    const float4 o = make_float4(acc[r].x * inv, acc[r].y * inv, acc[r].z * inv, acc[r].w * inv);
    if (a.out_f32) {
      *reinterpret_cast<float4*>(static_cast<float*>(a.out) + g * kNope + d0) = o;
    } else {
      const __nv_bfloat162 x = __floats2bfloat162_rn(o.x, o.y);
      const __nv_bfloat162 y = __floats2bfloat162_rn(o.z, o.w);
      *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + g * kNope + d0) =
          make_uint2(*reinterpret_cast<const uint32_t*>(&x), *reinterpret_cast<const uint32_t*>(&y));
    }
    if (threadIdx.x == 0) a.lse[g] = z[r] > 0.f ? m[r] + __logf(z[r]) : -INFINITY;
  }
}

}  // namespace mla
