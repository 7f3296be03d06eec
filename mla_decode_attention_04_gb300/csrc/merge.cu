// merge.cu -- DCP LSE-weighted merge, optionally fused with the W_UV projection.
//
// "[Attention] DCP sparse MLA output-merge optimizations", summary: the D
// shard results (o_r, lse_r) of one (token, head) are merged as
//   LSE = log sum_r exp(lse_r),  o = sum_r exp(lse_r - LSE) o_r
// over the shards that hold keys for the row (per-row valid counts; a shard
// row with count 0 is skipped without reading its partial), and the
// up-projection y = o . W_UV[h] commutes with the merge.
#include "common.cuh"
#include "decode_kernels.h"
#include "pdl_launch.h"

namespace mla {

namespace {

// Merge weights of one (token, head) row; returns false when no shard takes part.
__device__ __forceinline__ bool merge_weights(const MergeArgs& a, int t, int h, float* w, float* lse_row) {
  const int D = a.dcp_world, T = a.num_tokens, H = a.num_heads;
  float m = -INFINITY;
  for (int r = 0; r < D; ++r) {
    const bool part = a.valid_counts ? a.valid_counts[r * T + t] > 0 : true;
    const float l = part ? a.lses[((int64_t)r * T + t) * H + h] : -INFINITY;
    w[r] = l;
    if (part) m = fmaxf(m, l);
  }
  if (!(m > -INFINITY)) {
    *lse_row = -INFINITY;
    return false;
  }
  float z = 0.f;
  for (int r = 0; r < D; ++r) z += (w[r] > -INFINITY) ? __expf(w[r] - m) : 0.f;
  const float L = m + __logf(z);
  for (int r = 0; r < D; ++r) w[r] = (w[r] > -INFINITY) ? __expf(w[r] - L) : 0.f;
  *lse_row = L;
  return true;
}

constexpr int kMaxD = 64;

// 16 dims per lane: dims 128k + 4 lane + {0..3}, k < 4.
__device__ __forceinline__ void accumulate_row(const MergeArgs& a, int64_t prow, float w, float* acc) {
  if (a.partial_f32) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(a.partials) + prow * kNope);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float4 v = p[k * 32 + (threadIdx.x & 31)];
      acc[4 * k] += w * v.x;
      acc[4 * k + 1] += w * v.y;
      acc[4 * k + 2] += w * v.z;
      acc[4 * k + 3] += w * v.w;
    }
  } else {
    const uint2* p = reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(a.partials) + prow * kNope);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint2 v = p[k * 32 + (threadIdx.x & 31)];
      acc[4 * k] += w * bf16_lo(v.x);
      acc[4 * k + 1] += w * bf16_hi(v.x);
      acc[4 * k + 2] += w * bf16_lo(v.y);
      acc[4 * k + 3] += w * bf16_hi(v.y);
    }
  }
}

// One warp per (token, head) row, 512-wide output.
__global__ void __launch_bounds__(256) merge_rows_kernel(MergeArgs a) {
  grid_dep_sync();
  const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int T = a.num_tokens, H = a.num_heads;
  if (row >= T * H) return;
  const int t = row / H, h = row % H;
  float w[kMaxD];
  float lse;
  float acc[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) acc[k] = 0.f;
  if (merge_weights(a, t, h, w, &lse)) {
    for (int r = 0; r < a.dcp_world; ++r)
      if (w[r] != 0.f) accumulate_row(a, ((int64_t)r * T + t) * H + h, w[r], acc);
  }
  if (a.out_f32) {
    float4* o = reinterpret_cast<float4*>(static_cast<float*>(a.out) + (int64_t)row * kNope);
#pragma unroll
    for (int k = 0; k < 4; ++k) o[k * 32 + lane] = make_float4(acc[4 * k], acc[4 * k + 1], acc[4 * k + 2], acc[4 * k + 3]);
  } else {
    uint2* o = reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + (int64_t)row * kNope);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      __nv_bfloat162 x = __floats2bfloat162_rn(acc[4 * k], acc[4 * k + 1]);
      __nv_bfloat162 y = __floats2bfloat162_rn(acc[4 * k + 2], acc[4 * k + 3]);
      o[k * 32 + lane] = make_uint2(*reinterpret_cast<uint32_t*>(&x), *reinterpret_cast<uint32_t*>(&y));
    }
  }
  if (a.lse_out && lane == 0) a.lse_out[row] = lse;
}

}  // namespace

cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream) {
  if (a.num_tokens <= 0) return cudaSuccess;
  if (a.w_uv == nullptr) {
    const int64_t rows = (int64_t)a.num_tokens * a.num_heads;
    const int grid = (int)((rows + 7) / 8);
    return launch_pdl(merge_rows_kernel, dim3(grid), dim3(256), 0, stream, a);
  }
  return launch_merge_wuv_tc(a, stream);
}

}  // namespace mla
