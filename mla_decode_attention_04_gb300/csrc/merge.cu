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

constexpr int kMaxD = 64;
constexpr int kRowsPerBlock = 8;  // one warp per (token, head) row

// Merge weights of row (t, h) into w[0..D) (shared memory of this row's
// warp): lane r covers shards r, r + 32; returns the row's LSE (-inf when
// no shard takes part: every weight is then 0).
__device__ __forceinline__ float merge_weights(const MergeArgs& a, int t, int h, float* w) {
  const int D = a.dcp_world, T = a.num_tokens, H = a.num_heads;
  const int lane = threadIdx.x & 31;
  float m = -INFINITY;
  for (int r = lane; r < D; r += 32) {
    const bool part = a.valid_counts ? a.valid_counts[(int64_t)r * T + t] > 0 : true;
    float l = part ? a.lses[((int64_t)r * T + t) * H + h] : -INFINITY;
    if (!(l > -INFINITY)) l = -INFINITY;  // NaN from a non-participating shard never enters
    w[r] = l;
    m = fmaxf(m, l);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float z = 0.f;
  for (int r = lane; r < D; r += 32) z += (m > -INFINITY) ? __expf(w[r] - m) : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  const float L = m > -INFINITY ? m + __logf(z) : -INFINITY;
  for (int r = lane; r < D; r += 32) w[r] = (L > -INFINITY) ? __expf(w[r] - L) : 0.f;
  __syncwarp();
  return L;
}

// 16 dims per lane: dims 128k + 4 lane + {0..3}, k < 4; two shards' loads
// in flight at a time.
__device__ __forceinline__ void accumulate_rows(const MergeArgs& a, int t, int h, const float* w, float* acc) {
  const int D = a.dcp_world, T = a.num_tokens, H = a.num_heads;
  const int lane = threadIdx.x & 31;
  for (int r0 = 0; r0 < D; r0 += 2) {
    float wr[2];
    int64_t prow[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int r = r0 + i;
      wr[i] = r < D ? w[r] : 0.f;
      prow[i] = ((int64_t)(r < D ? r : 0) * T + t) * H + h;
    }
    if (a.partial_f32) {
      float4 v[2][4];
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int k = 0; k < 4; ++k)
          v[i][k] = wr[i] != 0.f ? reinterpret_cast<const float4*>(static_cast<const float*>(a.partials) +
                                                                   prow[i] * kNope)[k * 32 + lane]
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          acc[4 * k] += wr[i] * v[i][k].x;
          acc[4 * k + 1] += wr[i] * v[i][k].y;
          acc[4 * k + 2] += wr[i] * v[i][k].z;
          acc[4 * k + 3] += wr[i] * v[i][k].w;
        }
    } else {
      uint2 v[2][4];
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int k = 0; k < 4; ++k)
          v[i][k] = wr[i] != 0.f ? reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(a.partials) +
                                                                  prow[i] * kNope)[k * 32 + lane]
                                 : make_uint2(0u, 0u);
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          acc[4 * k] += wr[i] * bf16_lo(v[i][k].x);
          acc[4 * k + 1] += wr[i] * bf16_hi(v[i][k].x);
          acc[4 * k + 2] += wr[i] * bf16_lo(v[i][k].y);
          acc[4 * k + 3] += wr[i] * bf16_hi(v[i][k].y);
        }
    }
  }
}

// One warp per (token, head) row, 512-wide output.
__global__ void __launch_bounds__(32 * kRowsPerBlock) merge_rows_kernel(MergeArgs a) {
  __shared__ float s_w[kRowsPerBlock][kMaxD];
  grid_dep_sync();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kRowsPerBlock + warp;
  const int T = a.num_tokens, H = a.num_heads;
  if (row >= (int64_t)T * H) return;
  const int t = (int)(row / H), h = (int)(row % H);
  float* w = s_w[warp];
  const float lse = merge_weights(a, t, h, w);
  float acc[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) acc[k] = 0.f;
  if (lse > -INFINITY) accumulate_rows(a, t, h, w, acc);
  if (a.out_f32) {
    float4* o = reinterpret_cast<float4*>(static_cast<float*>(a.out) + row * kNope);
#pragma unroll
    for (int k = 0; k < 4; ++k) o[k * 32 + lane] = make_float4(acc[4 * k], acc[4 * k + 1], acc[4 * k + 2], acc[4 * k + 3]);
  } else {
    uint2* o = reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + row * kNope);
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
    const int grid = (int)((rows + kRowsPerBlock - 1) / kRowsPerBlock);
    return launch_pdl(merge_rows_kernel, dim3(grid), dim3(32 * kRowsPerBlock), 0, stream, a);
  }
  return launch_merge_wuv_tc(a, stream);
}

}  // namespace mla
