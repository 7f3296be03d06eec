// merge_wuv_tc.cu -- DCP LSE merge fused with the W_UV projection on tcgen05.
//
// "[Attention] DCP sparse MLA output-merge optimizations", summary: the
// per-shard results are merged by LSE and projected through W_UV (512 -> 128
// per head); the projection is linear, so it is applied once to the merged
// row.  Per head h and a block of 32 tokens this is a dense contraction
//   Y^T [128 x 32] = W_UV[h]^T [128 x 512] . O^T [512 x 32]
// done as tcgen05.mma kind::f16 with M = 128 output dims, N = 32 tokens,
// K = 512 in 8 chunks of 64.  A = the W_UV chunk read MN-major straight from
// its row-major layout (TMA, 128-byte swizzle); B = the merged rows, kept in
// fp32 by the merge and handed to the MMA as two bf16 terms hi + lo (hi =
// bf16(o), lo = bf16(o - hi)), so the projection adds no bf16 rounding of o
// beyond ~2^-17.  The accumulator is 32 TMEM columns.
#include "common.cuh"
#include "decode_kernels.h"
#include "pdl_launch.h"
#include "tc_ptx.cuh"
#include "tma_host.h"

namespace mla {

namespace {

using namespace tc;

constexpr int kNT = 32;         // tokens per CTA (MMA N)
constexpr int kThreads = 256;
constexpr int kMaxShards = 64;

struct MergeShared {
  uint64_t w_full, mma_done;
  uint32_t tmem_base;
  float wgt[kNT][kMaxShards];
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__global__ void __launch_bounds__(kThreads) merge_wuv_tc_kernel(const __grid_constant__ CUtensorMap w_map,
                                                                 MergeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* w_s = base;                  // [2 atoms of 64 out][64 dims][128 B]  16 KB
  uint8_t* b_hi = base + 16384;         // [32 tokens][64 dims] K-major SW128    4 KB
  uint8_t* b_lo = base + 16384 + 4096;  //                                        4 KB
  MergeShared& sh = *reinterpret_cast<MergeShared*>(base + 16384 + 8192);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.y, t0 = blockIdx.x * kNT;
  const int T = a.num_tokens, H = a.num_heads, D = a.dcp_world;

  if (warp == 0) {
    tmem_alloc(&sh.tmem_base, 32);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&sh.w_full, 1);
    mbar_init(&sh.mma_done, 1);
    fence_mbar_init();
    prefetch_tmap(&w_map);
  }
  grid_dep_sync();
  // merge weights: warp per token, lanes over shards
  for (int n = warp; n < kNT; n += kThreads / 32) {
    const int t = t0 + n;
    for (int r0 = 0; r0 < D; r0 += 32) {
      const int r = r0 + lane;
      float l = -INFINITY;
      if (t < T && r < D) {
        const bool part = a.valid_counts ? a.valid_counts[(int64_t)r * T + t] > 0 : true;
        if (part) l = a.lses[((int64_t)r * T + t) * H + h];
        if (!(l > -INFINITY)) l = -INFINITY;  // NaN from a non-participating shard never enters
      }
      if (r < kMaxShards) sh.wgt[n][r] = l;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;
  for (int n = warp; n < kNT; n += kThreads / 32) {
    float m = -INFINITY;
    for (int r = lane; r < D; r += 32) m = fmaxf(m, sh.wgt[n][r]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float z = 0.f;
    for (int r = lane; r < D; r += 32) z += m > -INFINITY ? __expf(sh.wgt[n][r] - m) : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    const float L = m > -INFINITY ? m + __logf(z) : -INFINITY;
    __syncwarp();
    for (int r = lane; r < D; r += 32) sh.wgt[n][r] = L > -INFINITY ? __expf(sh.wgt[n][r] - L) : 0.f;
    if (lane == 0 && a.lse_out && t0 + n < T) a.lse_out[(int64_t)(t0 + n) * H + h] = L;
  }
  __syncthreads();

  const uint32_t idesc = idesc_bf16_f32(128, kNT, 1, 0);
  const int n = tid >> 3;        // token of this thread in the merge
  const int piece = tid & 7;     // 8 dims (16 bytes of bf16) of the 64-dim chunk
  const int t = t0 + n;
  bool ok = true;
  for (int c = 0; c < 8; ++c) {
    if (tid == 0) {
      // previous chunk's MMAs must be done before W / B buffers are reused
      if (c > 0 && !mbar_wait(&sh.mma_done, (c - 1) & 1)) ok = false;
      mbar_arrive_expect_tx(&sh.w_full, 16384);
      const uint64_t pol = policy_evict_first();
      tma_load_3d(w_s, &w_map, 0, h * kNope + c * 64, 0, &sh.w_full, pol);
      tma_load_3d(w_s + 8192, &w_map, 64, h * kNope + c * 64, 0, &sh.w_full, pol);
    }
    __syncthreads();  // buffers free (thread 0 waited for the previous MMAs)
    float acc[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] = 0.f;
    if (t < T) {
      for (int r = 0; r < D; ++r) {
        const float wr = sh.wgt[n][r];
        if (wr == 0.f) continue;
        const int64_t prow = ((int64_t)r * T + t) * H + h;
        if (a.partial_f32) {
          const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(a.partials) + prow * kNope +
                                                            c * 64 + piece * 8);
          const float4 x = p[0], y = p[1];
          acc[0] += wr * x.x; acc[1] += wr * x.y; acc[2] += wr * x.z; acc[3] += wr * x.w;
          acc[4] += wr * y.x; acc[5] += wr * y.y; acc[6] += wr * y.z; acc[7] += wr * y.w;
        } else {
          const uint4 x = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.partials) +
                                                          prow * kNope + c * 64 + piece * 8);
          acc[0] += wr * bf16_lo(x.x); acc[1] += wr * bf16_hi(x.x);
          acc[2] += wr * bf16_lo(x.y); acc[3] += wr * bf16_hi(x.y);
          acc[4] += wr * bf16_lo(x.z); acc[5] += wr * bf16_hi(x.z);
          acc[6] += wr * bf16_lo(x.w); acc[7] += wr * bf16_hi(x.w);
        }
      }
    }
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float a0 = acc[2 * k], a1 = acc[2 * k + 1];
      const float h0 = __bfloat162float(__float2bfloat16_rn(a0));
      const float h1 = __bfloat162float(__float2bfloat16_rn(a1));
      hi[k] = pack_bf16(h0, h1);
      lo[k] = pack_bf16(a0 - h0, a1 - h1);
    }
    const int off = (n >> 3) * 1024 + (n & 7) * 128 + ((piece ^ (n & 7)) << 4);
    *reinterpret_cast<uint4*>(b_hi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(b_lo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      if (!mbar_wait(&sh.w_full, c & 1)) ok = false;
      tc_fence_after();
      const uint32_t wa = smem_u32(w_s), bh = smem_u32(b_hi), bl = smem_u32(b_lo);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t ad = smem_desc_sw128(wa + kk * 2048, 8192, 1024);
        mma_ss(tmem, ad, smem_desc_sw128(bh + kk * 32, 16, 1024), idesc, (c | kk) != 0);
        mma_ss(tmem, ad, smem_desc_sw128(bl + kk * 32, 16, 1024), idesc, 1);
      }
      mma_commit(&sh.mma_done);
    }
  }
  // epilogue: warps 0-3 read the 128 output dims (lanes) x 32 tokens (columns)
  if (warp < 4) {
    if (!mbar_wait(&sh.mma_done, 7 & 1)) ok = false;
    tc_fence_after();
    uint32_t y[32];
    tmem_ld<32>(tmem + ((uint32_t)(warp * 32) << 16), y);
    tmem_wait_ld();
    const int v = warp * 32 + lane;
    for (int k = 0; k < kNT; ++k) {
      const int tt = t0 + k;
      if (tt >= T) break;
      const int64_t idx = ((int64_t)tt * H + h) * kVHead + v;
      const float val = __uint_as_float(y[k]);
      if (a.out_f32) static_cast<float*>(a.out)[idx] = val;
      else static_cast<__nv_bfloat16*>(a.out)[idx] = __float2bfloat16_rn(val);
    }
  }
  (void)ok;  // a give-up leaves this block's output unspecified; waits are bounded so the kernel returns
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 32);
}

// Tensor map over W_UV viewed as [H * 512 rows][128 columns] bf16, box of 64
// columns (128 bytes, 128-byte swizzle) x 64 rows (one 3-D map with a unit
// outer dimension, so the same TMA wrapper serves it).
bool make_wuv_tensor_map(CUtensorMap* map, const void* w, int64_t rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {128, (cuuint64_t)rows, 1};
  const cuuint64_t strides[2] = {256, (cuuint64_t)rows * 256};
  const cuuint32_t box[3] = {64, 64, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(w), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_merge_wuv_tc(const MergeArgs& a, cudaStream_t stream) {
  if (a.num_tokens <= 0) return cudaSuccess;
  CUtensorMap map;
  if (!make_wuv_tensor_map(&map, a.w_uv, (int64_t)a.num_heads * kNope)) return cudaErrorInvalidValue;
  const size_t smem = 1024 + 16384 + 8192 + sizeof(MergeShared);
  cudaError_t e = cudaFuncSetAttribute(merge_wuv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((a.num_tokens + kNT - 1) / kNT, a.num_heads);
  return launch_pdl(merge_wuv_tc_kernel, grid, dim3(kThreads), smem, stream, map, a);
}

}  // namespace mla
