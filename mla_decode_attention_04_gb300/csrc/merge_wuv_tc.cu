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
constexpr int kWChunk = 16384;            // W_UV[h] rows of one 64-dim chunk: 64 dims x 128 outputs
constexpr int kWBufs = 2;                 // W_UV chunk ring
constexpr int kBChunk = kNT * 128;        // merged rows of one 64-dim chunk: 32 tokens x 128 B
constexpr int kOffBHi = kWBufs * kWChunk;
constexpr int kOffBLo = kOffBHi + 8 * kBChunk;
constexpr int kOffShared = kOffBLo + 8 * kBChunk;

struct MergeShared {
  uint64_t w_full[kWBufs], w_empty[kWBufs], mma_done;
  uint32_t tmem_base;
  int32_t w_ok;  // every W_UV chunk landed and its MMAs were issued
  float wgt[kNT][kMaxShards];
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void load_w_chunk(const CUtensorMap* w_map, uint8_t* dst, int h, int c, uint64_t* bar) {
  mbar_arrive_expect_tx(bar, kWChunk);
  const uint64_t pol = policy_evict_normal();  // every CTA of head h reads it
  tma_load_3d(dst, w_map, 0, h * kNope + c * 64, 0, bar, pol);
  tma_load_3d(dst + 8192, w_map, 64, h * kNope + c * 64, 0, bar, pol);
}

// One CTA per head h and 32 tokens (two CTAs fit on an SM; heads vary
// fastest over the grid).  W_UV[h] streams
// through a 2-chunk TMA ring; its first two chunks are requested before the
// wait for the kernel that wrote the partials (W_UV is an input of the
// call, not of that kernel).  Each thread merges one 8-dim piece of one
// chunk for 8 of the tokens, all its partial loads in flight at once, and
// writes the merged values as bf16 hi + lo; one thread then issues the
// projection chunk by chunk as W_UV lands; four warps store the 128 x 32
// result.
__global__ void __launch_bounds__(kThreads, 2) merge_wuv_tc_kernel(const __grid_constant__ CUtensorMap w_map,
                                                                    MergeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* w_s = base;              // [2][2 atoms of 64 outputs][64 dims][128 B]
  uint8_t* b_hi = base + kOffBHi;   // [8 chunks][32 tokens][64 dims] K-major SW128
  uint8_t* b_lo = base + kOffBLo;
  MergeShared& sh = *reinterpret_cast<MergeShared*>(base + kOffShared);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // heads vary fastest over the grid, so the CTAs resident together read
  // different heads' W_UV (not one head's lines from 15 SMs at once)
  const int h = blockIdx.x, t0 = blockIdx.y * kNT;
  const int T = a.num_tokens, H = a.num_heads, D = a.dcp_world;

  if (warp == 0) {
    tmem_alloc(&sh.tmem_base, 32);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int b = 0; b < kWBufs; ++b) {
      mbar_init(&sh.w_full[b], 1);
      mbar_init(&sh.w_empty[b], 1);
    }
    mbar_init(&sh.mma_done, 1);
    fence_mbar_init();
    prefetch_tmap(&w_map);
    for (int b = 0; b < kWBufs; ++b) load_w_chunk(&w_map, w_s + b * kWChunk, h, b, &sh.w_full[b]);
  }
  grid_dep_sync();
  // merge weights.  One partial (the shard-fused route's merged rows): the
  // weight is 1 for a row with keys and its LSE passes through, one thread
  // per token.  Otherwise a warp per token, lanes over shards.
  if (D == 1) {
    if (tid < kNT) {
      const int t = t0 + tid;
      float l = -INFINITY;
      if (t < T) {
        const bool part = a.valid_counts ? a.valid_counts[t] > 0 : true;
        if (part) l = a.lses[(int64_t)t * H + h];
        if (!(l > -INFINITY)) l = -INFINITY;  // NaN from a non-participating shard never enters
        if (a.lse_out) a.lse_out[(int64_t)t * H + h] = l;
      }
      sh.wgt[tid][0] = l > -INFINITY ? 1.f : 0.f;
    }
  } else {
  for (int n = warp; n < kNT; n += kThreads / 32) {
    const int t = t0 + n;
    float m = -INFINITY;
    for (int r = lane; r < D; r += 32) {
      float l = -INFINITY;
      if (t < T) {
        const bool part = a.valid_counts ? a.valid_counts[(int64_t)r * T + t] > 0 : true;
        if (part) l = a.lses[((int64_t)r * T + t) * H + h];
        if (!(l > -INFINITY)) l = -INFINITY;  // NaN from a non-participating shard never enters
      }
      sh.wgt[n][r] = l;
      m = fmaxf(m, l);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float z = 0.f;
    for (int r = lane; r < D; r += 32) z += m > -INFINITY ? __expf(sh.wgt[n][r] - m) : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    const float L = m > -INFINITY ? m + __logf(z) : -INFINITY;
    for (int r = lane; r < D; r += 32) sh.wgt[n][r] = L > -INFINITY ? __expf(sh.wgt[n][r] - L) : 0.f;
    if (lane == 0 && a.lse_out && t < T) a.lse_out[(int64_t)t * H + h] = L;
  }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;

  // this thread's piece: dims c * 64 + 8 piece .. + 7 of tokens n0 + 4 i, i < 8
  const int c = (tid >> 3) & 7, piece = tid & 7, n0 = tid >> 6;
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[i][k] = 0.f;
  for (int r = 0; r < D; ++r) {
    float wr[8];
    int64_t prow[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int n = n0 + 4 * i, t = t0 + n;
      wr[i] = t < T ? sh.wgt[n][r] : 0.f;
      prow[i] = ((int64_t)r * T + (t < T ? t : 0)) * H + h;
    }
    if (a.partial_f32) {
      float4 x[8], y[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        x[i] = y[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (wr[i] != 0.f) {
          const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(a.partials) +
                                                            prow[i] * kNope + c * 64 + piece * 8);
          x[i] = p[0];
          y[i] = p[1];
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        acc[i][0] += wr[i] * x[i].x; acc[i][1] += wr[i] * x[i].y; acc[i][2] += wr[i] * x[i].z;
        acc[i][3] += wr[i] * x[i].w; acc[i][4] += wr[i] * y[i].x; acc[i][5] += wr[i] * y[i].y;
        acc[i][6] += wr[i] * y[i].z; acc[i][7] += wr[i] * y[i].w;
      }
    } else {
      uint4 x[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        x[i] = make_uint4(0u, 0u, 0u, 0u);
        if (wr[i] != 0.f)
          x[i] = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.partials) + prow[i] * kNope +
                                                 c * 64 + piece * 8);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        acc[i][0] += wr[i] * bf16_lo(x[i].x); acc[i][1] += wr[i] * bf16_hi(x[i].x);
        acc[i][2] += wr[i] * bf16_lo(x[i].y); acc[i][3] += wr[i] * bf16_hi(x[i].y);
        acc[i][4] += wr[i] * bf16_lo(x[i].z); acc[i][5] += wr[i] * bf16_hi(x[i].z);
        acc[i][6] += wr[i] * bf16_lo(x[i].w); acc[i][7] += wr[i] * bf16_hi(x[i].w);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int n = n0 + 4 * i;
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float a0 = acc[i][2 * k], a1 = acc[i][2 * k + 1];
      const float h0 = __bfloat162float(__float2bfloat16_rn(a0));
      const float h1 = __bfloat162float(__float2bfloat16_rn(a1));
      hi[k] = pack_bf16(h0, h1);
      lo[k] = pack_bf16(a0 - h0, a1 - h1);
    }
    const int off = c * kBChunk + (n >> 3) * 1024 + (n & 7) * 128 + ((piece ^ (n & 7)) << 4);
    *reinterpret_cast<uint4*>(b_hi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(b_lo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  if (tid == 0) {
    // Y^T [128 x 32] = W_UV[h]^T . O^T over 8 chunks of 64 dims (hi and lo
    // terms); chunk cc + 2 is requested once chunk cc's MMAs are done
    const uint32_t idesc = idesc_bf16_f32(128, kNT, 1, 0);
    const uint32_t bh = smem_u32(b_hi), bl = smem_u32(b_lo);
    bool ok = true;
    uint32_t armed = 0x3u;  // W buffers with a load in flight (landing on phase armed_ph[b])
    uint32_t armed_ph[kWBufs] = {0, 0};
    for (int cc = 0; cc < 8 && ok; ++cc) {
      const int b = cc & (kWBufs - 1);
      if (!mbar_wait(&sh.w_full[b], (cc >> 1) & 1)) {
        ok = false;
        break;
      }
      armed &= ~(1u << b);
      tc_fence_after();
      const uint32_t wa = smem_u32(w_s + b * kWChunk);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t ad = smem_desc_sw128(wa + kk * 2048, 8192, 1024);
        mma_ss(tmem, ad, smem_desc_sw128(bh + cc * kBChunk + kk * 32, 16, 1024), idesc, (cc | kk) != 0);
        mma_ss(tmem, ad, smem_desc_sw128(bl + cc * kBChunk + kk * 32, 16, 1024), idesc, 1);
      }
      mma_commit(&sh.w_empty[b]);
      if (cc + kWBufs < 8) {
        if (!mbar_wait(&sh.w_empty[b], (cc >> 1) & 1)) {
          ok = false;
          break;
        }
        load_w_chunk(&w_map, w_s + b * kWChunk, h, cc + kWBufs, &sh.w_full[b]);
        armed |= 1u << b;
        armed_ph[b] = ((cc + kWBufs) >> 1) & 1;
      }
    }
    mma_commit(&sh.mma_done);  // every MMA issued above (none: arrives at once)
    sh.w_ok = ok ? 1 : 0;
    // a give-up leaves copies in flight: they land before the CTA exits
    for (int b = 0; b < kWBufs; ++b)
      if ((armed >> b) & 1u) mbar_wait(&sh.w_full[b], armed_ph[b]);
  }
  __syncthreads();
  // epilogue: warps 0-3 read the 128 output dims (lanes) x 32 tokens (columns)
  if (warp < 4) {
    const bool done = mbar_wait(&sh.mma_done, 0) && sh.w_ok;
    tc_fence_after();
    uint32_t y[32];
    tmem_ld<32>(tmem + ((uint32_t)(warp * 32) << 16), y);
    tmem_wait_ld();
    const int v = warp * 32 + lane;
    for (int k = 0; k < kNT && done; ++k) {
      const int tt = t0 + k;
      if (tt >= T) break;
      const int64_t idx = ((int64_t)tt * H + h) * kVHead + v;
      const float val = __uint_as_float(y[k]);
      if (a.out_f32) static_cast<float*>(a.out)[idx] = val;
      else static_cast<__nv_bfloat16*>(a.out)[idx] = __float2bfloat16_rn(val);
    }
  }
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
  const size_t smem = 1024 + kOffShared + sizeof(MergeShared);
  cudaError_t e = cudaFuncSetAttribute(merge_wuv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.num_heads, (a.num_tokens + kNT - 1) / kNT);
  return launch_pdl(merge_wuv_tc_kernel, grid, dim3(kThreads), smem, stream, map, a);
}

}  // namespace mla
