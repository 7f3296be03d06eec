// decode_simt.cu -- CUDA-core (fp32 FMA) MLA decode kernels, dense and sparse.
//
// Same tiles, masks, online softmax and outputs as the tensor-core kernels;
// every product is an fp32 FMA on CUDA cores.  One CTA of 256 threads owns NR
// (token, head) rows and walks its keys in blocks of 32, gathering each key's
// 576-wide row through the block table.
#include "common.cuh"
#include "decode_args.h"
#include "decode_kernels.h"

namespace mla {

namespace {

constexpr int kThreads = 256;
constexpr int kKB = 32;          // keys per block
constexpr int kKW = kRow / 2 + 1;  // 289 32-bit words per smem key row (one pad word: conflict-free dot products)

template <int NR>
struct SimtSmem {
  float q[NR][kRow];
  uint32_t k[kKB][kKW];
  float p[NR][kKB + 1];
  float m[NR], l[NR], alpha[NR];
  int32_t kend[NR];
  int32_t slot[kKB];
};

template <int NR, bool SPARSE>
__global__ void __launch_bounds__(kThreads) decode_simt_kernel(DecodeArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SimtSmem<NR>& s = *reinterpret_cast<SimtSmem<NR>*>(smem_raw);
  const int tid = threadIdx.x;
  const int H = a.num_heads, D = a.dcp_world, r = a.dcp_rank;

  // ---- which rows / keys
  int b, row0, nrows, key0, key1, q0;
  int split = 0, nsplit = 1, pbase = 0, req_rows = 0;
  int q_len = 0, seq_len = 0;
  int t_sparse = 0;
  if constexpr (SPARSE) {
    t_sparse = blockIdx.x / a.groups_per_token;
    const int g = blockIdx.x % a.groups_per_token;
    if (t_sparse >= a.num_tokens) return;
    b = a.tok_req[t_sparse];
    row0 = g * NR;
    nrows = min(NR, H - row0);
    key0 = 0;
    key1 = a.list_count[t_sparse];
    q0 = t_sparse;
  } else {
    if ((int)blockIdx.x >= a.hdr->num_tiles) return;
    const Tile tile = a.tiles[blockIdx.x];
    const ReqInfo ri = a.req[tile.b];
    b = tile.b;
    row0 = tile.row0;
    nrows = min(NR, ri.rows - row0);
    key0 = tile.key0;
    key1 = tile.key1;
    q0 = ri.q0;
    split = tile.split;
    nsplit = tile.nsplit;
    pbase = tile.pbase;
    req_rows = ri.rows;
    q_len = ri.q_len;
    seq_len = ri.seq_len;
  }
  if (b < 0 || nrows <= 0) return;

  // global (token, head) row index of local row i: dense rows are i*H + h of
  // the request; sparse rows are the heads of one token
  auto grow = [&](int i) -> int64_t {
    if constexpr (SPARSE) return (int64_t)t_sparse * H + row0 + i;
    else return (int64_t)q0 * H + row0 + i;
  };

  // ---- Q rows to smem (fp32)
  for (int idx = tid; idx < NR * (kRow / 2); idx += kThreads) {
    const int i = idx / (kRow / 2), w = idx % (kRow / 2), d = 2 * w;
    float x0 = 0.f, x1 = 0.f;
    if (i < nrows) {
      const int64_t g = grow(i);
      const __nv_bfloat16* src = d < kNope ? a.q_nope + g * a.q_nope_stride + d : a.q_pe + g * a.q_pe_stride + (d - kNope);
      const uint32_t v = *reinterpret_cast<const uint32_t*>(src);
      x0 = bf16_lo(v);
      x1 = bf16_hi(v);
    }
    s.q[i][d] = x0;
    s.q[i][d + 1] = x1;
  }
  if (tid < NR) {
    s.m[tid] = -INFINITY;
    s.l[tid] = 0.f;
    int kend = 0;
    if (tid < nrows) {
      if constexpr (SPARSE) {
        kend = key1;
      } else {
        const int i = (row0 + tid) / H;  // query token index within the request
        const int P = seq_len - q_len + i;
        kend = min(visible_keys(P, D, r), key1);
      }
    }
    s.kend[tid] = kend;
  }

  constexpr int TPR = kThreads / NR;  // threads per row in the PV update
  constexpr int DPT = kNope / TPR;    // dims per thread
  const int my_row = tid / TPR;
  const int my_d0 = (tid % TPR) * DPT;
  float acc[DPT];
#pragma unroll
  for (int k = 0; k < DPT; ++k) acc[k] = 0.f;

  for (int kb = key0; kb < key1; kb += kKB) {
    __syncthreads();
    if (tid < kKB) {
      const int j = kb + tid;
      int slot = -1;
      if (j < key1) {
        int loc = j;
        if constexpr (SPARSE) loc = a.lists[(int64_t)t_sparse * a.list_stride + j];
        const int pidx = loc / a.page_size;
        const int page = pidx < a.bt_stride ? a.block_table[(int64_t)b * a.bt_stride + pidx] : -1;
        if (page < 0 || page >= a.num_blocks) {
          record_check(a.hdr, kCheckPageOutOfRange);
        } else {
          slot = page * a.page_size + loc % a.page_size;
        }
      }
      s.slot[tid] = slot;
    }
    __syncthreads();
    for (int idx = tid; idx < kKB * (kRow / 2); idx += kThreads) {
      const int k = idx / (kRow / 2), w = idx % (kRow / 2);
      const int slot = s.slot[k];
      s.k[k][w] = slot >= 0 ? reinterpret_cast<const uint32_t*>(a.kv + (int64_t)slot * kRow)[w] : 0u;
    }
    __syncthreads();
    // scores
    for (int idx = tid; idx < NR * kKB; idx += kThreads) {
      const int i = idx / kKB, k = idx % kKB;
      float sc = -INFINITY;
      if (i < nrows && kb + k < s.kend[i] && s.slot[k] >= 0) {
        float accd = 0.f;
#pragma unroll 8
        for (int w = 0; w < kRow / 2; ++w) {
          const uint32_t v = s.k[k][w];
          accd = fmaf(s.q[i][2 * w], bf16_lo(v), accd);
          accd = fmaf(s.q[i][2 * w + 1], bf16_hi(v), accd);
        }
        sc = accd * a.scale;
      }
      s.p[i][k] = sc;
    }
    __syncthreads();
    // online softmax, one thread per row
    if (tid < NR) {
      float mx = s.m[tid];
      for (int k = 0; k < kKB; ++k) mx = fmaxf(mx, s.p[tid][k]);
      const float mref = mx == -INFINITY ? 0.f : mx;
      const float alpha = __expf(s.m[tid] - mref);
      float sum = 0.f;
      for (int k = 0; k < kKB; ++k) {
        const float p = __expf(s.p[tid][k] - mref);
        s.p[tid][k] = p;
        sum += p;
      }
      s.l[tid] = s.l[tid] * alpha + sum;
      s.m[tid] = mx;
      s.alpha[tid] = alpha;
    }
    __syncthreads();
    // O update
    {
      const float alpha = s.alpha[my_row];
#pragma unroll
      for (int k = 0; k < DPT; ++k) acc[k] *= alpha;
      for (int k = 0; k < kKB; ++k) {
        const float p = s.p[my_row][k];
        if (p == 0.f) continue;
#pragma unroll
        for (int w = 0; w < DPT / 2; ++w) {
          const uint32_t v = s.k[k][my_d0 / 2 + w];
          acc[2 * w] = fmaf(p, bf16_lo(v), acc[2 * w]);
          acc[2 * w + 1] = fmaf(p, bf16_hi(v), acc[2 * w + 1]);
        }
      }
    }
  }
  __syncthreads();

  // ---- epilogue
  if (my_row >= nrows) return;
  const float l = s.l[my_row];
  const float m = s.m[my_row];
  const float inv = l > 0.f ? 1.f / l : 0.f;
  const float lse = (l > 0.f && m > -INFINITY) ? m + __logf(l) : -INFINITY;
  const bool partial = !SPARSE && nsplit > 1;
  if (partial) {
    const int64_t slot = (int64_t)pbase + (int64_t)split * req_rows + row0 + my_row;
    float* dst = a.part_o + slot * kNope + my_d0;
#pragma unroll
    for (int k = 0; k < DPT; k += 4)
      *reinterpret_cast<float4*>(dst + k) = make_float4(acc[k] * inv, acc[k + 1] * inv, acc[k + 2] * inv, acc[k + 3] * inv);
    if (tid % TPR == 0) a.part_lse[slot] = lse;
  } else {
    const int64_t g = grow(my_row);
    if (a.out_f32) {
      float* dst = static_cast<float*>(a.out) + g * kNope + my_d0;
#pragma unroll
      for (int k = 0; k < DPT; k += 4)
        *reinterpret_cast<float4*>(dst + k) = make_float4(acc[k] * inv, acc[k + 1] * inv, acc[k + 2] * inv, acc[k + 3] * inv);
    } else {
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out) + g * kNope + my_d0;
#pragma unroll
      for (int k = 0; k < DPT; k += 2)
        *reinterpret_cast<__nv_bfloat162*>(dst + k) = __floats2bfloat162_rn(acc[k] * inv, acc[k + 1] * inv);
    }
    if (tid % TPR == 0) a.lse[g] = lse;
  }
}

template <int NR, bool SPARSE>
cudaError_t launch_one(const DecodeArgs& a, int grid, cudaStream_t stream) {
  const size_t smem = sizeof(SimtSmem<NR>);
  cudaError_t e = cudaFuncSetAttribute(decode_simt_kernel<NR, SPARSE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  decode_simt_kernel<NR, SPARSE><<<grid, kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_simt(const DecodeArgs& a, int rows_per_group, bool sparse, int grid, cudaStream_t stream) {
  if (grid <= 0) return cudaSuccess;
  if (sparse) return rows_per_group == 16 ? launch_one<16, true>(a, grid, stream) : launch_one<32, true>(a, grid, stream);
  return rows_per_group == 16 ? launch_one<16, false>(a, grid, stream) : launch_one<32, false>(a, grid, stream);
}

}  // namespace mla
