// plan.cu -- split-KV scheduler and split combine of the dense decode.
//
// The scheduler runs on the device (one CTA) so that no host synchronisation
// is needed to turn seq_lens / query_start_loc into work: the backend review
// on "[Attention][DCP] Support DCP with query length > 1 (MTP) with FA3"
// rejects a host sync for the DCP local lengths, and
// "vllm.v1.attention.backends.mla.flashattn_mla" (metadata builder,
// _schedule_decode / num_splits) computes the split schedule ahead of the
// kernel.  Here every request's rows (q_len * H, token-major) are cut into
// row groups and its shard-local keys into equal chunks, so that the number
// of (request, row group, chunk) tiles is close to a target derived from the
// SM count; chunks of one request are merged by LSE afterwards.
#include "common.cuh"
#include "plan.h"

namespace mla {

namespace {

// Exclusive block-wide scan of one int per thread (blockDim.x == 1024).
__device__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = warp_sums[lane];
    int s = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    warp_sums[lane] = s - w;  // exclusive warp offsets
    if (lane == 31) *total = s;
  }
  __syncthreads();
  int r = warp_sums[warp] + x - v;
  __syncthreads();
  return r;
}

}  // namespace

__global__ void __launch_bounds__(1024) schedule_kernel(SchedArgs a) {
  __shared__ int warp_sums[32];
  __shared__ int s_total;
  __shared__ long long s_work;
  __shared__ int s_overflow;
  WorkspaceHeader* hdr = a.hdr;
  if (threadIdx.x == 0) s_overflow = 0;
  const int D = a.dcp_world, r = a.dcp_rank, H = a.num_heads, NR = a.rows_per_group;

  for (int t = threadIdx.x; t < a.num_tokens; t += blockDim.x) a.tok2req[t] = -1;
  __syncthreads();

  // pass 1: total work in (row group x key tile) units, for the chunk size
  long long work = 0;
  for (int b = threadIdx.x; b < a.num_requests; b += blockDim.x) {
    int q0 = a.query_start_loc[b], q1 = a.query_start_loc[b + 1], L = a.seq_lens[b];
    int q_len = q1 - q0;
    if (q_len < 0 || q_len > L || q0 < 0 || q1 > a.num_tokens) continue;
    int groups = (q_len * H + NR - 1) / NR;
    int nt = (local_len(L, D, r) + kKeyTile - 1) / kKeyTile;
    work += (long long)groups * (nt > 0 ? nt : 1);
  }
  if (threadIdx.x == 0) s_work = 0;
  __syncthreads();
  atomicAdd((unsigned long long*)&s_work, (unsigned long long)work);
  __syncthreads();
  long long total_work = s_work;
  int chunk_tiles = (int)((total_work + a.target_tiles - 1) / a.target_tiles);
  if (chunk_tiles < 1) chunk_tiles = 1;

  // pass 2: per-request split plan, prefix sums of tiles and partial rows
  int tile_carry = 0, part_carry = 0;
  for (int base = 0; base < a.num_requests; base += blockDim.x) {
    int b = base + threadIdx.x;
    ReqInfo ri = {};
    int ntiles = 0, nparts = 0, groups = 0;
    if (b < a.num_requests) {
      int q0 = a.query_start_loc[b], q1 = a.query_start_loc[b + 1], L = a.seq_lens[b];
      int q_len = q1 - q0;
      if (q_len < 0 || q_len > L || q0 < 0 || q1 > a.num_tokens) {
        record_check(hdr, kCheckBadQueryLayout);
        q_len = 0;
        q0 = q0 < 0 ? 0 : q0;
      }
      int Lr = local_len(L, D, r);
      int nt = (Lr + kKeyTile - 1) / kKeyTile;
      int ns = (nt + chunk_tiles - 1) / chunk_tiles;
      if (ns > a.max_splits) ns = a.max_splits;
      if (ns < 1) ns = 1;
      int chunk = ((nt + ns - 1) / ns) * kKeyTile;
      if (chunk < kKeyTile) chunk = kKeyTile;
      ns = Lr > 0 ? (Lr + chunk - 1) / chunk : 1;
      groups = (q_len * H + NR - 1) / NR;
      ri.q0 = q0;
      ri.q_len = q_len;
      ri.seq_len = L;
      ri.local_len = Lr;
      ri.nsplit = ns;
      ri.rows = q_len * H;
      ri.chunk = chunk;
      ntiles = groups * ns;
      nparts = ns > 1 ? ns * q_len * H : 0;
    }
    int tile_off = block_exclusive_scan(ntiles, warp_sums, &s_total) + tile_carry;
    int tile_tot = s_total;
    int part_off = block_exclusive_scan(nparts, warp_sums, &s_total) + part_carry;
    int part_tot = s_total;
    if (b < a.num_requests) {
      ri.pbase = part_off;
      bool fits = tile_off + ntiles <= a.max_tiles && part_off + nparts <= a.max_partial_rows;
      if (!fits) ri.nsplit = 1;  // nothing of this request is computed or combined
      a.req[b] = ri;
      if (!fits) {
        record_check(hdr, kCheckTileOverflow);
        s_overflow = 1;
      } else {
        int k = tile_off;
        for (int g = 0; g < groups; ++g)
          for (int s = 0; s < ri.nsplit; ++s) {
            Tile t;
            t.b = b;
            t.row0 = g * NR;
            t.key0 = s * ri.chunk;
            t.key1 = min((s + 1) * ri.chunk, ri.local_len);
            t.split = s;
            t.nsplit = ri.nsplit;
            t.pbase = ri.pbase;
            t.group = g;
            a.tiles[k++] = t;
          }
      }
      // per-token facts: owning request, visible key count
      for (int i = 0; i < ri.q_len; ++i) {
        int t = ri.q0 + i;
        a.tok2req[t] = b;
        if (a.row_counts) {
          int P = ri.seq_len - ri.q_len + i;
          a.row_counts[t] = min(visible_keys(P, D, r), ri.local_len);
        }
      }
    }
    tile_carry += tile_tot;
    part_carry += part_tot;
  }
  __syncthreads();
  // on overflow (the host bound makes it impossible) no tile runs at all
  if (threadIdx.x == 0) hdr->num_tiles = s_overflow ? 0 : tile_carry;
}

// Merge the per-chunk partial results of requests split into several KV
// chunks: the same LSE-weighted merge as the DCP merge, over chunks.  One warp
// per (token, head) row.
__global__ void __launch_bounds__(256) combine_kernel(CombineArgs a) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int H = a.num_heads;
  if (warp >= a.num_tokens * H) return;
  const int t = warp / H, h = warp % H;
  const int b = a.tok2req[t];
  if (b < 0) return;
  const ReqInfo ri = a.req[b];
  if (ri.nsplit <= 1) return;
  const int row = (t - ri.q0) * H + h;
  float m = -INFINITY;
  for (int s = 0; s < ri.nsplit; ++s) m = fmaxf(m, a.part_lse[ri.pbase + s * ri.rows + row]);
  float acc[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) acc[k] = 0.f;
  float lse = -INFINITY;
  if (m > -INFINITY) {
    float z = 0.f;
    for (int s = 0; s < ri.nsplit; ++s) z += __expf(a.part_lse[ri.pbase + s * ri.rows + row] - m);
    lse = m + __logf(z);
    for (int s = 0; s < ri.nsplit; ++s) {
      const int slot = ri.pbase + s * ri.rows + row;
      const float w = __expf(a.part_lse[slot] - lse);
      if (w == 0.f) continue;
      const float4* p = reinterpret_cast<const float4*>(a.part_o + (size_t)slot * kNope);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float4 v = p[k * 32 + lane];
        acc[4 * k + 0] += w * v.x;
        acc[4 * k + 1] += w * v.y;
        acc[4 * k + 2] += w * v.z;
        acc[4 * k + 3] += w * v.w;
      }
    }
  }
  const size_t orow = ((size_t)t * H + h) * kNope;
  if (a.out_f32) {
    float4* o = reinterpret_cast<float4*>(static_cast<float*>(a.out) + orow);
#pragma unroll
    for (int k = 0; k < 4; ++k) o[k * 32 + lane] = make_float4(acc[4 * k], acc[4 * k + 1], acc[4 * k + 2], acc[4 * k + 3]);
  } else {
    uint2* o = reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + orow);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      __nv_bfloat162 x = __floats2bfloat162_rn(acc[4 * k], acc[4 * k + 1]);
      __nv_bfloat162 y = __floats2bfloat162_rn(acc[4 * k + 2], acc[4 * k + 3]);
      o[k * 32 + lane] = make_uint2(*reinterpret_cast<uint32_t*>(&x), *reinterpret_cast<uint32_t*>(&y));
    }
  }
  if (lane == 0) a.lse[(size_t)t * H + h] = lse;
}

}  // namespace mla
