// common.cuh -- shared device/host definitions of the MLA-DCP CUDA library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mla_dcp.h"

namespace mla {

constexpr int kNope = MLA_KV_LORA_RANK;  // 512: width of kv_c and q_nope
constexpr int kRope = MLA_ROPE_DIM;      // 64: width of k_pe and q_pe
constexpr int kRow = MLA_KV_ROW;         // 576: one latent cache row
constexpr int kVHead = MLA_V_HEAD_DIM;   // 128: W_UV output width per head
constexpr int kKeyTile = 64;             // keys per pipeline tile of the decode kernels
constexpr int kMaxHeads = 128;

// Device status word codes (first failure wins).
enum DeviceCheck : int32_t {
  kCheckOk = 0,
  kCheckPageOutOfRange = 1,
  kCheckBadQueryLayout = 2,
  kCheckWaitTimeout = 3,
  kCheckTileOverflow = 4,
};

// Workspace header, at offset 0 of every decode workspace.
struct WorkspaceHeader {
  int32_t status;      // 0 or MLA_ERR_DEVICE_CHECK
  int32_t detail;      // DeviceCheck code of the first failure
  int32_t num_tiles;   // tiles written by the scheduler
  int32_t pad[61];     // header is 256 bytes
};
static_assert(sizeof(WorkspaceHeader) == 256, "header size");

// One unit of decode work: rows [row0, row0 + nrows) of request b against its
// local keys [key0, key1) (the KV chunk of split `split` of `nsplit`).
struct Tile {
  int32_t b;
  int32_t row0;     // first row (i * H + h) of the request handled
  int32_t key0;     // first local key of the chunk
  int32_t key1;     // one past the last local key of the chunk
  int32_t split;    // index of this chunk among the request's chunks
  int32_t nsplit;   // chunks of this request (1 => write final output)
  int32_t pbase;    // first partial slot of the request (nsplit > 1)
  int32_t group;    // row-group index (row0 / rows_per_group)
};

// Per-request facts derived on the device by the scheduler.
struct ReqInfo {
  int32_t q0;       // query_start_loc[b]
  int32_t q_len;
  int32_t seq_len;  // global
  int32_t local_len;
  int32_t nsplit;
  int32_t pbase;    // first partial slot (slot = pbase + split * rows + row)
  int32_t rows;     // q_len * H
  int32_t chunk;    // keys per split (multiple of kKeyTile)
};

__device__ __forceinline__ void record_check(WorkspaceHeader* hdr, int32_t code) {
  if (atomicCAS(&hdr->status, 0, (int32_t)MLA_ERR_DEVICE_CHECK) == 0) hdr->detail = code;
}

// Local length on shard r of D of a request of global length L: the number of
// p < L with p mod D == r.
__host__ __device__ __forceinline__ int32_t local_len(int32_t L, int32_t D, int32_t r) {
  return L > r ? (L - r - 1) / D + 1 : 0;
}

// Local keys visible to the query at global position P on shard r of D: the
// j with j*D + r <= P.
__host__ __device__ __forceinline__ int32_t visible_keys(int32_t P, int32_t D, int32_t r) {
  return P >= r ? (P - r) / D + 1 : 0;
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

}  // namespace mla
