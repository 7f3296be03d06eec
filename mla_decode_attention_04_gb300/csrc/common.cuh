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
// A decode CTA that starts a (request, row group) unit pays for loading its Q
// into TMEM and for the previous unit's epilogue, about as long as streaming
// this many key tiles; the split scheduler charges it to every unit.
constexpr int kUnitPenalty = 4;
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
  int32_t status;       // 0 or MLA_ERR_DEVICE_CHECK
  int32_t detail;       // DeviceCheck code of the first failure
  int32_t num_pairs;    // (request, row group) pairs written by the scheduler
  int32_t pad0;
  int64_t total_items;  // key tiles over all pairs (0: nothing to run)
  int32_t pad[58];      // header is 256 bytes
};
static_assert(sizeof(WorkspaceHeader) == 256, "header size");

// Per-request facts derived on the device by the scheduler.
struct ReqInfo {
  int32_t q0;         // query_start_loc[b]
  int32_t q_len;
  int32_t seq_len;    // global
  int32_t local_len;  // keys this shard holds
  int32_t rows;       // q_len * H (token-major: row = i * H + h)
  int32_t pair_base;  // first (request, row group) pair of the request
  int64_t item_base;  // the request's first item in the flattened work list
};

// One (request, row group): rows [row0, row0 + nrows) of request b and the
// nt 64-key tiles of its local keys, which are the work items
// [item0, item0 + nt) of the flattened list that the decode grid divides into
// equal contiguous ranges.  Each pair with keys is preceded in that list by
// kUnitPenalty items without work (the cost of starting a unit), so a range
// that starts units gets fewer key tiles.  A pair crossing range boundaries is computed in
// nsplit chunks whose partial results sit at slots pbase + split * NR + row
// and are merged by the decode CTA that finishes the pair's last chunk.  The
// request's facts are repeated here so that a decode CTA reads one record per
// unit.
struct __align__(16) PairInfo {
  int64_t item0;
  int32_t b;
  int32_t row0;
  int32_t nrows;
  int32_t nt;
  int32_t nsplit;
  int32_t pbase;
  int32_t q0;         // the request's query_start_loc
  int32_t q_len;
  int32_t seq_len;    // global
  int32_t local_len;  // keys this shard holds
  int32_t cta0;       // decode CTA that owns item0 (chunk index = CTA - cta0)
  int32_t pad[3];
};
static_assert(sizeof(PairInfo) == 64, "pair size");

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

// Programmatic dependent launch.  Every kernel of the library is launched
// so that it may start while the previous kernel in the stream finishes;
// it lets its own successor launch at once and waits, before its first
// global access, until the predecessor has completed and its writes are
// visible (a no-op when launched without the attribute).
__device__ __forceinline__ void grid_dep_sync() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

}  // namespace mla
