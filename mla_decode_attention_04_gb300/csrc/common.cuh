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
// A decode CTA that starts a (request, row group) unit pays for moving its Q
// into TMEM and for the previous unit's epilogue, about as long as streaming
// this many key tiles; the split-KV balance charges it to every unit.
constexpr int kUnitPenalty = 4;
constexpr int kMaxHeads = 128;

// Device status word codes (first failure wins).
enum DeviceCheck : int32_t {
  kCheckOk = 0,
  kCheckPageOutOfRange = 1,
  kCheckBadQueryLayout = 2,
  kCheckWaitTimeout = 3,
  kCheckBadSplitEntry = 4,  // a split-table entry out of range (internal consistency)
};

// Workspace header, at offset 0 of every decode workspace.
struct WorkspaceHeader {
  int32_t status;  // 0 or MLA_ERR_DEVICE_CHECK
  int32_t detail;  // DeviceCheck code of the first failure
  int32_t where;   // after a wait gave up (detail 3): the site of the first one (diagnostic)
  int32_t pad[61];  // header is 256 bytes
};
static_assert(sizeof(WorkspaceHeader) == 256, "header size");

__device__ __forceinline__ void record_check(WorkspaceHeader* hdr, int32_t code) {
  if (atomicCAS(&hdr->status, 0, (int32_t)MLA_ERR_DEVICE_CHECK) == 0) hdr->detail = code;
}

// A pipeline wait that gave up: the check, and the first give-up site.
__device__ __forceinline__ void record_wait_timeout(WorkspaceHeader* hdr, int32_t site) {
  record_check(hdr, kCheckWaitTimeout);
  atomicCAS(&hdr->where, 0, site);
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

// First partial row of chunk k of a split row group whose first chunk decode
// CTA cta0 holds: chunk 0 is cta0's last unit (its second slot), chunk k > 0
// is the first unit of CTA cta0 + k * stride (that CTA's first slot); the
// stride is 1, or the gang size when the CTAs run in gangs (the gang
// members hold the other row groups of the same requests).  NR rows each.
__host__ __device__ __forceinline__ int64_t chunk_slot(int cta0, int k, int NR, int stride) {
  return (int64_t)(k == 0 ? 2 * cta0 + 1 : 2 * (cta0 + k * stride)) * NR;
}

// Most DCP shards one call can cover (the shard-fused entry points).
constexpr int kMaxShards = 8;

// Element k of a per-shard kernel-parameter array, read with a static index.
template <typename T>
__device__ __forceinline__ T pick_shard(const T (&arr)[kMaxShards], int k) {
  switch (k) {
    case 0: return arr[0];
    case 1: return arr[1];
    case 2: return arr[2];
    case 3: return arr[3];
    case 4: return arr[4];
    case 5: return arr[5];
    case 6: return arr[6];
    default: return arr[7];
  }
}

// What the dense decode needs to know about request b, from seq_lens and
// query_start_loc alone (the prep kernel and every decode CTA derive it the
// same way).  A call covers nshard consecutive shards from rank shard0 (one
// shard, or all D when fused); nt is the request's key tiles over all of
// them, each shard's local keys padded to whole tiles.  A malformed query
// range (ok false) is treated as q_len 0.
struct ReqFacts {
  int32_t q0, q_len, seq_len, local_len, groups, nt;  // local_len: on shard0
  bool ok;
};

// The facts of request b from its raw inputs q0 = query_start_loc[b],
// q1 = query_start_loc[b + 1] and L = seq_lens[b].
// causal = false: the non-causal context pass of the two-stage
// decomposition, whose length L is the request's context only (q_len may
// exceed it).
__device__ __forceinline__ ReqFacts request_facts_of(int q0, int q1, int L, int num_tokens, int H, int D, int shard0,
                                                     int nshard, int NR, bool causal = true) {
  ReqFacts f;
  f.ok = !(q1 - q0 < 0 || (causal && q1 - q0 > L) || q0 < 0 || q1 > num_tokens);
  f.q0 = q0 < 0 ? 0 : q0;
  f.q_len = f.ok ? q1 - q0 : 0;
  f.seq_len = L;
  f.local_len = local_len(L, D, shard0);
  f.groups = (f.q_len * H + NR - 1) / NR;
  f.nt = 0;
  for (int k = 0; k < nshard; ++k) f.nt += (local_len(L, D, shard0 + k) + kKeyTile - 1) / kKeyTile;
  return f;
}

__device__ __forceinline__ ReqFacts request_facts(const int32_t* seq_lens, const int32_t* query_start_loc, int b,
                                                  int num_tokens, int H, int D, int shard0, int nshard, int NR,
                                                  bool causal = true) {
  return request_facts_of(query_start_loc[b], query_start_loc[b + 1], seq_lens[b], num_tokens, H, D, shard0, nshard,
                          NR, causal);
}

// Walks a request's key-tile sequence (shard k's local keys as whole tiles,
// k = 0 .. nshard-1 in turn) in increasing tile order: for tile t it names
// the shard index k within the call, the shard's tiles [t_begin, t_end) and
// the request's local length Lr on that shard.  A unit's tiles are visited
// in order, so moving on costs nothing until a shard boundary.
struct ShardCursor {
  int32_t k, t_begin, t_end, Lr;

  __device__ __forceinline__ void start(int L, int D, int shard0) {
    k = 0;
    t_begin = 0;
    Lr = local_len(L, D, shard0);
    t_end = (Lr + kKeyTile - 1) / kKeyTile;
  }
  // moves to the shard holding tile t (t >= t_begin); true if it moved
  __device__ __forceinline__ bool seek(int t, int L, int D, int shard0, int nshard) {
    bool moved = false;
    while (t >= t_end && k + 1 < nshard) {
      ++k;
      t_begin = t_end;
      Lr = local_len(L, D, shard0 + k);
      t_end += (Lr + kKeyTile - 1) / kKeyTile;
      moved = true;
    }
    return moved;
  }
};

// floor(t / W) for t >= 0, W > 0: a float estimate of the quotient corrected
// with exact integer products (64-bit division is a long dependent sequence).
__device__ __forceinline__ int64_t quot_floor(int64_t t, int64_t W) {
  int64_t q = (int64_t)((float)t * (1.0f / (float)W));
  while (q > 0 && q * W > t) --q;
  while ((q + 1) * W <= t) ++q;
  return q;
}

// CTA owning item i when W items are cut into G ranges
// [floor(c W / G), floor((c + 1) W / G)): ceil((i + 1) G / W) - 1.
__device__ __forceinline__ int64_t range_owner(int64_t i, int64_t W, int64_t G) {
  return quot_floor((i + 1) * G - 1, W);
}

// Programmatic dependent launch.  Every kernel of the library is launched
// so that it may start while the previous kernel in the stream finishes.
// grid_dep_launch lets this kernel's successor launch; grid_dep_wait blocks
// until the predecessor has completed and its writes are visible (both are
// no-ops when the kernel was launched without the attribute).
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_sync() {
  grid_dep_launch();
  grid_dep_wait();
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

}  // namespace mla
