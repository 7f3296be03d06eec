// noalloc_decode.cu -- dense decode for callers that cannot allocate device memory.
//
// Some callers of this library cannot call cudaMalloc (or any allocating
// routine) at the point where they run a decode step: code running under a
// strict memory budget that was fixed at start-up, custom allocators that
// only hand out their own pool, or host frameworks that forbid allocation on
// their latency-critical path.  mla_dcp_decode needs a caller-supplied
// workspace; this file gives such callers a variant whose scratch lives in a
// fixed, file-scope device array instead.
//
// The array is MLA_STATIC_SCRATCH_BYTES (24 MiB) per device and lives as long
// as the library stays loaded: every GPU that loads the library holds it until
// the process exits.  All calls share it, so calls that may overlap on the GPU
// (different streams without ordering between them) race on it; calls issued
// on one stream, or otherwise ordered, are fine.  The array keeps the last
// call's contents; the decode clears what must start at zero (its status word)
// at the start of every call.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdio.h>

#include <mutex>

#include "common.cuh"

namespace {

static __device__ __align__(256) uint8_t g_static_scratch[MLA_STATIC_SCRATCH_BYTES];

// The array's device address, looked up once per CUDA context.  In host code
// the array's name is only a host-side stand-in, so the address comes from
// cudaGetSymbolAddress, with the device current.  A context is identified
// by its driver-assigned unique id, so a context created after a
// cudaDeviceReset (which unloads the module and frees the array) gets a
// fresh lookup instead of a dangling address.
constexpr int kMaxDevices = 64;
struct ScratchEntry {
  unsigned long long ctx_id;
  void* addr;
};
ScratchEntry g_scratch[kMaxDevices] = {};
std::mutex g_scratch_mu;

typedef CUresult (*PfnCtxGetCurrent)(CUcontext*);
typedef CUresult (*PfnCtxGetId)(CUcontext, unsigned long long*);

void* driver_entry(const char* name, unsigned version) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, version, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return p;
}

// Unique id of the current context (0 if there is none yet).
unsigned long long current_context_id() {
  static PfnCtxGetCurrent get_current = reinterpret_cast<PfnCtxGetCurrent>(driver_entry("cuCtxGetCurrent", 4000));
  static PfnCtxGetId get_id = reinterpret_cast<PfnCtxGetId>(driver_entry("cuCtxGetId", 12000));
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the array in the current context of the current device.
cudaError_t static_scratch_address(void** out, int* device) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  *device = dev;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  const unsigned long long id = current_context_id();
  if (id != 0 && g_scratch[dev].addr != nullptr && g_scratch[dev].ctx_id == id) {
    *out = g_scratch[dev].addr;
    return cudaSuccess;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_static_scratch);  // also makes the device's primary context current
  if (e != cudaSuccess) return e;
  g_scratch[dev].addr = p;
  g_scratch[dev].ctx_id = current_context_id();
  *out = p;
  return cudaSuccess;
}

}  // namespace

namespace mla {
int set_last_error(int code, const char* msg);
int check_dense_decode_args(const void* q_nope, int64_t q_nope_row_stride, const void* q_pe, int64_t q_pe_row_stride,
                            const void* kv_cache, int64_t num_blocks, int32_t page_size, int32_t kv_cache_dtype,
                            const int32_t* block_table, int32_t block_table_stride, const int32_t* seq_lens,
                            const int32_t* query_start_loc, int32_t num_requests, int32_t num_tokens,
                            int32_t num_heads, int32_t max_query_len, int32_t max_seq_len, int32_t dcp_world,
                            int32_t dcp_rank, float scale, void* out, int32_t out_dtype, float* lse,
                            int32_t num_splits);
}  // namespace mla

extern "C" int mla_dcp_decode_static_scratch(
    const void* q_nope, int64_t q_nope_row_stride, const void* q_pe, int64_t q_pe_row_stride, const void* kv_cache,
    int64_t num_blocks, int32_t page_size, int32_t kv_cache_dtype, const int32_t* block_table,
    int32_t block_table_stride, const int32_t* seq_lens, const int32_t* query_start_loc, int32_t num_requests,
    int32_t num_tokens, int32_t num_heads, int32_t max_query_len, int32_t max_seq_len, int32_t dcp_world,
    int32_t dcp_rank, float scale, void* out, int32_t out_dtype, float* lse, int32_t* row_counts,
    int32_t num_splits, void* stream) {
  // argument errors first, reported as such (not as a scratch shortfall)
  const int rc = mla::check_dense_decode_args(q_nope, q_nope_row_stride, q_pe, q_pe_row_stride, kv_cache, num_blocks,
                                              page_size, kv_cache_dtype, block_table, block_table_stride, seq_lens,
                                              query_start_loc, num_requests, num_tokens, num_heads, max_query_len,
                                              max_seq_len, dcp_world, dcp_rank, scale, out, out_dtype, lse,
                                              num_splits);
  if (rc != MLA_OK) return rc;
  const size_t need = mla_dcp_decode_workspace_size(num_requests, num_tokens, num_heads, max_query_len, max_seq_len,
                                                    dcp_world, num_splits);
  if (need > (size_t)MLA_STATIC_SCRATCH_BYTES) {
    char msg[256];
    snprintf(msg, sizeof msg,
             "this problem needs %zu bytes of decode scratch, more than the %zu-byte static array; use "
             "mla_dcp_decode with a caller workspace",
             need, (size_t)MLA_STATIC_SCRATCH_BYTES);
    return mla::set_last_error(MLA_ERR_WORKSPACE, msg);
  }
  void* scratch = nullptr;
  int dev = 0;
  const cudaError_t e = static_scratch_address(&scratch, &dev);
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof msg, "static scratch address on device %d: %s", dev, cudaGetErrorString(e));
    return mla::set_last_error(MLA_ERR_CUDA, msg);
  }
  return mla_dcp_decode(q_nope, q_nope_row_stride, q_pe, q_pe_row_stride, kv_cache, num_blocks, page_size,
                        kv_cache_dtype, block_table, block_table_stride, seq_lens, query_start_loc, num_requests,
                        num_tokens, num_heads, max_query_len, max_seq_len, dcp_world, dcp_rank, scale, out, out_dtype,
                        lse, row_counts, num_splits, scratch, (size_t)MLA_STATIC_SCRATCH_BYTES, stream);
}
