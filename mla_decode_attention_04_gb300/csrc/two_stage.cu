// two_stage.cu -- the device-side inputs of the two-stage decomposition.
//
// "[Attention] add DCP support for FLASH_ATTN_MLA backend", review thread:
// instead of a custom DCP mask, a decode step with q_len > 1 can run in two
// stages -- the request's context keys with the causal mask off (every query
// row sees all of them), and the query's own q_len new keys with the causal
// mask on -- and merge the two results.  For request b with L keys and q_len
// queries, the context is positions [0, L - q_len) and the new keys are
// [L - q_len, L); query i (position L - q_len + i) sees new keys
// L - q_len .. L - q_len + i.  This kernel derives, on the device, the
// context length of every request (the first stage's sequence lengths) and
// every token's list of new-key positions (the second stage's key lists,
// served by the sparse decode), so the two-stage call needs no host copy of
// the lengths.
#include "common.cuh"
#include "decode_kernels.h"
#include "pdl_launch.h"

namespace mla {

namespace {

__global__ void __launch_bounds__(256) two_stage_prep_kernel(TwoStageArgs a) {
  // No early launch of the next kernel: the first stage's decode reads the
  // context lengths before it waits for its own prep kernel, so it may only
  // start once this kernel has completed.
  grid_dep_wait();
  const int nthreads = gridDim.x * blockDim.x, tid = blockIdx.x * blockDim.x + threadIdx.x;
  for (int b = tid; b < a.num_requests; b += nthreads) {
    const int q0 = a.query_start_loc[b], q1 = a.query_start_loc[b + 1], L = a.seq_lens[b];
    const int q_len = q1 - q0;
    // a malformed request (the second stage's checks record it) gets an
    // empty context here
    const bool ok = q_len >= 0 && q_len <= L && q0 >= 0 && q1 <= a.num_tokens;
    const int C = ok ? L - q_len : 0;
    a.ctx_lens[b] = C;
    if (!ok) continue;
    for (int i = 0; i < q_len; ++i) {
      const int64_t t = q0 + i;
      int32_t* list = a.new_keys + t * a.list_stride;
      for (int j = 0; j < a.list_stride; ++j) list[j] = j <= i ? C + j : -1;
      a.new_valid[t] = min(i + 1, a.list_stride);
    }
  }
}

// Folds the second stage's status word into the first stage's (the one the
// call's workspace exposes at offset 0): the first failure is kept.
__global__ void fold_status_kernel(WorkspaceHeader* main, const WorkspaceHeader* other) {
  grid_dep_sync();
  if (threadIdx.x == 0 && main->status == 0 && other->status != 0) {
    main->detail = other->detail;
    main->where = other->where;
    main->status = other->status;
  }
}

}  // namespace

cudaError_t launch_two_stage_prep(const TwoStageArgs& a, cudaStream_t stream) {
  int blocks = (a.num_requests + 255) / 256;
  if (blocks < 1) blocks = 1;
  if (blocks > 64) blocks = 64;
  return launch_pdl(two_stage_prep_kernel, dim3(blocks), dim3(256), 0, stream, a);
}

cudaError_t launch_fold_status(WorkspaceHeader* main, const WorkspaceHeader* other, cudaStream_t stream) {
  return launch_pdl(fold_status_kernel, dim3(1), dim3(32), 0, stream, main, other);
}

}  // namespace mla
