// Host-side interface between the C-ABI layer and the kernel translation
// units. Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include <utility>

#include "qsfm.h"

namespace qsfm {

// Partial-output workspace: per split piece slot, lse [64] fp32 then
// O [64][512] fp32. Two slots per planned CTA.
struct Workspace {
  float* lse;  // [slots][64]
  float* out;  // [slots][64][512]
  int slots;
};

size_t workspace_bytes(int num_ctas);
Workspace workspace_view(void* base, int num_ctas);

// Launches `kernel` so that it may start while the kernel before it on the
// stream is still running (programmatic stream serialization); the kernel
// calls grid_dependency_wait() before it reads anything its predecessor
// writes.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_after_predecessor(void (*kernel)(KArgs...), dim3 grid, dim3 block,
                                            size_t smem, cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

cudaError_t launch_plan(const qsfm_params& p, int num_tokens, int num_ctas, int split,
                        int32_t* metadata, int* fault, cudaStream_t s);
cudaError_t launch_attention(const qsfm_params& p, int num_tokens, int num_ctas,
                             const Workspace& ws, int* fault, cudaStream_t s);
cudaError_t launch_combine(const qsfm_params& p, int num_tokens, int num_ctas,
                           const Workspace& ws, int* fault, cudaStream_t s);
// Lightning indexer: score kernel then select kernel; the workspace holds
// num_tokens fp32 score rows.
size_t indexer_workspace_bytes(const qsfm_indexer_params& p, int num_tokens);
cudaError_t launch_indexer(const qsfm_indexer_params& p, int num_tokens, void* workspace, int* fault,
                           cudaStream_t s);
cudaError_t launch_bounded_wait(uint64_t timeout_ns, unsigned long long* elapsed, int* fault,
                                cudaStream_t s);
cudaError_t launch_debug_gather(const qsfm_params& p, const int32_t* tokens, int n,
                                int max_rows, uint8_t* rows_out, float* scales_out,
                                int32_t* row_ids_out, int32_t* counts_out, int* fault,
                                cudaStream_t s);

}  // namespace qsfm
