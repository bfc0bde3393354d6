// qsfm_forward_noalloc(): the forward pass without any device allocation.
//
// Some callers cannot call cudaMalloc: code that runs inside another
// framework's memory pool and may not allocate behind its back, plugin
// hosts that hand out only the input and output buffers, and serving loops
// that forbid allocation once they are running. For them this entry point
// takes the split-KV partial results from a fixed scratch array that the
// library reserves in device memory when it is loaded, instead of from a
// caller-provided workspace.
//
// The scratch is one file-scope __device__ array of QSFM_NOALLOC_SCRATCH_BYTES.
// Every GPU that loads the library holds it until the process exits. Its
// device address is looked up once per device, on the first call made with
// that device current; make that first call before any stream capture.
// Every call shares the array and it keeps the previous call's contents;
// nothing in it has to start at zero, because a call reads only the partial
// results it has written itself. Calls whose kernels overlap on the GPU
// (other streams, other threads) race on the array.
#include <cuda_runtime.h>

#include <mutex>

#include "qsfm.h"
#include "qsfm_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[QSFM_NOALLOC_SCRATCH_BYTES];

std::mutex g_lock;
void* g_scratch_addr[64] = {nullptr};

// Device address of g_noalloc_scratch on the current device (set-up on the
// first call per device).
qsfm_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return QSFM_ERR_CUDA;
  std::lock_guard<std::mutex> guard(g_lock);
  if (g_scratch_addr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
      return QSFM_ERR_CUDA;
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return QSFM_OK;
}

}  // namespace

extern "C" qsfm_status qsfm_forward_noalloc(const qsfm_params* p, void* stream) {
  size_t need = 0;
  qsfm_status st = qsfm_forward_workspace_size(p, &need);
  if (st != QSFM_OK) return st;
  if (need > QSFM_NOALLOC_SCRATCH_BYTES) return QSFM_ERR_WORKSPACE;
  void* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != QSFM_OK) return st;
  return qsfm_forward(p, scratch, QSFM_NOALLOC_SCRATCH_BYTES, stream);
}
