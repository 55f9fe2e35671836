// bea_flash_mha_bwd_noalloc: the backward for callers that cannot allocate
// device memory.
//
// bea_flash_mha_bwd needs a device workspace (the fp32 dQ accumulator plus
// two floats per query row) that the caller allocates. Some callers have no
// way to do that: code reached through a plain C function pointer from
// another language or plugin host that only hands over the tensors it owns,
// or a serving loop that must not call cudaMalloc (which can synchronise the
// device) once it is running. For them this entry point takes its workspace
// from a fixed-size array in the library's own device memory instead.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds BEA_NOALLOC_BWD_SCRATCH_BYTES of it until the process exits.
// Host code only sees a host-side stand-in for that symbol; its device address
// is looked up with cudaGetSymbolAddress once per device, the first time the
// entry point runs with that device current, and cached.
#include <cstddef>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/bea.h"

namespace {

static __device__ __align__(256) unsigned char g_bwd_scratch[BEA_NOALLOC_BWD_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of this device's scratch array (looked up on first use).
int scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return BEA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || p == nullptr) return BEA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return BEA_OK;
}

}  // namespace

extern "C" int bea_flash_mha_bwd_noalloc(const bea_tensor* dout, const bea_tensor* q, const bea_tensor* k,
                                         const bea_tensor* v, const bea_tensor* out, const bea_tensor* lse,
                                         const bea_tensor* dq, const bea_tensor* dk, const bea_tensor* dv,
                                         float softmax_scale, int is_causal, int window_left, int window_right,
                                         int accumulate, void* stream) {
  if (q == nullptr) return BEA_ERR_ARG;
  if (q->ndim != 4) return BEA_ERR_SHAPE;
  for (int i = 0; i < 4; ++i)
    if (q->shape[i] < 0) return BEA_ERR_SHAPE;
  const size_t need = bea_flash_mha_bwd_workspace_size(q->shape[0], q->shape[1], q->shape[2], q->shape[3]);
  if (need > (size_t)BEA_NOALLOC_BWD_SCRATCH_BYTES) return BEA_ERR_WORKSPACE;  // problem too large for the array
  void* scratch = nullptr;
  const int rc = scratch_for_current_device(&scratch);
  if (rc != BEA_OK) return rc;
  // Same validation and kernels as bea_flash_mha_bwd; the preprocess kernel
  // rewrites every part of the workspace the call reads, so what an earlier
  // call left in the array does not matter.
  return bea_flash_mha_bwd(dout, q, k, v, out, lse, dq, dk, dv, softmax_scale, is_causal, window_left,
                           window_right, accumulate, scratch, (size_t)BEA_NOALLOC_BWD_SCRATCH_BYTES, stream);
}
