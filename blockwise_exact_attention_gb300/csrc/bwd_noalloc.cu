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
// is looked up with cudaGetSymbolAddress the first time the entry point runs
// in a device's context, and cached for that context (a context created after
// cudaDeviceReset looks it up again).
#include <cstddef>

#include <cuda_runtime.h>

#include "../../include/bea.h"
#include "launch_cache.cuh"

namespace bea {
// Every check of bea_flash_mha_bwd except the workspace's (api.cu); on success
// *workspace_bytes is the workspace that call needs.
int check_bwd_call(const bea_tensor* dout, const bea_tensor* q, const bea_tensor* k, const bea_tensor* v,
                   const bea_tensor* out, const bea_tensor* lse, const bea_tensor* dq, const bea_tensor* dk,
                   const bea_tensor* dv, float softmax_scale, int is_causal, int window_left, int window_right,
                   int accumulate, size_t* workspace_bytes);
}  // namespace bea

namespace {

static __device__ __align__(256) unsigned char g_bwd_scratch[BEA_NOALLOC_BWD_SCRATCH_BYTES];

bea::PerContext<void*> g_scratch_addr;

// Device address of the current device's scratch array (looked up once per context).
int scratch_for_current_device(void** out) {
  const cudaError_t e = g_scratch_addr.get(
      [](void** v) {
        cudaError_t r = cudaGetSymbolAddress(v, g_bwd_scratch);
        if (r == cudaSuccess && *v == nullptr) r = cudaErrorInvalidSymbol;
        return r;
      },
      out);
  return e == cudaSuccess ? BEA_OK : BEA_ERR_CUDA;
}

}  // namespace

extern "C" int bea_flash_mha_bwd_noalloc(const bea_tensor* dout, const bea_tensor* q, const bea_tensor* k,
                                         const bea_tensor* v, const bea_tensor* out, const bea_tensor* lse,
                                         const bea_tensor* dq, const bea_tensor* dk, const bea_tensor* dv,
                                         float softmax_scale, int is_causal, int window_left, int window_right,
                                         int accumulate, void* stream) {
  // The arguments are checked exactly as bea_flash_mha_bwd checks them, so a
  // malformed call gets the same error code; only then is the size compared
  // with the array (sizes saturate instead of overflowing).
  size_t need = 0;
  int rc = bea::check_bwd_call(dout, q, k, v, out, lse, dq, dk, dv, softmax_scale, is_causal, window_left,
                               window_right, accumulate, &need);
  if (rc != BEA_OK) return rc;
  if (need > (size_t)BEA_NOALLOC_BWD_SCRATCH_BYTES) return BEA_ERR_WORKSPACE;  // problem too large for the array
  void* scratch = nullptr;
  if ((rc = scratch_for_current_device(&scratch)) != BEA_OK) return rc;
  // Same kernels as bea_flash_mha_bwd; the preprocess kernel rewrites every
  // part of the workspace the call reads (the dQ accumulator rows, D and the
  // scaled log-sum-exp of every padded row), so what an earlier call left in
  // the array does not matter.
  return bea_flash_mha_bwd(dout, q, k, v, out, lse, dq, dk, dv, softmax_scale, is_causal, window_left,
                           window_right, accumulate, scratch, (size_t)BEA_NOALLOC_BWD_SCRATCH_BYTES, stream);
}
