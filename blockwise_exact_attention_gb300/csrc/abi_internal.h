// Host-side helpers of the C ABI shared by its translation units (api.cu
// defines them; ring_host.cu drives the ring replay with them): argument
// validation, tensor-map construction, the backward workspace layout and the
// per-device status word.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/bea.h"
#include "common.cuh"

namespace bea {
namespace abi {

// Records the launch count of a successful call (bea_last_launch_count) and
// maps a CUDA error to BEA_ERR_CUDA.
int finish(cudaError_t e, int launches);

int status_ptr_for_current_device(uint32_t** out);
int take_inject_abort();

// Structural checks of one tensor (rank, dtype, shape, contiguous last dim,
// alignment: 16 bytes for [n,l,h,d] tensors, the element size otherwise).
int check_tensor(const bea_tensor* t, int ndim);
bool same_shape(const bea_tensor* a, const bea_tensor* b);
Seq4 seq4(const bea_tensor* t);
Lse3 lse3(const bea_tensor* t);
// q, k, v, the scale and the mask, folded into AttnDims; key_offset nullptr =
// the bottom-right alignment lq - lk.
int check_qkv(const bea_tensor* q, const bea_tensor* k, const bea_tensor* v, float scale, int is_causal, int wl,
              int wr, const int64_t* key_offset, AttnDims* a);
int check_lse(const bea_tensor* lse, const AttnDims& a);
// TMA descriptor over a [n, l, h, d] bf16 tensor: 64-column boxes of 128 rows, 128-byte swizzle.
int make_seq_map(const bea_tensor* t, CUtensorMap* map);
int make_acc_map(const bea_tensor* t, CUtensorMap* map);
int make_grad_map(const bea_tensor* g, CUtensorMap* map);

// Backward workspace: [dq_acc | D | lse2], each region [n, h, lq_pad(, d)] and 256-byte aligned.
struct BwdWorkspace {
  size_t dq_off, d_off, l_off, total;
};
BwdWorkspace bwd_workspace_layout(int64_t n, int64_t lq, int64_t h, int64_t d);
int check_workspace(const void* workspace, size_t workspace_bytes, const BwdWorkspace& w);
void set_workspace(BwdParams* p, void* workspace, const BwdWorkspace& w);

}  // namespace abi
}  // namespace bea
