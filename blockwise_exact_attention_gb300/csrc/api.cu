// C ABI of libbea: argument validation, tensor-map construction and kernel
// dispatch. Every check runs before any CUDA call, so a rejected request
// touches neither the device nor the stream.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "../../include/bea.h"
#include "abi_internal.h"
#include "common.cuh"
#include "launch_cache.cuh"
#include "status.cuh"

namespace bea {
namespace abi {

thread_local int g_last_launches = 0;

// Status word of each device the library runs on: kernels OR flags into it.
__device__ uint32_t g_status_word;

std::mutex g_mutex;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
bea::PerContext<uint32_t*> g_status_ptr;

int status_ptr_for_current_device(uint32_t** out) {
  const cudaError_t e = g_status_ptr.get(
      [](uint32_t** v) {
        void* p = nullptr;
        cudaError_t r = cudaGetSymbolAddress(&p, g_status_word);
        if (r == cudaSuccess && p == nullptr) r = cudaErrorInvalidSymbol;
        *v = static_cast<uint32_t*>(p);
        return r;
      },
      out);
  return e == cudaSuccess ? BEA_OK : BEA_ERR_CUDA;
}

// Pending abort injection (tile + 1, 0 = none), taken by the next main-kernel launch.
std::atomic<int> g_inject_abort{0};
int take_inject_abort() { return g_inject_abort.exchange(0); }

int get_encoder(PFN_cuTensorMapEncodeTiled_v12000* out) {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        fn == nullptr || q != cudaDriverEntryPointSuccess)
      return BEA_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  *out = g_encode;
  return BEA_OK;
}

using PFN_ctxGetCurrent = CUresult (*)(CUcontext*);
using PFN_ctxGetId = CUresult (*)(CUcontext, unsigned long long*);
std::once_flag g_ctx_fn_once;
PFN_ctxGetCurrent g_ctx_get_current = nullptr;
PFN_ctxGetId g_ctx_get_id = nullptr;

void load_ctx_fns() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      fn != nullptr && q == cudaDriverEntryPointSuccess)
    g_ctx_get_current = reinterpret_cast<PFN_ctxGetCurrent>(fn);
  fn = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      fn != nullptr && q == cudaDriverEntryPointSuccess)
    g_ctx_get_id = reinterpret_cast<PFN_ctxGetId>(fn);
}

int64_t esize(int32_t dtype) { return dtype == BEA_BF16 ? 2 : 4; }

bool valid_dtype(int32_t dt) { return dt == BEA_BF16 || dt == BEA_F32; }

// Element count, saturating (shapes are validated non-negative first).
int64_t numel(const bea_tensor* t) {
  int64_t n = 1;
  for (int i = 0; i < t->ndim; ++i) {
    if (t->shape[i] == 0) return 0;
    if (__builtin_mul_overflow(n, t->shape[i], &n)) n = INT64_MAX;
  }
  return n;
}

// Structural checks of one tensor: rank, dtype, non-negative shape/strides,
// contiguous last dim, and (when non-empty) a base pointer and outer strides
// aligned to `align` bytes: 16 for [n,l,h,d] tensors (TMA and vector
// accesses), 4 for [n,h,l] log-sum-exp tensors (scalar accesses).
int check_tensor(const bea_tensor* t, int ndim) {
  if (t == nullptr) return BEA_ERR_ARG;
  if (t->ndim != ndim) return BEA_ERR_SHAPE;
  if (!valid_dtype(t->dtype)) return BEA_ERR_DTYPE;
  for (int i = 0; i < ndim; ++i) {
    if (t->shape[i] < 0 || t->shape[i] > (int64_t(1) << 31) - 1) return BEA_ERR_SHAPE;
    if (t->stride[i] < 0) return BEA_ERR_ALIGN;
  }
  if (numel(t) == 0) return BEA_OK;
  if (t->data == nullptr) return BEA_ERR_ARG;
  const int64_t es = esize(t->dtype);
  const int64_t align = (ndim == 4) ? 16 : es;
  if (t->shape[ndim - 1] > 1 && t->stride[ndim - 1] != 1) return BEA_ERR_ALIGN;
  if (reinterpret_cast<uintptr_t>(t->data) % align != 0) return BEA_ERR_ALIGN;
  for (int i = 0; i < ndim - 1; ++i)
    if (t->shape[i] > 1 && (t->stride[i] * es) % align != 0) return BEA_ERR_ALIGN;
  return BEA_OK;
}

bool same_shape(const bea_tensor* a, const bea_tensor* b) {
  if (a->ndim != b->ndim) return false;
  for (int i = 0; i < a->ndim; ++i)
    if (a->shape[i] != b->shape[i]) return false;
  return true;
}

Seq4 seq4(const bea_tensor* t) { return Seq4{t->data, t->stride[0], t->stride[1], t->stride[2]}; }
Lse3 lse3(const bea_tensor* t) { return Lse3{static_cast<float*>(t->data), t->stride[0], t->stride[1]}; }

// Fold the caller's window (-1 = unbounded), the causal flag (right = 0) and
// the key position offset (key j sits at query position j + key_offset) into
// the kernels' signed band: key j visible to query i iff i - ewl <= j <= i + ewr.
int check_window(int is_causal, int wl, int wr, int64_t key_offset, int* ewl, int* ewr) {
  if (wl < -1 || wr < -1) return BEA_ERR_ARG;
  if (is_causal != 0 && is_causal != 1) return BEA_ERR_ARG;
  if (is_causal && wr > 0) return BEA_ERR_ARG;
  if (key_offset < -(int64_t)bea::kUnbounded || key_offset > (int64_t)bea::kUnbounded) return BEA_ERR_ARG;
  auto clamp = [](int64_t x) {
    return (int)std::max<int64_t>(-bea::kUnbounded, std::min<int64_t>(bea::kUnbounded, x));
  };
  const int right = is_causal ? 0 : wr;
  *ewl = (wl < 0) ? bea::kUnbounded : clamp((int64_t)wl + key_offset);
  *ewr = (right < 0) ? bea::kUnbounded : clamp((int64_t)right - key_offset);
  return BEA_OK;
}

// Shared validation of q, k, v (and the mask) for forward and backward.
// key_offset: the position of key 0 relative to query 0; nullptr = the
// bottom-right alignment lq - lk (0 when lq == lk).
int check_qkv(const bea_tensor* q, const bea_tensor* k, const bea_tensor* v, float scale, int is_causal, int wl,
              int wr, const int64_t* key_offset, AttnDims* a) {
  int rc;
  if ((rc = check_tensor(q, 4)) || (rc = check_tensor(k, 4)) || (rc = check_tensor(v, 4))) return rc;
  if (q->dtype != k->dtype || q->dtype != v->dtype) return BEA_ERR_DTYPE;
  if (!same_shape(k, v)) return BEA_ERR_SHAPE;
  if (k->shape[0] != q->shape[0] || k->shape[3] != q->shape[3]) return BEA_ERR_SHAPE;
  const int64_t h = q->shape[2], hkv = k->shape[2];
  if (hkv <= 0 || h % hkv != 0) return BEA_ERR_SHAPE;
  if (!std::isfinite(scale) || !(scale > 0.f)) return BEA_ERR_ARG;
  if (q->shape[1] >= bea::kUnbounded || k->shape[1] >= bea::kUnbounded) return BEA_ERR_SHAPE;
  const int64_t off = key_offset ? *key_offset : q->shape[1] - k->shape[1];
  int ewl, ewr;
  if ((rc = check_window(is_causal, wl, wr, off, &ewl, &ewr))) return rc;
  const int64_t d = q->shape[3];
  if (q->dtype == BEA_BF16) {
    if (d != 64 && d != 128) return BEA_ERR_UNSUPPORTED;
  } else {
    if (d < 4 || d > 128 || d % 4 != 0) return BEA_ERR_UNSUPPORTED;
  }
  if (q->shape[0] * h > (int64_t(1) << 31) - 1) return BEA_ERR_SHAPE;
  a->n = (int)q->shape[0];
  a->lq = (int)q->shape[1];
  a->lk = (int)k->shape[1];
  a->h = (int)h;
  a->hkv = (int)hkv;
  a->d = (int)d;
  a->wl = ewl;
  a->wr = ewr;
  a->scale = scale;
  return BEA_OK;
}

int check_lse(const bea_tensor* lse, const AttnDims& a) {
  int rc;
  if ((rc = check_tensor(lse, 3))) return rc;
  if (lse->dtype != BEA_F32) return BEA_ERR_DTYPE;
  if (lse->shape[0] != a.n || lse->shape[1] != a.h || lse->shape[2] != a.lq) return BEA_ERR_SHAPE;
  return BEA_OK;
}

// [n, l, h, d] tensor -> TMA descriptor with boxes of 128 rows x 128 bytes
// (box_cols elements of es bytes), 128-byte swizzled.
static int make_map4(const bea_tensor* t, CUtensorMapDataType dt, int64_t es, cuuint32_t box_cols,
                     CUtensorMap* map) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  int rc = get_encoder(&enc);
  if (rc) return rc;
  const int64_t d = t->shape[3], hh = t->shape[2], l = t->shape[1], n = t->shape[0];
  // A size-1 dimension never moves the address; give it a harmless stride.
  const cuuint64_t s_h = (hh > 1) ? t->stride[2] * es : d * es;
  const cuuint64_t s_l = (l > 1) ? t->stride[1] * es : s_h * hh;
  const cuuint64_t s_n = (n > 1) ? t->stride[0] * es : s_l * l;
  cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)hh, (cuuint64_t)l, (cuuint64_t)n};
  cuuint64_t strides[3] = {s_h, s_l, s_n};
  cuuint32_t box[4] = {box_cols, 1, 128, 1};
  cuuint32_t es1[4] = {1, 1, 1, 1};
  CUresult r = enc(map, dt, 4, t->data, dims, strides, box, es1, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? BEA_OK : BEA_ERR_CUDA;
}

// bf16 [n, l, h, d]: 64-column boxes (the layout the MMA descriptors expect; also the fused
// ring step's bf16 final copy)
int make_seq_map(const bea_tensor* t, CUtensorMap* map) { return make_map4(t, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 64, map); }

// dK / dV of the backward: bf16 64-column or fp32 32-column boxes
int make_grad_map(const bea_tensor* g, CUtensorMap* map) {
  return g->dtype == BEA_F32 ? make_acc_map(g, map) : make_seq_map(g, map);
}

// fp32 [n, l, h, d] (the fused ring step's accumulator): 32-column boxes
int make_acc_map(const bea_tensor* t, CUtensorMap* map) { return make_map4(t, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, 32, map); }

int finish(cudaError_t e, int launches) {
  if (e != cudaSuccess) return BEA_ERR_CUDA;
  g_last_launches = launches;
  return BEA_OK;
}

// Workspace layout of the backward: [dq_acc | D | lse2], each 256-byte aligned.
// Byte sizes saturate at SIZE_MAX instead of wrapping: a size no buffer can
// have, which check_workspace then rejects.
size_t mul_sat(size_t a, size_t b) {
  size_t r;
  return __builtin_mul_overflow(a, b, &r) ? SIZE_MAX : r;
}
size_t add_sat(size_t a, size_t b) {
  size_t r;
  return __builtin_add_overflow(a, b, &r) ? SIZE_MAX : r;
}

BwdWorkspace bwd_workspace_layout(int64_t n, int64_t lq, int64_t h, int64_t d) {
  auto up = [](size_t x) { return x > SIZE_MAX - 255 ? SIZE_MAX : (x + 255) / 256 * 256; };
  const size_t lq_pad = mul_sat((size_t)(lq / 128 + (lq % 128 != 0)), 128);
  const size_t rows = mul_sat(mul_sat((size_t)n, (size_t)h), lq_pad);
  BwdWorkspace w;
  w.dq_off = 0;
  w.d_off = up(mul_sat(mul_sat(rows, (size_t)d), 4));
  w.l_off = add_sat(w.d_off, up(mul_sat(rows, 4)));
  w.total = add_sat(w.l_off, up(mul_sat(rows, 4)));
  return w;
}

int check_workspace(const void* workspace, size_t workspace_bytes, const BwdWorkspace& w) {
  if (workspace == nullptr || reinterpret_cast<uintptr_t>(workspace) % 256 != 0 || workspace_bytes < w.total)
    return BEA_ERR_WORKSPACE;
  return BEA_OK;
}

// Workspace pointers of the bf16 backward stages.
void set_workspace(BwdParams* p, void* workspace, const BwdWorkspace& w) {
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p->dq_acc = reinterpret_cast<float*>(ws + w.dq_off);
  p->d_row = reinterpret_cast<float*>(ws + w.d_off);
  p->lse2 = reinterpret_cast<float*>(ws + w.l_off);
  p->lq_pad = (p->a.lq + 127) / 128 * 128;
}

// Every check of bea_flash_mha_bwd except the workspace's.
int check_bwd_args(const bea_tensor* dout, const bea_tensor* q, const bea_tensor* k, const bea_tensor* v,
                   const bea_tensor* out, const bea_tensor* lse, const bea_tensor* dq, const bea_tensor* dk,
                   const bea_tensor* dv, float softmax_scale, int is_causal, int window_left, int window_right,
                   int accumulate, AttnDims* a) {
  int rc;
  if ((rc = check_qkv(q, k, v, softmax_scale, is_causal, window_left, window_right, nullptr, a))) return rc;
  if ((rc = check_tensor(dout, 4)) || (rc = check_tensor(out, 4)) || (rc = check_tensor(dq, 4)) ||
      (rc = check_tensor(dk, 4)) || (rc = check_tensor(dv, 4)))
    return rc;
  if (!same_shape(dout, q) || !same_shape(out, q) || !same_shape(dq, q) || !same_shape(dk, k) ||
      !same_shape(dv, k))
    return BEA_ERR_SHAPE;
  if ((rc = check_lse(lse, *a))) return rc;
  if (accumulate != 0 && accumulate != 1) return BEA_ERR_ARG;
  if (dout->dtype != q->dtype) return BEA_ERR_DTYPE;
  if (out->dtype != q->dtype && out->dtype != BEA_F32) return BEA_ERR_DTYPE;
  const bool f32 = q->dtype == BEA_F32;
  for (const bea_tensor* g : {dq, dk, dv}) {
    if (accumulate && g->dtype != BEA_F32) return BEA_ERR_DTYPE;
    if (f32 && g->dtype != BEA_F32) return BEA_ERR_DTYPE;
  }
  if (f32 && out->dtype != BEA_F32) return BEA_ERR_DTYPE;
  return BEA_OK;
}

// Dims of a stage that sees only [n, lq, h, d] query-side tensors (bf16 path).
int query_side_dims(const bea_tensor* t, AttnDims* a) {
  const int64_t d = t->shape[3];
  if (d != 64 && d != 128) return BEA_ERR_UNSUPPORTED;
  if (t->shape[0] * t->shape[2] > (int64_t(1) << 31) - 1) return BEA_ERR_SHAPE;
  a->n = (int)t->shape[0];
  a->lq = a->lk = (int)t->shape[1];
  a->h = a->hkv = (int)t->shape[2];
  a->d = (int)d;
  a->wl = a->wr = -1;
  a->scale = 1.f;
  return BEA_OK;
}

}  // namespace abi

using namespace abi;

unsigned long long current_context_id() {
  std::call_once(g_ctx_fn_once, load_ctx_fns);
  if (g_ctx_get_current == nullptr || g_ctx_get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  unsigned long long id = 0;
  if (g_ctx_get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

int check_bwd_call(const bea_tensor* dout, const bea_tensor* q, const bea_tensor* k, const bea_tensor* v,
                   const bea_tensor* out, const bea_tensor* lse, const bea_tensor* dq, const bea_tensor* dk,
                   const bea_tensor* dv, float softmax_scale, int is_causal, int window_left, int window_right,
                   int accumulate, size_t* workspace_bytes) {
  AttnDims a;
  const int rc = check_bwd_args(dout, q, k, v, out, lse, dq, dk, dv, softmax_scale, is_causal, window_left,
                                window_right, accumulate, &a);
  if (rc == BEA_OK) *workspace_bytes = bwd_workspace_layout(a.n, a.lq, a.h, a.d).total;
  return rc;
}

cudaError_t device_sm_count(int* sms) {
  static PerContext<int> cache;
  return cache.get(
      [](int* v) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        return cudaDeviceGetAttribute(v, cudaDevAttrMultiProcessorCount, dev);
      },
      sms);
}

}  // namespace bea

using namespace bea::abi;
using bea::AttnDims;
using bea::Seq4;

extern "C" {

int bea_version(void) { return BEA_VERSION; }

int bea_last_launch_count(void) { return g_last_launches; }

const char* bea_status_string(int code) {
  switch (code) {
    case BEA_OK: return "ok";
    case BEA_ERR_ARG: return "invalid argument (null pointer, scale, window or flag)";
    case BEA_ERR_SHAPE: return "inconsistent tensor shapes";
    case BEA_ERR_DTYPE: return "dtype not allowed for this argument";
    case BEA_ERR_ALIGN: return "pointer or stride not 16-byte aligned, or last dimension not contiguous";
    case BEA_ERR_UNSUPPORTED: return "unsupported configuration (head dim or dtype combination)";
    case BEA_ERR_CUDA: return "CUDA runtime or driver call failed";
    case BEA_ERR_TIMEOUT: return "a kernel wait ran past its time limit";
    case BEA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    default: return "unknown status";
  }
}

int bea_flash_mha_fwd(const bea_tensor* q, const bea_tensor* k, const bea_tensor* v, const bea_tensor* out,
                      const bea_tensor* lse, float softmax_scale, int is_causal, int window_left, int window_right,
                      void* stream) {
  AttnDims a;
  int rc;
  if ((rc = check_qkv(q, k, v, softmax_scale, is_causal, window_left, window_right, nullptr, &a))) return rc;
  if ((rc = check_tensor(out, 4))) return rc;
  if (!same_shape(out, q)) return BEA_ERR_SHAPE;
  if ((rc = check_lse(lse, a))) return rc;
  if (q->dtype == BEA_F32 && out->dtype != BEA_F32) return BEA_ERR_DTYPE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int launches = 0;
  if (a.n == 0 || a.h == 0 || a.lq == 0) return finish(cudaSuccess, 0);
  if (q->dtype == BEA_F32) {
    bea::F32FwdParams p{a, seq4(q), seq4(k), seq4(v), seq4(out), lse3(lse)};
    return finish(bea::launch_fwd_f32(p, s, &launches), launches);
  }
  bea::FwdParams p;
  std::memset(&p, 0, sizeof(p));
  p.a = a;
  p.out = seq4(out);
  p.out_is_f32 = out->dtype == BEA_F32;
  p.lse = lse3(lse);
  p.merge = 0;
  if ((rc = status_ptr_for_current_device(&p.status))) return rc;
  p.inject_abort = take_inject_abort();
  CUtensorMap tq, tk, tv;
  std::memset(&tk, 0, sizeof(tk));
  std::memset(&tv, 0, sizeof(tv));
  if ((rc = make_seq_map(q, &tq))) return rc;
  if (a.lk > 0) {
    if ((rc = make_seq_map(k, &tk)) || (rc = make_seq_map(v, &tv))) return rc;
  }
  CUtensorMap tout;  // a bf16 output leaves through TMA stores
  if (!p.out_is_f32 && (rc = make_seq_map(out, &tout))) return rc;
  return finish(bea::launch_fwd_bf16(p, tq, tk, tv, nullptr, p.out_is_f32 ? nullptr : &tout, s, &launches), launches);
}

int bea_flash_mha_fwd_merge(const bea_tensor* q, const bea_tensor* k, const bea_tensor* v, const bea_tensor* out_acc,
                            const bea_tensor* lse_acc, const bea_tensor* out_final, float softmax_scale, int is_causal,
                            int window_left, int window_right, int64_t key_offset, void* stream) {
  AttnDims a;
  int rc;
  if ((rc = check_qkv(q, k, v, softmax_scale, is_causal, window_left, window_right, &key_offset, &a))) return rc;
  if ((rc = check_tensor(out_acc, 4))) return rc;
  if (!same_shape(out_acc, q)) return BEA_ERR_SHAPE;
  if (out_acc->dtype != BEA_F32) return BEA_ERR_DTYPE;
  if ((rc = check_lse(lse_acc, a))) return rc;
  if (out_final != nullptr) {
    if ((rc = check_tensor(out_final, 4))) return rc;
    if (!same_shape(out_final, q)) return BEA_ERR_SHAPE;
    if (out_final->dtype != BEA_BF16) return BEA_ERR_DTYPE;
  }
  if (q->dtype != BEA_BF16) return BEA_ERR_UNSUPPORTED;
  int launches = 0;
  if (a.n == 0 || a.h == 0 || a.lq == 0) return finish(cudaSuccess, 0);
  bea::FwdParams p;
  std::memset(&p, 0, sizeof(p));
  p.a = a;
  p.out = seq4(out_acc);
  p.out_is_f32 = 1;
  p.lse = lse3(lse_acc);
  p.merge = 1;
  p.fin = out_final ? seq4(out_final) : Seq4{nullptr, 0, 0, 0};
  p.fin_b0 = 0;
  p.fin_b1 = a.n;
  if ((rc = status_ptr_for_current_device(&p.status))) return rc;
  p.inject_abort = take_inject_abort();
  CUtensorMap tq, tk, tv;
  std::memset(&tk, 0, sizeof(tk));
  std::memset(&tv, 0, sizeof(tv));
  if ((rc = make_seq_map(q, &tq))) return rc;
  if (a.lk > 0) {
    if ((rc = make_seq_map(k, &tk)) || (rc = make_seq_map(v, &tv))) return rc;
  }
  CUtensorMap tacc, tfin;
  std::memset(&tfin, 0, sizeof(tfin));
  if ((rc = make_acc_map(out_acc, &tacc))) return rc;
  if (out_final && (rc = make_seq_map(out_final, &tfin))) return rc;
  return finish(bea::launch_fwd_bf16(p, tq, tk, tv, &tacc, out_final ? &tfin : nullptr,
                                     static_cast<cudaStream_t>(stream), &launches),
                launches);
}

size_t bea_flash_mha_bwd_workspace_size(int64_t n, int64_t lq, int64_t h, int64_t d) {
  if (n < 0 || lq < 0 || h < 0 || d < 0) return 0;
  return bwd_workspace_layout(n, lq, h, d).total;
}

int bea_flash_mha_bwd(const bea_tensor* dout, const bea_tensor* q, const bea_tensor* k, const bea_tensor* v,
                      const bea_tensor* out, const bea_tensor* lse, const bea_tensor* dq, const bea_tensor* dk,
                      const bea_tensor* dv, float softmax_scale, int is_causal, int window_left, int window_right,
                      int accumulate, void* workspace, size_t workspace_bytes, void* stream) {
  AttnDims a;
  int rc;
  if ((rc = check_bwd_args(dout, q, k, v, out, lse, dq, dk, dv, softmax_scale, is_causal, window_left, window_right,
                           accumulate, &a)))
    return rc;
  const bool f32 = q->dtype == BEA_F32;
  const BwdWorkspace w = bwd_workspace_layout(a.n, a.lq, a.h, a.d);
  if ((rc = check_workspace(workspace, workspace_bytes, w))) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int launches = 0;
  if (a.n == 0 || a.h == 0) return finish(cudaSuccess, 0);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (f32) {
    bea::F32BwdParams p{a,        seq4(dout), seq4(q),   seq4(k),
                        seq4(v),  seq4(out),  seq4(dq),  seq4(dk),
                        seq4(dv), lse3(lse),  reinterpret_cast<float*>(ws + w.d_off), accumulate};
    return finish(bea::launch_bwd_f32(p, s, &launches), launches);
  }
  bea::BwdParams p;
  std::memset(&p, 0, sizeof(p));
  p.a = a;
  p.dout = seq4(dout);
  p.out = seq4(out);
  p.dq = seq4(dq);
  p.dk = seq4(dk);
  p.dv = seq4(dv);
  p.out_is_f32 = out->dtype == BEA_F32;
  p.dq_is_f32 = dq->dtype == BEA_F32;
  p.dk_is_f32 = dk->dtype == BEA_F32;
  p.dv_is_f32 = dv->dtype == BEA_F32;
  p.lse = lse3(lse);
  p.accumulate = accumulate;
  set_workspace(&p, workspace, w);
  if ((rc = status_ptr_for_current_device(&p.status))) return rc;
  p.inject_abort = take_inject_abort();
  CUtensorMap tq, tk, tv, tdo, tdk, tdv;
  std::memset(&tq, 0, sizeof(tq));
  std::memset(&tk, 0, sizeof(tk));
  std::memset(&tv, 0, sizeof(tv));
  std::memset(&tdo, 0, sizeof(tdo));
  std::memset(&tdk, 0, sizeof(tdk));
  std::memset(&tdv, 0, sizeof(tdv));
  if (a.lq > 0 && a.lk > 0) {
    if ((rc = make_seq_map(q, &tq)) || (rc = make_seq_map(k, &tk)) || (rc = make_seq_map(v, &tv)) ||
        (rc = make_seq_map(dout, &tdo)))
      return rc;
  }
  if (a.lk > 0 && ((rc = make_grad_map(dk, &tdk)) || (rc = make_grad_map(dv, &tdv)))) return rc;
  return finish(bea::launch_bwd_bf16(p, tq, tk, tv, tdo, tdk, tdv, s, &launches), launches);
}

int bea_flash_mha_bwd_prepare(const bea_tensor* dout, const bea_tensor* out, const bea_tensor* lse,
                              void* workspace, size_t workspace_bytes, void* stream) {
  int rc;
  if ((rc = check_tensor(dout, 4)) || (rc = check_tensor(out, 4))) return rc;
  if (dout->dtype != BEA_BF16) return dout->dtype == BEA_F32 ? BEA_ERR_UNSUPPORTED : BEA_ERR_DTYPE;
  if (!same_shape(out, dout)) return BEA_ERR_SHAPE;
  if (out->dtype != BEA_BF16 && out->dtype != BEA_F32) return BEA_ERR_DTYPE;
  bea::BwdParams p;
  std::memset(&p, 0, sizeof(p));
  if ((rc = query_side_dims(dout, &p.a))) return rc;
  if ((rc = check_lse(lse, p.a))) return rc;
  const BwdWorkspace w = bwd_workspace_layout(p.a.n, p.a.lq, p.a.h, p.a.d);
  if ((rc = check_workspace(workspace, workspace_bytes, w))) return rc;
  p.dout = seq4(dout);
  p.out = seq4(out);
  p.out_is_f32 = out->dtype == BEA_F32;
  p.lse = lse3(lse);
  set_workspace(&p, workspace, w);
  int launches = 0;
  return finish(bea::launch_bwd_prepare(p, static_cast<cudaStream_t>(stream), &launches), launches);
}

int bea_flash_mha_bwd_kv_block(const bea_tensor* dout, const bea_tensor* q, const bea_tensor* k,
                               const bea_tensor* v, const bea_tensor* dk, const bea_tensor* dv,
                               float softmax_scale, int is_causal, int window_left, int window_right,
                               int64_t key_offset, int accumulate, void* workspace, size_t workspace_bytes,
                               void* stream) {
  AttnDims a;
  int rc;
  if ((rc = check_qkv(q, k, v, softmax_scale, is_causal, window_left, window_right, &key_offset, &a))) return rc;
  if (q->dtype != BEA_BF16) return BEA_ERR_UNSUPPORTED;
  if ((rc = check_tensor(dout, 4)) || (rc = check_tensor(dk, 4)) || (rc = check_tensor(dv, 4))) return rc;
  if (!same_shape(dout, q) || !same_shape(dk, k) || !same_shape(dv, k)) return BEA_ERR_SHAPE;
  if (dout->dtype != BEA_BF16) return BEA_ERR_DTYPE;
  if (accumulate != 0 && accumulate != 1) return BEA_ERR_ARG;
  for (const bea_tensor* g : {dk, dv}) {
    if (g->dtype != BEA_BF16 && g->dtype != BEA_F32) return BEA_ERR_DTYPE;
    if (accumulate && g->dtype != BEA_F32) return BEA_ERR_DTYPE;
  }
  const BwdWorkspace w = bwd_workspace_layout(a.n, a.lq, a.h, a.d);
  if ((rc = check_workspace(workspace, workspace_bytes, w))) return rc;
  int launches = 0;
  if (a.n == 0 || a.h == 0) return finish(cudaSuccess, 0);
  bea::BwdParams p;
  std::memset(&p, 0, sizeof(p));
  p.a = a;
  p.dk = seq4(dk);
  p.dv = seq4(dv);
  p.dk_is_f32 = dk->dtype == BEA_F32;
  p.dv_is_f32 = dv->dtype == BEA_F32;
  p.accumulate = accumulate;
  set_workspace(&p, workspace, w);
  if ((rc = status_ptr_for_current_device(&p.status))) return rc;
  p.inject_abort = take_inject_abort();
  CUtensorMap tq, tk, tv, tdo, tdk, tdv;
  std::memset(&tq, 0, sizeof(tq));
  std::memset(&tk, 0, sizeof(tk));
  std::memset(&tv, 0, sizeof(tv));
  std::memset(&tdo, 0, sizeof(tdo));
  std::memset(&tdk, 0, sizeof(tdk));
  std::memset(&tdv, 0, sizeof(tdv));
  if (a.lq > 0 && a.lk > 0) {
    if ((rc = make_seq_map(q, &tq)) || (rc = make_seq_map(k, &tk)) || (rc = make_seq_map(v, &tv)) ||
        (rc = make_seq_map(dout, &tdo)))
      return rc;
  }
  if (a.lk > 0 && ((rc = make_grad_map(dk, &tdk)) || (rc = make_grad_map(dv, &tdv)))) return rc;
  return finish(bea::launch_bwd_main(p, tq, tk, tv, tdo, tdk, tdv, static_cast<cudaStream_t>(stream), &launches),
                launches);
}

int bea_flash_mha_bwd_finish(const bea_tensor* dq, float softmax_scale, int accumulate, void* workspace,
                             size_t workspace_bytes, void* stream) {
  int rc;
  if ((rc = check_tensor(dq, 4))) return rc;
  if (!std::isfinite(softmax_scale) || !(softmax_scale > 0.f)) return BEA_ERR_ARG;
  if (accumulate != 0 && accumulate != 1) return BEA_ERR_ARG;
  if (dq->dtype != BEA_BF16 && dq->dtype != BEA_F32) return BEA_ERR_DTYPE;
  if (accumulate && dq->dtype != BEA_F32) return BEA_ERR_DTYPE;
  bea::BwdParams p;
  std::memset(&p, 0, sizeof(p));
  if ((rc = query_side_dims(dq, &p.a))) return rc;
  p.a.scale = softmax_scale;
  const BwdWorkspace w = bwd_workspace_layout(p.a.n, p.a.lq, p.a.h, p.a.d);
  if ((rc = check_workspace(workspace, workspace_bytes, w))) return rc;
  p.dq = seq4(dq);
  p.dq_is_f32 = dq->dtype == BEA_F32;
  p.accumulate = accumulate;
  set_workspace(&p, workspace, w);
  int launches = 0;
  return finish(bea::launch_bwd_finish(p, static_cast<cudaStream_t>(stream), &launches), launches);
}

int bea_ring_merge(const bea_tensor* out_acc, const bea_tensor* lse_acc, const bea_tensor* out_blk,
                   const bea_tensor* lse_blk, const bea_tensor* out_final, void* stream) {
  int rc;
  if ((rc = check_tensor(out_acc, 4)) || (rc = check_tensor(lse_acc, 3)) || (rc = check_tensor(out_blk, 4)) ||
      (rc = check_tensor(lse_blk, 3)))
    return rc;
  if (out_acc->dtype != BEA_F32 || lse_acc->dtype != BEA_F32 || lse_blk->dtype != BEA_F32) return BEA_ERR_DTYPE;
  if (!same_shape(out_acc, out_blk) || !same_shape(lse_acc, lse_blk)) return BEA_ERR_SHAPE;
  const int64_t n = out_acc->shape[0], l = out_acc->shape[1], h = out_acc->shape[2], d = out_acc->shape[3];
  if (lse_acc->shape[0] != n || lse_acc->shape[1] != h || lse_acc->shape[2] != l) return BEA_ERR_SHAPE;
  if (d != 16 && d != 32 && d != 64 && d != 128) return BEA_ERR_UNSUPPORTED;
  if (out_final != nullptr) {
    if ((rc = check_tensor(out_final, 4))) return rc;
    if (out_final->dtype != BEA_BF16) return BEA_ERR_DTYPE;
    if (!same_shape(out_final, out_acc)) return BEA_ERR_SHAPE;
  }
  bea::MergeParams p;
  p.n = (int)n;
  p.l = (int)l;
  p.h = (int)h;
  p.d = (int)d;
  p.acc = seq4(out_acc);
  p.lse_acc = lse3(lse_acc);
  p.blk = seq4(out_blk);
  p.blk_is_f32 = out_blk->dtype == BEA_F32;
  p.lse_blk = lse3(lse_blk);
  p.fin = out_final ? seq4(out_final) : Seq4{nullptr, 0, 0, 0};
  int launches = 0;
  return finish(bea::launch_ring_merge(p, static_cast<cudaStream_t>(stream), &launches), launches);
}

int bea_get_device_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return BEA_ERR_CUDA;
  uint32_t* dptr = nullptr;
  if (status_ptr_for_current_device(&dptr)) return BEA_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, dptr, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return BEA_ERR_CUDA;
  if (cudaMemset(dptr, 0, sizeof(word)) != cudaSuccess) return BEA_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return BEA_ERR_CUDA;
  if (word & bea::BEA_STATUS_TIMEOUT) return BEA_ERR_TIMEOUT;
  if (word & bea::BEA_STATUS_CONFIG) return BEA_ERR_UNSUPPORTED;
  return BEA_OK;
}

int bea_selftest_inject_abort(int tile) {
  if (tile < -1) return BEA_ERR_ARG;
  g_inject_abort.store(tile + 1);
  return BEA_OK;
}

int bea_selftest_wait_timeout(int limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 2000000) return BEA_ERR_ARG;
  uint32_t* dptr = nullptr;
  if (status_ptr_for_current_device(&dptr)) return BEA_ERR_CUDA;
  return finish(bea::launch_selftest_wait_timeout(dptr, (uint64_t)limit_us * 1000ull,
                                                  static_cast<cudaStream_t>(stream)),
                1);
}

}  // extern "C"
