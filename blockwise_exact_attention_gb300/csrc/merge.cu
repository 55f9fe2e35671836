// Log-sum-exp merge of a block result into a running (out, lse) accumulator.
//
// The fold of flash_attn_jax flash_sharding.py, section "Ring Forward":
//   mx = max(La, Lb), mn = min(La, Lb), L = log1p(exp(mn - mx)) + mx,
//   O = Oa exp(La - L) + Ob exp(Lb - L).
// A row whose two log-sum-exps are both -inf is left as it is (the formula
// would produce NaN there; the pages never reach that case because the first
// ring step is the diagonal block).
//
// HBM-bound elementwise kernel. Rows are enumerated (b, head, i) with the
// sequence index fastest, so that the lse reads of a block are contiguous and
// each row's d values are one contiguous, 16-byte-vectorised run. One group
// of d/4 threads owns a row; each thread moves 4 elements.
#include <cuda_bf16.h>

#include "common.cuh"

namespace bea {
namespace {

constexpr int kMergeThreads = 256;

template <bool kBlkF32, bool kFinal>
__global__ void __launch_bounds__(kMergeThreads) ring_merge_kernel(MergeParams p) {
  const int tpr = p.d >> 2;                        // threads per row (divides 32 or equals 32)
  const int rows_per_block = kMergeThreads / tpr;
  const int64_t nrows = (int64_t)p.n * p.h * p.l;
  const int sub = threadIdx.x / tpr;
  const int c = (threadIdx.x % tpr) * 4;
  // lanes of one row group share a trip count, so they can sync among themselves
  const unsigned lane0 = (threadIdx.x & 31u) / tpr * tpr;
  const unsigned group_mask = (tpr >= 32) ? 0xffffffffu : (((1u << tpr) - 1u) << lane0);
  for (int64_t r = (int64_t)blockIdx.x * rows_per_block + sub; r < nrows;
       r += (int64_t)gridDim.x * rows_per_block) {
    const int i = (int)(r % p.l);
    const int64_t bh = r / p.l;
    const int hh = (int)(bh % p.h);
    const int b = (int)(bh / p.h);
    float* la_ptr = p.lse_acc.ptr + b * p.lse_acc.sn + hh * p.lse_acc.sh + i;
    const float la = *la_ptr;
    const float lb = p.lse_blk.ptr[b * p.lse_blk.sn + hh * p.lse_blk.sh + i];
    __syncwarp(group_mask);  // every lane has read La before lane c == 0 rewrites it
    float* acc = reinterpret_cast<float*>(p.acc.ptr) + b * p.acc.sn + (int64_t)i * p.acc.sl + hh * p.acc.sh + c;
    const float mx = fmaxf(la, lb);
    float4 o = *reinterpret_cast<const float4*>(acc);
    if (mx != -INFINITY) {
      const float mn = fminf(la, lb);
      const float L = mx + log1pf(expf(mn - mx));
      const float wa = expf(la - L);
      const float wb = expf(lb - L);
      float4 ob;
      if constexpr (kBlkF32) {
        const float* src = reinterpret_cast<const float*>(p.blk.ptr) + b * p.blk.sn + (int64_t)i * p.blk.sl +
                           hh * p.blk.sh + c;
        ob = *reinterpret_cast<const float4*>(src);
      } else {
        const __nv_bfloat16* src = reinterpret_cast<const __nv_bfloat16*>(p.blk.ptr) + b * p.blk.sn +
                                   (int64_t)i * p.blk.sl + hh * p.blk.sh + c;
        const uint2 raw = *reinterpret_cast<const uint2*>(src);
        const float2 flo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
        const float2 fhi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
        ob = make_float4(flo.x, flo.y, fhi.x, fhi.y);
      }
      o.x = o.x * wa + ob.x * wb;
      o.y = o.y * wa + ob.y * wb;
      o.z = o.z * wa + ob.z * wb;
      o.w = o.w * wa + ob.w * wb;
      *reinterpret_cast<float4*>(acc) = o;
      if (c == 0) *la_ptr = L;
    }
    if constexpr (kFinal) {
      __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.fin.ptr) + b * p.fin.sn + (int64_t)i * p.fin.sl +
                           hh * p.fin.sh + c;
      const __nv_bfloat162 lo = __floats2bfloat162_rn(o.x, o.y);
      const __nv_bfloat162 hi = __floats2bfloat162_rn(o.z, o.w);
      uint2 raw;
      raw.x = *reinterpret_cast<const uint32_t*>(&lo);
      raw.y = *reinterpret_cast<const uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(dst) = raw;
    }
  }
}

}  // namespace

cudaError_t launch_ring_merge(const MergeParams& p, cudaStream_t s, int* nlaunch) {
  const int64_t nrows = (int64_t)p.n * p.h * p.l;
  if (nrows == 0) return cudaSuccess;
  const int rows_per_block = kMergeThreads / (p.d >> 2);
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t blocks = (nrows + rows_per_block - 1) / rows_per_block;
  const int64_t cap = (int64_t)sms * 8;  // 8 resident blocks of 256 threads per SM
  if (blocks > cap) blocks = cap;
  const bool f32 = p.blk_is_f32 != 0, fin = p.fin.ptr != nullptr;
  if (f32 && fin) ring_merge_kernel<true, true><<<(unsigned)blocks, kMergeThreads, 0, s>>>(p);
  else if (f32) ring_merge_kernel<true, false><<<(unsigned)blocks, kMergeThreads, 0, s>>>(p);
  else if (fin) ring_merge_kernel<false, true><<<(unsigned)blocks, kMergeThreads, 0, s>>>(p);
  else ring_merge_kernel<false, false><<<(unsigned)blocks, kMergeThreads, 0, s>>>(p);
  *nlaunch += 1;
  return cudaGetLastError();
}

}  // namespace bea
