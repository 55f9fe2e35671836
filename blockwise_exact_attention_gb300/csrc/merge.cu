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
// each row's d values are one contiguous, 16-byte-vectorised run. A group of
// d/8 threads owns a row, each thread 8 consecutive elements; every thread
// keeps two rows in flight, and all loads of both rows (the two log-sum-exps,
// the accumulator and the block) are issued before any arithmetic, so that a
// thread has ~100 bytes of independent reads outstanding.
#include <cuda_bf16.h>

#include "common.cuh"
#include "launch_cache.cuh"

namespace bea {
namespace {

constexpr int kMergeThreads = 256;
constexpr int kRowsInFlight = 2;

struct RowData {
  float la, lb;
  float4 a0, a1;  // accumulator, 8 elements
  float4 b0, b1;  // block, 8 elements (converted to fp32)
};

template <bool kBlkF32>
__device__ __forceinline__ void load_row(const MergeParams& p, int64_t r, int c, RowData& x, float*& acc,
                                         float*& la_ptr) {
  const int i = (int)(r % p.l);
  const int64_t bh = r / p.l;
  const int hh = (int)(bh % p.h);
  const int b = (int)(bh / p.h);
  la_ptr = p.lse_acc.ptr + b * p.lse_acc.sn + hh * p.lse_acc.sh + i;
  x.la = *la_ptr;
  x.lb = __ldcs(p.lse_blk.ptr + b * p.lse_blk.sn + hh * p.lse_blk.sh + i);
  acc = reinterpret_cast<float*>(p.acc.ptr) + b * p.acc.sn + (int64_t)i * p.acc.sl + hh * p.acc.sh + c;
  x.a0 = *reinterpret_cast<const float4*>(acc);
  x.a1 = *reinterpret_cast<const float4*>(acc + 4);
  if constexpr (kBlkF32) {
    const float* src =
        reinterpret_cast<const float*>(p.blk.ptr) + b * p.blk.sn + (int64_t)i * p.blk.sl + hh * p.blk.sh + c;
    x.b0 = __ldcs(reinterpret_cast<const float4*>(src));
    x.b1 = __ldcs(reinterpret_cast<const float4*>(src + 4));
  } else {
    const __nv_bfloat16* src = reinterpret_cast<const __nv_bfloat16*>(p.blk.ptr) + b * p.blk.sn +
                               (int64_t)i * p.blk.sl + hh * p.blk.sh + c;
    const uint4 raw = __ldcs(reinterpret_cast<const uint4*>(src));
    const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
    const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
    const float2 f2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.z));
    const float2 f3 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.w));
    x.b0 = make_float4(f0.x, f0.y, f1.x, f1.y);
    x.b1 = make_float4(f2.x, f2.y, f3.x, f3.y);
  }
}

template <bool kFinal>
__device__ __forceinline__ void merge_row(const MergeParams& p, int64_t r, int c, RowData& x, float* acc,
                                          float* la_ptr) {
  const float mx = fmaxf(x.la, x.lb);
  if (mx != -INFINITY) {
    const float mn = fminf(x.la, x.lb);
    const float L = mx + log1pf(expf(mn - mx));
    const float wa = expf(x.la - L);
    const float wb = expf(x.lb - L);
    x.a0 = make_float4(x.a0.x * wa + x.b0.x * wb, x.a0.y * wa + x.b0.y * wb, x.a0.z * wa + x.b0.z * wb,
                       x.a0.w * wa + x.b0.w * wb);
    x.a1 = make_float4(x.a1.x * wa + x.b1.x * wb, x.a1.y * wa + x.b1.y * wb, x.a1.z * wa + x.b1.z * wb,
                       x.a1.w * wa + x.b1.w * wb);
    *reinterpret_cast<float4*>(acc) = x.a0;
    *reinterpret_cast<float4*>(acc + 4) = x.a1;
    if (c == 0) *la_ptr = L;
  }
  if constexpr (kFinal) {
    const int i = (int)(r % p.l);
    const int64_t bh = r / p.l;
    const int hh = (int)(bh % p.h);
    const int b = (int)(bh / p.h);
    __nv_bfloat16* dst =
        reinterpret_cast<__nv_bfloat16*>(p.fin.ptr) + b * p.fin.sn + (int64_t)i * p.fin.sl + hh * p.fin.sh + c;
    const __nv_bfloat162 v0 = __floats2bfloat162_rn(x.a0.x, x.a0.y);
    const __nv_bfloat162 v1 = __floats2bfloat162_rn(x.a0.z, x.a0.w);
    const __nv_bfloat162 v2 = __floats2bfloat162_rn(x.a1.x, x.a1.y);
    const __nv_bfloat162 v3 = __floats2bfloat162_rn(x.a1.z, x.a1.w);
    uint4 raw;
    raw.x = *reinterpret_cast<const uint32_t*>(&v0);
    raw.y = *reinterpret_cast<const uint32_t*>(&v1);
    raw.z = *reinterpret_cast<const uint32_t*>(&v2);
    raw.w = *reinterpret_cast<const uint32_t*>(&v3);
    __stcs(reinterpret_cast<uint4*>(dst), raw);
  }
}

template <bool kBlkF32, bool kFinal>
__global__ void __launch_bounds__(kMergeThreads) ring_merge_kernel(MergeParams p) {
  const int tpr = p.d >> 3;                        // threads per row (2, 4, 8 or 16)
  const int rows_per_pass = kMergeThreads / tpr;   // rows one block covers per row slot
  const int64_t nrows = (int64_t)p.n * p.h * p.l;
  const int sub = threadIdx.x / tpr;
  const int c = (threadIdx.x % tpr) * 8;
  // lanes of one row group share their rows and trip count, so they can sync among themselves
  const unsigned lane0 = (threadIdx.x & 31u) / tpr * tpr;
  const unsigned group_mask = ((1u << tpr) - 1u) << lane0;
  const int64_t stride = (int64_t)gridDim.x * rows_per_pass * kRowsInFlight;
  for (int64_t r0 = ((int64_t)blockIdx.x * rows_per_pass * kRowsInFlight) + sub; r0 < nrows; r0 += stride) {
    const int64_t r1 = r0 + rows_per_pass;
    const bool two = r1 < nrows;
    RowData x0, x1;
    float *acc0, *acc1 = nullptr, *la0, *la1 = nullptr;
    load_row<kBlkF32>(p, r0, c, x0, acc0, la0);
    if (two) load_row<kBlkF32>(p, r1, c, x1, acc1, la1);
    __syncwarp(group_mask);  // every lane of the group has read La before lane c == 0 rewrites it
    merge_row<kFinal>(p, r0, c, x0, acc0, la0);
    if (two) merge_row<kFinal>(p, r1, c, x1, acc1, la1);
  }
}

}  // namespace

cudaError_t launch_ring_merge(const MergeParams& p, cudaStream_t s, int* nlaunch) {
  const int64_t nrows = (int64_t)p.n * p.h * p.l;
  if (nrows == 0) return cudaSuccess;
  const int rows_per_block = kMergeThreads / (p.d >> 3) * kRowsInFlight;
  const bool f32 = p.blk_is_f32 != 0, fin = p.fin.ptr != nullptr;
  auto kern = f32 ? (fin ? ring_merge_kernel<true, true> : ring_merge_kernel<true, false>)
                  : (fin ? ring_merge_kernel<false, true> : ring_merge_kernel<false, false>);
  static PerContext<int> caps[4];  // one wave of resident blocks, per kernel variant and device context
  int cap = 0;
  const cudaError_t e = wave_cap(caps[(f32 ? 2 : 0) + (fin ? 1 : 0)], kern, kMergeThreads, 0, &cap);
  if (e != cudaSuccess) return e;
  int64_t blocks = (nrows + rows_per_block - 1) / rows_per_block;
  if (blocks > cap) blocks = cap;
  kern<<<(unsigned)blocks, kMergeThreads, 0, s>>>(p);
  *nlaunch += 1;
  return cudaGetLastError();
}

}  // namespace bea
