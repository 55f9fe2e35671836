// Exact fp32 attention on the SIMT cores (no tensor cores): the path for f32
// inputs, where tcgen05 kind::tf32 would round the operands to 10 mantissa
// bits.
//
// Forward: one warp per query row; K/V stream through shared memory in tiles
// of 32 keys, each lane scores one key of the tile, and the running max/sum
// of the online softmax are warp reductions (picotron context_parallel.py,
// ring_attention_forward, computed one key tile at a time).
// Backward (same page, ring_attention_backward, Steps 1-6): one kernel forms
// D = rowsum(dO * O), one kernel walks keys per query row for dQ, and one
// walks queries per key row for dK and dV, summing over the query heads that
// share the K/V head.
#include <cmath>

#include "common.cuh"

namespace bea {
namespace {

constexpr int kWarps = 8;
constexpr int kTile = 32;
constexpr int kMaxD = 128;
constexpr int kPad = kMaxD + 1;  // row pitch in floats: avoids shared-memory bank conflicts

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__device__ __forceinline__ const float* row_ptr(const Seq4& t, int b, int i, int hh) {
  return reinterpret_cast<const float*>(t.ptr) + b * t.sn + (int64_t)i * t.sl + hh * t.sh;
}
__device__ __forceinline__ float* row_ptr_w(const Seq4& t, int b, int i, int hh) {
  return reinterpret_cast<float*>(t.ptr) + b * t.sn + (int64_t)i * t.sl + hh * t.sh;
}

__global__ void __launch_bounds__(kWarps * 32) fwd_f32_kernel(F32FwdParams p) {
  __shared__ float sK[kTile][kPad];
  __shared__ float sV[kTile][kPad];
  __shared__ float sQ[kWarps][kPad];
  const AttnDims& a = p.a;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int hq = blockIdx.y, b = blockIdx.z, kvh = hq / (a.h / a.hkv);
  const int i0 = blockIdx.x * kWarps;
  const int i = i0 + warp;
  const int d = a.d;
  const bool row_ok = i < a.lq;
  if (row_ok)
    for (int c = lane; c < d; c += 32) sQ[warp][c] = row_ptr(p.q, b, i, hq)[c];
  const int last = min(a.lq - 1, i0 + kWarps - 1);
  const int j_lo = (int)max(0LL, (long long)i0 - a.wl);
  const int j_hi = (int)max((long long)j_lo, min((long long)a.lk, (long long)last + a.wr + 1));
  float m = -INFINITY, l = 0.f;
  float acc[kMaxD / 32];
#pragma unroll
  for (int t = 0; t < kMaxD / 32; ++t) acc[t] = 0.f;
  for (int j0 = j_lo; j0 < j_hi; j0 += kTile) {
    __syncthreads();
    for (int e = threadIdx.x; e < kTile * d; e += blockDim.x) {
      const int jj = e / d, c = e % d, j = j0 + jj;
      sK[jj][c] = (j < a.lk) ? row_ptr(p.k, b, j, kvh)[c] : 0.f;
      sV[jj][c] = (j < a.lk) ? row_ptr(p.v, b, j, kvh)[c] : 0.f;
    }
    __syncthreads();
    if (!row_ok) continue;
    const int j = j0 + lane;
    float s = -INFINITY;
    if (j < j_hi && key_visible(i, j, a.wl, a.wr)) {
      float dot = 0.f;
      for (int c = 0; c < d; ++c) dot = fmaf(sQ[warp][c], sK[lane][c], dot);
      s = dot * a.scale;
    }
    const float m_new = fmaxf(m, warp_max(s));
    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
    const float alpha = expf(m - m_use);
    const float pj = expf(s - m_use);
    l = l * alpha + warp_sum(pj);
    m = m_new;
#pragma unroll
    for (int t = 0; t < kMaxD / 32; ++t) {
      const int c = lane + 32 * t;
      float x = acc[t] * alpha;
      for (int jj = 0; jj < kTile; ++jj) {
        const float w = __shfl_sync(0xffffffffu, pj, jj);
        if (c < d) x = fmaf(w, sV[jj][c], x);
      }
      acc[t] = x;
    }
  }
  if (!row_ok) return;
  const float inv = (l > 0.f) ? 1.f / l : 0.f;
  float* o = row_ptr_w(p.out, b, i, hq);
#pragma unroll
  for (int t = 0; t < kMaxD / 32; ++t) {
    const int c = lane + 32 * t;
    if (c < d) o[c] = acc[t] * inv;
  }
  if (lane == 0) p.lse.ptr[b * p.lse.sn + hq * p.lse.sh + i] = (l > 0.f) ? m + logf(l) : -INFINITY;
}

// D[b, h, i] = sum_c dO[b, i, h, c] * O[b, i, h, c]   (Step 3)
__global__ void __launch_bounds__(kWarps * 32) bwd_f32_rowdot_kernel(F32BwdParams p) {
  const AttnDims& a = p.a;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int i = blockIdx.x * kWarps + warp, hq = blockIdx.y, b = blockIdx.z;
  if (i >= a.lq) return;
  const float* o = row_ptr(p.out, b, i, hq);
  const float* g = row_ptr(p.dout, b, i, hq);
  float s = 0.f;
  for (int c = lane; c < a.d; c += 32) s = fmaf(o[c], g[c], s);
  s = warp_sum(s);
  if (lane == 0) p.D[((int64_t)b * a.h + hq) * a.lq + i] = s;
}

// dQ_i = scale * sum_j P_ij (dO_i . v_j - D_i) k_j   (Steps 4-5)
__global__ void __launch_bounds__(kWarps * 32) bwd_f32_dq_kernel(F32BwdParams p) {
  __shared__ float sK[kTile][kPad];
  __shared__ float sV[kTile][kPad];
  __shared__ float sQ[kWarps][kPad];
  __shared__ float sG[kWarps][kPad];
  const AttnDims& a = p.a;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int hq = blockIdx.y, b = blockIdx.z, kvh = hq / (a.h / a.hkv);
  const int i0 = blockIdx.x * kWarps, i = i0 + warp, d = a.d;
  const bool row_ok = i < a.lq;
  float lse = -INFINITY, Dv = 0.f;
  if (row_ok) {
    for (int c = lane; c < d; c += 32) {
      sQ[warp][c] = row_ptr(p.q, b, i, hq)[c];
      sG[warp][c] = row_ptr(p.dout, b, i, hq)[c];
    }
    lse = p.lse.ptr[b * p.lse.sn + hq * p.lse.sh + i];
    Dv = p.D[((int64_t)b * a.h + hq) * a.lq + i];
  }
  const int last = min(a.lq - 1, i0 + kWarps - 1);
  const int j_lo = (int)max(0LL, (long long)i0 - a.wl);
  const int j_hi = (int)max((long long)j_lo, min((long long)a.lk, (long long)last + a.wr + 1));
  float acc[kMaxD / 32];
#pragma unroll
  for (int t = 0; t < kMaxD / 32; ++t) acc[t] = 0.f;
  for (int j0 = j_lo; j0 < j_hi; j0 += kTile) {
    __syncthreads();
    for (int e = threadIdx.x; e < kTile * d; e += blockDim.x) {
      const int jj = e / d, c = e % d, j = j0 + jj;
      sK[jj][c] = (j < a.lk) ? row_ptr(p.k, b, j, kvh)[c] : 0.f;
      sV[jj][c] = (j < a.lk) ? row_ptr(p.v, b, j, kvh)[c] : 0.f;
    }
    __syncthreads();
    if (!row_ok) continue;
    const int j = j0 + lane;
    float ds = 0.f;
    if (j < j_hi && key_visible(i, j, a.wl, a.wr) && lse != -INFINITY) {
      float s = 0.f, dp = 0.f;
      for (int c = 0; c < d; ++c) {
        s = fmaf(sQ[warp][c], sK[lane][c], s);
        dp = fmaf(sG[warp][c], sV[lane][c], dp);
      }
      const float pij = expf(s * a.scale - lse);
      ds = pij * (dp - Dv);
    }
#pragma unroll
    for (int t = 0; t < kMaxD / 32; ++t) {
      const int c = lane + 32 * t;
      float x = acc[t];
      for (int jj = 0; jj < kTile; ++jj) {
        const float w = __shfl_sync(0xffffffffu, ds, jj);
        if (c < d) x = fmaf(w, sK[jj][c], x);
      }
      acc[t] = x;
    }
  }
  if (!row_ok) return;
  float* dq = row_ptr_w(p.dq, b, i, hq);
#pragma unroll
  for (int t = 0; t < kMaxD / 32; ++t) {
    const int c = lane + 32 * t;
    if (c < d) dq[c] = p.accumulate ? dq[c] + acc[t] * a.scale : acc[t] * a.scale;
  }
}

// dV_j = sum_{hq in group, i} P_ij dO_i ;  dK_j = scale * sum P_ij (dO_i . v_j - D_i) q_i   (Steps 1, 4, 6)
__global__ void __launch_bounds__(kWarps * 32) bwd_f32_dkv_kernel(F32BwdParams p) {
  __shared__ float sQ[kTile][kPad];
  __shared__ float sG[kTile][kPad];
  __shared__ float sK[kWarps][kPad];
  __shared__ float sV[kWarps][kPad];
  __shared__ float sL[kTile], sD[kTile];
  const AttnDims& a = p.a;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int kvh = blockIdx.y, b = blockIdx.z, g = a.h / a.hkv;
  const int j0 = blockIdx.x * kWarps, j = j0 + warp, d = a.d;
  const bool row_ok = j < a.lk;
  if (row_ok)
    for (int c = lane; c < d; c += 32) {
      sK[warp][c] = row_ptr(p.k, b, j, kvh)[c];
      sV[warp][c] = row_ptr(p.v, b, j, kvh)[c];
    }
  const int jlast = min(a.lk - 1, j0 + kWarps - 1);
  const int i_lo = (int)max(0LL, (long long)j0 - a.wr);
  const int i_hi = (int)max((long long)i_lo, min((long long)a.lq, (long long)jlast + a.wl + 1));
  float accK[kMaxD / 32], accV[kMaxD / 32];
#pragma unroll
  for (int t = 0; t < kMaxD / 32; ++t) accK[t] = accV[t] = 0.f;
  for (int hq = kvh * g; hq < (kvh + 1) * g; ++hq) {
    for (int i0 = i_lo; i0 < i_hi; i0 += kTile) {
      __syncthreads();
      for (int e = threadIdx.x; e < kTile * d; e += blockDim.x) {
        const int ii = e / d, c = e % d, i = i0 + ii;
        sQ[ii][c] = (i < a.lq) ? row_ptr(p.q, b, i, hq)[c] : 0.f;
        sG[ii][c] = (i < a.lq) ? row_ptr(p.dout, b, i, hq)[c] : 0.f;
      }
      if (threadIdx.x < kTile) {
        const int i = i0 + threadIdx.x;
        sL[threadIdx.x] = (i < a.lq) ? p.lse.ptr[b * p.lse.sn + hq * p.lse.sh + i] : -INFINITY;
        sD[threadIdx.x] = (i < a.lq) ? p.D[((int64_t)b * a.h + hq) * a.lq + i] : 0.f;
      }
      __syncthreads();
      if (!row_ok) continue;
      const int i = i0 + lane;
      float pij = 0.f, ds = 0.f;
      if (i < i_hi && key_visible(i, j, a.wl, a.wr) && sL[lane] != -INFINITY) {
        float s = 0.f, dp = 0.f;
        for (int c = 0; c < d; ++c) {
          s = fmaf(sQ[lane][c], sK[warp][c], s);
          dp = fmaf(sG[lane][c], sV[warp][c], dp);
        }
        pij = expf(s * a.scale - sL[lane]);
        ds = pij * (dp - sD[lane]);
      }
#pragma unroll
      for (int t = 0; t < kMaxD / 32; ++t) {
        const int c = lane + 32 * t;
        float xk = accK[t], xv = accV[t];
        for (int ii = 0; ii < kTile; ++ii) {
          const float wp = __shfl_sync(0xffffffffu, pij, ii);
          const float wd = __shfl_sync(0xffffffffu, ds, ii);
          if (c < d) {
            xv = fmaf(wp, sG[ii][c], xv);
            xk = fmaf(wd, sQ[ii][c], xk);
          }
        }
        accK[t] = xk;
        accV[t] = xv;
      }
    }
  }
  if (!row_ok) return;
  float* dk = row_ptr_w(p.dk, b, j, kvh);
  float* dv = row_ptr_w(p.dv, b, j, kvh);
#pragma unroll
  for (int t = 0; t < kMaxD / 32; ++t) {
    const int c = lane + 32 * t;
    if (c < d) {
      dk[c] = p.accumulate ? dk[c] + accK[t] * a.scale : accK[t] * a.scale;
      dv[c] = p.accumulate ? dv[c] + accV[t] : accV[t];
    }
  }
}

}  // namespace

cudaError_t launch_fwd_f32(const F32FwdParams& p, cudaStream_t s, int* nlaunch) {
  if (p.a.lq == 0 || p.a.n == 0 || p.a.h == 0) return cudaSuccess;
  dim3 grid((p.a.lq + kWarps - 1) / kWarps, p.a.h, p.a.n);
  fwd_f32_kernel<<<grid, kWarps * 32, 0, s>>>(p);
  *nlaunch += 1;
  return cudaGetLastError();
}

cudaError_t launch_bwd_f32(const F32BwdParams& p, cudaStream_t s, int* nlaunch) {
  const AttnDims& a = p.a;
  if (a.n == 0 || a.h == 0) return cudaSuccess;
  if (a.lq > 0) {
    dim3 gq((a.lq + kWarps - 1) / kWarps, a.h, a.n);
    bwd_f32_rowdot_kernel<<<gq, kWarps * 32, 0, s>>>(p);
    bwd_f32_dq_kernel<<<gq, kWarps * 32, 0, s>>>(p);
    *nlaunch += 2;
  }
  if (a.lk > 0) {
    dim3 gk((a.lk + kWarps - 1) / kWarps, a.hkv, a.n);
    bwd_f32_dkv_kernel<<<gk, kWarps * 32, 0, s>>>(p);
    *nlaunch += 1;
  }
  return cudaGetLastError();
}

}  // namespace bea
