// Attention backward on sm_103a tensor cores, recomputed from the log-sum-exp.
//
// picotron context_parallel.py, ring_attention_backward, Steps 1-6:
//   P = exp(scale Q K^T - L)  (masked entries 0)
//   dV = P^T dO,  dP = dO V^T,  D = rowsum(dO * O),  dS = P * (dP - D),
//   dQ = scale dS K,  dK = scale dS^T Q,
// with dK, dV summed over the query heads that share a K/V head
// (RingAttention._repeat_kv read backwards). O and L are the caller's, not
// recomputed, so partial gradients of ring chunk pairs add up exactly.
//
// Three launches:
//   1. preprocess: D and L*log2(e) per query row into the workspace (padding
//      rows get D = 0, L2 = +inf so that their P is exactly 0), and the fp32
//      dQ accumulator rows zeroed;
//   2. main: one CTA per (128-key block, batch, K/V head). K and V stay in
//      shared memory; the CTA walks the group's query heads x the 128-row
//      query tiles the causal/window band lets it see, each tile as two
//      64-query halves:
//        warp 12     producer: K, V once; per tile Q_i and dO_i (TMA) and the
//                    tile's L2 and D rows (bulk copies) into 2 stages,
//        warp 13     MMA issuer (the whole warp, one elected lane issues):
//                    per half h, S_h^T = K Q_h^T and dP_h^T = V dO_h^T into
//                    TMEM slot h; then, per half as soon as its P^T / dS^T
//                    are ready, dQ_h^T = K^T dS_h^T (dS^T from shared
//                    memory), dV += P_h^T dO_h and dK += dS_h^T Q_h (P^T,
//                    dS^T from TMEM). Each half's products for this tile are
//                    followed at once by that half's S^T / dP^T for the
//                    next tile, so the key warps' work on one half hides
//                    behind the tensor work of the other,
//        warps 0-7   two warpgroups, one thread per key each: warpgroup c
//                    forms P^T and dS^T of queries [32c, 32c+32) of every
//                    half from S^T, dP^T, L2, D; finally warpgroup 0 writes
//                    dV and warpgroup 1 dK,
//        warps 8-11  one thread per head-dim index: read dQ_h^T out of TMEM
//                    and add it into the fp32 accumulator, four query rows per
//                    16-byte reduction; the 32 lanes of a warp cover 32
//                    consecutive entries, one contiguous 512-byte span.
//      Two TMEM slots let the tensor core compute one half while the key
//      warps work on the other, and the drain of one half's dQ^T overlaps
//      the other half's products. dK and dV accumulate in TMEM across the
//      whole group: no atomics.
//   3. convert: dQ = scale * accumulator, cast or added into the caller's dq.
//
// TMEM (512 columns): slot h = [128h, 128h+128) holds S_h^T in its first 64
// columns and dP_h^T in the last 64 (later dQ_h^T); dV [256,256+D), dK
// [384,384+D). Key warpgroup c overwrites the 32 S^T columns it has read,
// [128h + 32c, +32), with its queries' P^T (16 columns of packed bf16 pairs)
// and dS^T (16 columns): the TMEM A operands of dV += P^T dO and dK += dS^T Q.
#include <cuda_bf16.h>

#include "common.cuh"
#include "launch_cache.cuh"
#include "ptx.cuh"

namespace bea {
namespace {

constexpr int kBM = 128;  // query rows per iteration
constexpr int kBN = 128;  // keys per CTA
constexpr int kHeadBand = 4;  // K/V heads per band of the CTA order under a mask band
constexpr int kThreads = 512;  // 4 warpgroups
// Register split: launched at kRegsLaunch per thread (65536 / 512); the two
// key-row warpgroups rise to kRegsCompute, the dQ drain and the producer/MMA
// warpgroup drop to kRegsDrain and kRegsOther:
// 128 * (2 * 152 + 80 + 128) = 512 * 128.
constexpr int kRegsLaunch = 128;
constexpr int kRegsCompute = 152;
constexpr int kRegsDrain = 80;
constexpr int kRegsOther = 128;
static_assert(2 * kRegsCompute + kRegsDrain + kRegsOther == 4 * kRegsLaunch, "register split");
constexpr int kDrainWarp0 = 8;  // warps 8-11
constexpr int kProducerWarp = 12;
constexpr int kMmaWarp = 13;
// "P_h^T / dS_h^T written" goes from the 8 key warps to the MMA warp over
// hardware named barrier kReadyBar + h (one phase per tile; barrier 0 is
// __syncthreads). "dQ_h^T read out of slot h" goes from the drain to the MMA
// warp over an mbarrier: the drain must start its reductions at once, and an
// mbarrier arrival does not wait.
// A named barrier has no time limit, so the phases stay matched on every path:
// every side joins every phase of a barrier once, in tile/half order, with or
// without work (after an abort), and every join waits for the phase to
// complete (barrier.sync, never a bare arrive). No warp can then join phase
// k+1 while phase k is open; a bare arrive followed by an aborting warp's next
// join could land both in one phase and leave a later phase short. The key
// warps' next step waits for an MMA the MMA warp issues only after this phase,
// so the wait costs them nothing.
constexpr uint32_t kReadyBar = 1;
constexpr uint32_t kReadyThreads = 256 + 32;
// dK / dV epilogue of key warpgroup c: its 128 threads hand the staged chunk to one
// another over named barrier kEpiBar + c (every thread joins every phase, with or without work).
constexpr uint32_t kEpiBar = 3;

template <int D>
struct BwdCfg {
  static constexpr int kBoxes = D / 64;
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKOff + kTileBytes;
  static constexpr int kQOff = kVOff + kTileBytes;          // 2 stages
  static constexpr int kDOOff = kQOff + 2 * kTileBytes;     // 2 stages
  static constexpr int kDSOff = kDOOff + 2 * kTileBytes;    // dS^T [128 keys x 128 q] bf16
  static constexpr int kDSBytes = 128 * 128 * 2;
  static constexpr int kRowOff = kDSOff + kDSBytes;         // 2 stages of L2[128], D[128] fp32
  static constexpr int kBarOff = kRowOff + 2 * 1024;
  static constexpr int kNumBars = 2 + 2 + 2 + 2 + 2 + 2 + 2 + 1 + 1;
  static constexpr int kSmemBytes = kBarOff + kNumBars * 8 + 16 /*tmem slot, abort*/;
  static constexpr uint32_t kIdescS = idesc_bf16_f32(128, 64, false, false);    // S_h^T, dP_h^T
  static constexpr uint32_t kIdescKV = idesc_bf16_f32(128, D, false, true);     // dV (TMEM A), dK
  // dQ_h^T = K^T dS_h^T: M = 128 head-dim rows (for d = 64 the upper half are padding rows), N = 64 queries
  static constexpr uint32_t kIdescQ = idesc_bf16_f32(128, 64, true, true);
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// The fp32 dQ accumulator is [n, h, lq_pad, d], row-major.

// ---------------------------------------------------------------------------
// 1. preprocess and 3. convert: HBM-bound row kernels
// ---------------------------------------------------------------------------
//
// A group of D/8 threads owns a row, each thread 8 consecutive elements
// (16-byte loads and stores); every thread keeps two rows in flight and the
// grid is one wave of resident CTAs.

constexpr int kRowThreads = 256;

__device__ __forceinline__ void bf16x8_to_f32(const uint4 raw, float* f) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const float2 t = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[u]));
    f[2 * u] = t.x;
    f[2 * u + 1] = t.y;
  }
}

// Eight elements of row i of a [n, l, h, d] tensor starting at column c, as fp32.
__device__ __forceinline__ void load8(const Seq4& t, bool f32, int b, int i, int hh, int c, float* f) {
  if (f32) {
    const float* src = reinterpret_cast<const float*>(t.ptr) + b * t.sn + (int64_t)i * t.sl + hh * t.sh + c;
    const float4 lo = *reinterpret_cast<const float4*>(src);
    const float4 hi = *reinterpret_cast<const float4*>(src + 4);
    f[0] = lo.x; f[1] = lo.y; f[2] = lo.z; f[3] = lo.w;
    f[4] = hi.x; f[5] = hi.y; f[6] = hi.z; f[7] = hi.w;
  } else {
    const __nv_bfloat16* src =
        reinterpret_cast<const __nv_bfloat16*>(t.ptr) + b * t.sn + (int64_t)i * t.sl + hh * t.sh + c;
    bf16x8_to_f32(*reinterpret_cast<const uint4*>(src), f);
  }
}

// D = rowsum(dO * O), L * log2(e) (+inf for rows without keys and for padding
// rows, so that their P is exactly 0) and a zeroed row of the dQ accumulator,
// for every padded query row.
template <int D>
__global__ void __launch_bounds__(kRowThreads) bwd_preprocess_kernel(BwdParams p) {
  constexpr int kTpr = D / 8;
  constexpr int kRowsPerPass = kRowThreads / kTpr;
  const AttnDims& a = p.a;
  const int64_t total = (int64_t)a.n * a.h * p.lq_pad;
  const int sub = threadIdx.x / kTpr;
  const int c = (threadIdx.x % kTpr) * 8;
  const unsigned lane0 = (threadIdx.x & 31u) / kTpr * kTpr;
  const unsigned group_mask = (kTpr >= 32) ? 0xffffffffu : (((1u << kTpr) - 1u) << lane0);
  const int64_t stride = (int64_t)gridDim.x * kRowsPerPass * 2;
  for (int64_t r0 = (int64_t)blockIdx.x * kRowsPerPass * 2 + sub; r0 < total; r0 += stride) {
    float dsum[2] = {0.f, 0.f}, lse[2] = {-INFINITY, -INFINITY};
    int64_t rows[2] = {r0, r0 + kRowsPerPass};
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int64_t row = rows[u];
      if (row >= total) continue;
      const int i = (int)(row % p.lq_pad);
      const int bh = (int)(row / p.lq_pad);
      const int hq = bh % a.h, b = bh / a.h;
      if (i < a.lq) {
        float g[8], o[8];
        load8(p.dout, false, b, i, hq, c, g);
        load8(p.out, p.out_is_f32 != 0, b, i, hq, c, o);
#pragma unroll
        for (int e = 0; e < 8; ++e) dsum[u] = fmaf(g[e], o[e], dsum[u]);
        lse[u] = p.lse.ptr[b * p.lse.sn + hq * p.lse.sh + i];
      }
      float* acc = p.dq_acc + (size_t)row * D + c;
      *reinterpret_cast<float4*>(acc) = make_float4(0.f, 0.f, 0.f, 0.f);
      *reinterpret_cast<float4*>(acc + 4) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
#pragma unroll
      for (int off = kTpr / 2; off > 0; off >>= 1) dsum[u] += __shfl_xor_sync(group_mask, dsum[u], off);
      if (c == 0 && rows[u] < total) {
        p.d_row[rows[u]] = dsum[u];
        p.lse2[rows[u]] = (lse[u] == -INFINITY) ? INFINITY : lse[u] * 1.4426950408889634f;
      }
    }
  }
}

// dq = scale * accumulator, cast to bf16, written, or added to an fp32 dq. The
// accumulator is [n h][lq_pad / 4][D][4] (four query rows interleaved per
// head-dim index). A thread takes two consecutive head-dim entries of a group of
// four rows, 32 contiguous bytes: a warp reads one contiguous 1 KB span and
// writes 64 consecutive entries of each of the four rows. Every thread keeps two
// groups in flight.
template <int D>
__global__ void __launch_bounds__(kRowThreads) bwd_convert_dq_kernel(BwdParams p) {
  constexpr int kTpg = D / 2;                         // threads per group of four rows
  constexpr int kGroupsPerPass = kRowThreads / kTpg;  // groups of a block's pass, per half
  const AttnDims& a = p.a;
  const int64_t groups_bh = (a.lq + 3) / 4;
  const int64_t total = (int64_t)a.n * a.h * groups_bh;
  const int sub = threadIdx.x / kTpg;
  const int e = (threadIdx.x % kTpg) * 2;  // head-dim entries e and e + 1
  const int64_t stride = (int64_t)gridDim.x * kGroupsPerPass * 2;
  for (int64_t g0 = (int64_t)blockIdx.x * kGroupsPerPass * 2 + sub; g0 < total; g0 += stride) {
    const int64_t gs[2] = {g0, g0 + kGroupsPerPass};
    float4 q4[2][2];  // [u][k]: the four rows of group gs[u] at entry e + k
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (gs[u] >= total) continue;
      const int64_t bh = gs[u] / groups_bh;
      const int64_t gi = gs[u] % groups_bh;
      const float* acc = p.dq_acc + ((size_t)bh * (p.lq_pad / 4) + gi) * (D * 4) + e * 4;
      q4[u][0] = *reinterpret_cast<const float4*>(acc);
      q4[u][1] = *reinterpret_cast<const float4*>(acc + 4);
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (gs[u] >= total) continue;
      const int64_t bh = gs[u] / groups_bh;
      const int gi = (int)(gs[u] % groups_bh);
      const int hq = (int)(bh % a.h), b = (int)(bh / a.h);
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int i = 4 * gi + r;
        if (i >= a.lq) break;
        const float4& x0 = q4[u][0];
        const float4& x1 = q4[u][1];
        float v0 = (r == 0 ? x0.x : r == 1 ? x0.y : r == 2 ? x0.z : x0.w) * a.scale;
        float v1 = (r == 0 ? x1.x : r == 1 ? x1.y : r == 2 ? x1.z : x1.w) * a.scale;
        if (p.dq_is_f32) {
          float* dst = reinterpret_cast<float*>(p.dq.ptr) + b * p.dq.sn + (int64_t)i * p.dq.sl + hq * p.dq.sh + e;
          if (p.accumulate) {
            const float2 old = *reinterpret_cast<const float2*>(dst);
            v0 += old.x;
            v1 += old.y;
          }
          *reinterpret_cast<float2*>(dst) = make_float2(v0, v1);
        } else {
          __nv_bfloat16* dst =
              reinterpret_cast<__nv_bfloat16*>(p.dq.ptr) + b * p.dq.sn + (int64_t)i * p.dq.sl + hq * p.dq.sh + e;
          *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(v0, v1);
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// 2. main kernel
// ---------------------------------------------------------------------------

struct BwdSched {
  int k0;          // first key of the block
  int i_lo, i_hi;  // visible query tiles
  int g;           // query heads per K/V head
  int n_iter;      // g * (i_hi - i_lo)
};

__device__ __forceinline__ bool bwd_tile_needs_mask(const AttnDims& a, int k0, int q0) {
  if (k0 + kBN - 1 >= a.lk) return true;
  if ((long long)k0 < (long long)q0 + kBM - 1 - a.wl) return true;
  if ((long long)k0 + kBN - 1 > (long long)q0 + a.wr) return true;
  return false;
}

// One 32-query chunk of the compute warpgroup: P^T and dS^T for this
// thread's key row from S^T, dP^T (registers), L2 and D (shared memory).
// The mask decision is a template parameter so that the unrolled element
// loop has no branches and the 32 independent element chains interleave.
template <int D, bool kMask>
__device__ __forceinline__ void bwd_chunk(const uint32_t* sv, const uint32_t* pv, const float* l2s, const float* dds,
                                          int cc, const AttnDims& a, int kj, int q0, float scale_log2,
                                          uint32_t p_dst, uint8_t* ds_row, int j) {
  uint32_t pk[16], dk[16];
  const uint64_t sl2 = f2(scale_log2, scale_log2);
#pragma unroll
  for (int e4 = 0; e4 < 8; ++e4) {
    const float4 L4 = *reinterpret_cast<const float4*>(l2s + cc * 32 + e4 * 4);
    const float4 D4 = *reinterpret_cast<const float4*>(dds + cc * 32 + e4 * 4);
    const uint64_t nL[2] = {f2(-L4.x, -L4.y), f2(-L4.z, -L4.w)};
    const uint64_t nD[2] = {f2(-D4.x, -D4.y), f2(-D4.z, -D4.w)};
    // two queries per packed fp32 operation: P = exp2(S scale log2e - L log2e), dS = P (dP - D)
#pragma unroll
    for (int u2 = 0; u2 < 2; ++u2) {
      const int e = e4 * 4 + 2 * u2;
      const uint64_t x = f2_fma(f2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), sl2, nL[u2]);
      float p0 = ex2_approx(f2_lo(x));
      float p1 = ex2_approx(f2_hi(x));
      if constexpr (kMask) {
        const int qi = q0 + cc * 32 + e;
        p0 = ((kj < a.lk) & key_visible(qi, kj, a.wl, a.wr)) ? p0 : 0.f;
        p1 = ((kj < a.lk) & key_visible(qi + 1, kj, a.wl, a.wr)) ? p1 : 0.f;
      }
      const uint64_t ds = f2_mul(f2(p0, p1), f2_add(f2(__uint_as_float(pv[e]), __uint_as_float(pv[e + 1])), nD[u2]));
      pk[e4 * 2 + u2] = pack_bf16x2(p0, p1);
      dk[e4 * 2 + u2] = pack_bf16x2(f2_lo(ds), f2_hi(ds));
    }
  }
  // P^T and dS^T (packed bf16 pairs) over the 32 S^T columns this thread has just read:
  // P^T in the first 16, dS^T in the last 16 (the A operands of dV += P^T dO and dK += dS^T Q)
  tmem_st16(p_dst, pk);
  tmem_st16(p_dst + 16, dk);
  // dS^T row j, queries [32cc, 32cc+32): 4 chunks of 16 B, 128-byte swizzle
  uint8_t* half = ds_row + (cc >> 1) * 16384;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int chunk = (cc & 1) * 4 + u;
    const int phys = chunk ^ (j & 7);
    *reinterpret_cast<uint4*>(half + phys * 16) = make_uint4(dk[4 * u], dk[4 * u + 1], dk[4 * u + 2], dk[4 * u + 3]);
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_bf16_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                    const __grid_constant__ CUtensorMap tdk, const __grid_constant__ CUtensorMap tdv,
                    const BwdParams p, float scale_log2) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* k_full = bars;            // K and V of the CTA's key block land separately: S needs
  uint64_t* v_full = bars + 1;        // only K and Q, dP only V and dO
  uint64_t* q_full = bars + 2;        // Q_i, L2_i, D_i of a stage
  uint64_t* do_full = q_full + 2;
  uint64_t* qdo_empty = do_full + 2;
  uint64_t* sp_full = qdo_empty + 2;  // [2]: S_h^T and dP_h^T of half h are in TMEM slot h
  uint64_t* dq_full = sp_full + 2;    // [2]: dQ_h^T in TMEM slot h
  uint64_t* dq_empty = dq_full + 2;   // [2]: dQ_h^T read out of slot h (128 drain threads arrive)
  uint64_t* dkv_full = dq_empty + 2;
  uint64_t* mma_done = dkv_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  // The swizzled operand tiles need 1024-byte alignment; the dynamic shared
  // window starts there when the kernel has no static shared memory.
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) report_status(p.status, BEA_STATUS_CONFIG);
    return;
  }

  const AttnDims& a = p.a;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  // ---- work: key blocks in ascending order (under a causal mask the first see the most queries) ----
  // When the band covers every (query, key) pair (no mask, or a ring step's chunk pair that
  // lies wholly inside it) every CTA has the same work. With one query head per K/V head the
  // CTAs are then taken head by head, so that the ones running together share one head's
  // Q/dO tiles and dQ accumulator rows in L2 (measured: 32k d=64 full attention -12%, 8k d=128
  // -6%; the 16k ring's full chunk pairs, run as a batch of 7 chunks x 16 heads, would otherwise
  // spread ~150 heads' Q/dO/dQ over L2). Under a causal or window band the batches go one
  // after another and, within one, the key blocks in ascending order (longest first) with the
  // K/V heads fastest; so do grouped heads (their 4x longer CTAs measured 3% slower head by head).
  const int nkb = (a.lk + kBN - 1) / kBN;
  const bool full_band = a.wl >= a.lq - 1 && a.wr >= a.lk - 1;
  const bool head_major = full_band && a.h == a.hkv;
  // Under a band the K/V heads of a batch go in bands of kHeadBand, one band after another, so
  // that at most a band's Q/dO tiles and dQ rows are live in L2 at once; within a band the key
  // blocks in ascending order with the band's K/V heads fastest.
  const int per_batch = nkb * a.hkv;
  int kb, kvh;
  if (head_major) {
    kb = (int)(blockIdx.x % nkb);
    kvh = (int)((blockIdx.x / nkb) % a.hkv);
  } else {
    const int r = (int)(blockIdx.x % per_batch);
    const int band = r / (kHeadBand * nkb);
    const int h0 = band * kHeadBand;
    const int bw = min(kHeadBand, a.hkv - h0);  // K/V heads in this band
    const int rr = r - band * kHeadBand * nkb;
    kb = rr / bw;
    kvh = h0 + rr % bw;
  }
  const int b = (int)(blockIdx.x / per_batch);
  BwdSched sc;
  sc.k0 = kb * kBN;
  sc.g = a.h / a.hkv;
  {
    const int k1 = min(sc.k0 + kBN, a.lk) - 1;
    const int qmin = (int)max(0LL, (long long)sc.k0 - a.wr);
    const int qmax = (int)min((long long)a.lq, (long long)k1 + a.wl + 1);
    if (qmax > qmin) {
      sc.i_lo = qmin / kBM;
      sc.i_hi = (qmax + kBM - 1) / kBM;
    } else {
      sc.i_lo = sc.i_hi = 0;
    }
    sc.n_iter = sc.g * (sc.i_hi - sc.i_lo);
  }
  const int nt = sc.i_hi - sc.i_lo;

  // The producer's loads of iteration it: Q_i with its L log2e and D rows, the CTA's V (with the
  // first), dO_i. Load order K, Q_0, V, dO_0: the first S products need only K and Q_0 and run
  // while V and dO_0 arrive.
  auto issue_iter = [&](int it) {
    const int s = it & 1;
    const int hq = kvh * sc.g + it / nt;
    const int q0 = (sc.i_lo + it % nt) * kBM;
    mbar_arrive_expect_tx(&q_full[s], C::kTileBytes + 2 * kBM * 4);
    for (int x = 0; x < C::kBoxes; ++x)
      tma_load_4d(smem + C::kQOff + s * C::kTileBytes + x * 16384, &tq, &q_full[s], x * 64, hq, q0, b);
    const size_t row0 = (size_t)(b * a.h + hq) * p.lq_pad + q0;
    bulk_load(smem + C::kRowOff + s * 1024, p.lse2 + row0, kBM * 4, &q_full[s]);
    bulk_load(smem + C::kRowOff + s * 1024 + 512, p.d_row + row0, kBM * 4, &q_full[s]);
    if (it == 0) {
      mbar_arrive_expect_tx(v_full, C::kTileBytes);
      for (int x = 0; x < C::kBoxes; ++x)
        tma_load_4d(smem + C::kVOff + x * 16384, &tv, v_full, x * 64, kvh, sc.k0, b);
    }
    mbar_arrive_expect_tx(&do_full[s], C::kTileBytes);
    for (int x = 0; x < C::kBoxes; ++x)
      tma_load_4d(smem + C::kDOOff + s * C::kTileBytes + x * 16384, &tdo, &do_full[s], x * 64, hq, q0, b);
  };

  // The producer's lane initialises the barriers and sends the loads that wait on nothing (K and
  // the first two iterations' Q/dO) before the CTA-wide barrier, so that they are in flight while
  // TMEM is allocated and the other warps arrive.
  // The barriers of the first loads (K, V, Q/dO of two stages: bars[0, 6)) are the producer
  // lane's; the warp's other lanes initialise the rest meanwhile, one each.
  int it_early = 0;  // producer lane: iterations already issued
  constexpr int kFirstBars = 6;
  if (warp == kProducerWarp && lane > 0 && lane <= C::kNumBars - kFirstBars) {
    uint64_t* bar = &bars[kFirstBars + lane - 1];
    mbar_init(bar, (bar == &dq_empty[0] || bar == &dq_empty[1]) ? 128 : 1);
    fence_mbar_init();
  }
  if (threadIdx.x == kProducerWarp * 32) {
    *abort_flag = 0;
    mbar_init(k_full, 1);
    mbar_init(v_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&do_full[s], 1);
    }
    fence_mbar_init();
    if (sc.n_iter > 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
      prefetch_tmap(&tdo);
      prefetch_tmap(&tdk);
      prefetch_tmap(&tdv);
      mbar_arrive_expect_tx(k_full, C::kTileBytes);
      for (int x = 0; x < C::kBoxes; ++x)
        tma_load_4d(smem + C::kKOff + x * 16384, &tk, k_full, x * 64, kvh, sc.k0, b);
      for (; it_early < 2 && it_early < sc.n_iter; ++it_early) issue_iter(it_early);
    }
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // the next kernel on the stream may start as soon as every CTA of this one is running
  grid_launch_dependents();
  const uint32_t tmem = *tmem_slot;
  // TMEM slot h: S_h^T at 128h (then P^T / dS^T, 16 + 16 columns per key warpgroup), dP_h^T / dQ_h^T at 128h + 64
  const uint32_t T_DP = 64, T_DV = 256, T_DK = 384;

  if (warp >= kProducerWarp) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOther));
  if (warp == kProducerWarp) {
    // ========================== TMA producer ==========================
    if (lane == 0 && sc.n_iter > 0) {
      // (K and the first two iterations went out during the setup)
      int it = it_early;
      for (; it < sc.n_iter; ++it) {
        if (it >= 2 && !wait_parity(&qdo_empty[it & 1], ((it >> 1) & 1) ^ 1, abort_flag, p.status)) break;
        issue_iter(it);
      }
      // loads still in flight must land before shared memory goes away
      volatile int no_abort = 0;
      wait_parity(k_full, 0, &no_abort, p.status, 200000000ull);
      if (it > 0) wait_parity(v_full, 0, &no_abort, p.status, 200000000ull);  // V went out in the first pass
      for (int k = max(0, it - 2); k < it; ++k) {
        wait_parity(&q_full[k & 1], (k >> 1) & 1, &no_abort, p.status, 200000000ull);
        wait_parity(&do_full[k & 1], (k >> 1) & 1, &no_abort, p.status, 200000000ull);
      }
    }
  } else if (warp == kMmaWarp) {
    // ========================== MMA issuer ==========================
    // All 32 lanes run the loop and wait together; the issue calls elect one
    // lane (a lone issuing lane loses issue slots to the busy compute warps
    // on its scheduler and feeds the tensor core late).
    {
      // base descriptors (K-major: LBO unused; MN-major: 64-element blocks 16 KB apart)
      const uint64_t k_kmaj = sdesc_sw128(smem_u32(smem + C::kKOff), 16, 1024);
      const uint64_t k_mn = sdesc_sw128(smem_u32(smem + C::kKOff), 16384, 1024);
      const uint64_t v_kmaj = sdesc_sw128(smem_u32(smem + C::kVOff), 16, 1024);
      const uint64_t ds_mn = sdesc_sw128(smem_u32(smem + C::kDSOff), 16384, 1024);
      const uint64_t q_kmaj0 = sdesc_sw128(smem_u32(smem + C::kQOff), 16, 1024);
      const uint64_t q_mn0 = sdesc_sw128(smem_u32(smem + C::kQOff), 16384, 1024);
      const uint64_t do_kmaj0 = sdesc_sw128(smem_u32(smem + C::kDOOff), 16, 1024);
      const uint64_t do_mn0 = sdesc_sw128(smem_u32(smem + C::kDOOff), 16384, 1024);
      // S_h^T = K Q_h^T (M = keys, N = 64 queries, K = d; both K-major) into slot h. It
      // overwrites P_h^T of the previous tile, which that tile's dV product (issued
      // earlier) consumed.
      // descriptors as 32-bit halves: each operand step below is one 32-bit add
      const SDesc k_kmaj2 = sdesc_split(k_kmaj), k_mn2 = sdesc_split(k_mn), v_kmaj2 = sdesc_split(v_kmaj);
      const SDesc ds_mn2 = sdesc_split(ds_mn), q_kmaj2 = sdesc_split(q_kmaj0), q_mn2 = sdesc_split(q_mn0);
      const SDesc do_kmaj2 = sdesc_split(do_kmaj0), do_mn2 = sdesc_split(do_mn0);
      auto issue_s = [&](int h, int st) {
        const SDesc qd = sdesc_at(q_kmaj2, st * C::kTileBytes + h * 8192);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k / 4) * 16384 + (k % 4) * 32;
          umma_ss_warp(tmem + 128u * h, sdesc_at(k_kmaj2, off), sdesc_at(qd, off), C::kIdescS, k > 0 ? 1u : 0u);
        }
      };
      // dP_h^T = V dO_h^T into the second half of slot h (where dQ_h^T of the previous tile
      // was: the caller has waited for the drain)
      auto issue_dp = [&](int h, int st) {
        const SDesc dd = sdesc_at(do_kmaj2, st * C::kTileBytes + h * 8192);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k / 4) * 16384 + (k % 4) * 32;
          umma_ss_warp(tmem + 128u * h + T_DP, sdesc_at(v_kmaj2, off), sdesc_at(dd, off), C::kIdescS,
                       k > 0 ? 1u : 0u);
        }
      };
      // dQ_h^T = K^T dS_h^T (A = K read MN-major, B = dS_h^T from shared memory, MN-major)
      // into the second half of slot h.
      auto issue_dq = [&](int h) {
        const SDesc dsh = sdesc_at(ds_mn2, h * 16384);
#pragma unroll
        for (int k = 0; k < kBN / 16; ++k)
          umma_ss_warp(tmem + 128u * h + T_DP, sdesc_at(k_mn2, k * 2048), sdesc_at(dsh, k * 2048), C::kIdescQ,
                       k > 0 ? 1u : 0u);
      };
      // dV += P_h^T dO_h (A = P_h^T from TMEM, B = dO MN-major); dK += dS_h^T Q_h (A = dS_h^T
      // from TMEM, B = Q MN-major). Query step k (16 queries) of the half was formed by key
      // warpgroup k / 2, whose P^T / dS^T columns are [128h + 32 (k / 2), +16) /
      // [128h + 32 (k / 2) + 16, +16).
      auto issue_dkv = [&](int h, int st, bool first) {
        const SDesc q_mn = sdesc_at(q_mn2, st * C::kTileBytes + h * 8192);
        const SDesc do_mn = sdesc_at(do_mn2, st * C::kTileBytes + h * 8192);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          umma_ts_warp(tmem + T_DV, tmem + 128u * h + 32 * (k / 2) + 8 * (k % 2), sdesc_at(do_mn, k * 2048),
                       C::kIdescKV, (!first || k > 0) ? 1u : 0u);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          umma_ts_warp(tmem + T_DK, tmem + 128u * h + 32 * (k / 2) + 16 + 8 * (k % 2), sdesc_at(q_mn, k * 2048),
                       C::kIdescKV, (!first || k > 0) ? 1u : 0u);
      };
      // Issue order: S_0 dP_0 S_1 dP_1 (tile 0), then per tile i
      //   [P_0/dS_0 ready] dQ_0^T, dV, dK (i), S_0 dP_0 (tile i+1)
      //   [P_1/dS_1 ready] dQ_1^T, dV, dK (i), S_1 dP_1 (tile i+1)
      // dQ_h^T goes first, so that the drain reads it out of slot h while dV, dK and S_h run:
      // dP_h of the next tile waits for that read.
      // Slot 0 is free for tile i+1 once dV, dK (i) are issued and its dQ_0^T drained, so the
      // key warps' work on each half hides behind the tensor work of the other half.
      bool ok = sc.n_iter > 0 && warp_wait_parity(k_full, 0, abort_flag, p.status);
      if (ok) ok = warp_wait_parity(&q_full[0], 0, abort_flag, p.status);
      if (ok) {
        tc_fence_after();
        issue_s(0, 0);
      }
      if (ok) ok = warp_wait_parity(v_full, 0, abort_flag, p.status);
      if (ok) ok = warp_wait_parity(&do_full[0], 0, abort_flag, p.status);
      if (ok) {
        tc_fence_after();
        issue_dp(0, 0);
        umma_commit_warp(&sp_full[0]);
        issue_s(1, 0);
        issue_dp(1, 0);
        umma_commit_warp(&sp_full[1]);
      }
      int n_ready = 0;  // named-barrier phases joined, in (tile, half) order
      for (int it = 0; ok && it < sc.n_iter; ++it) {
        if (p.inject_abort == it + 1 && blockIdx.x == 0) {
          // test hook: behave exactly as if a wait of this warp had run out of time here
          if (lane == 0) {
            *abort_flag = 1;
            report_status(p.status, BEA_STATUS_TIMEOUT);
          }
          ok = false;
          break;
        }
        const int s = it & 1, s1 = s ^ 1;
        const uint32_t par1 = ((it + 1) >> 1) & 1;
        const bool more = it + 1 < sc.n_iter;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          named_bar_sync(kReadyBar + h, kReadyThreads);  // P_h^T / dS_h^T of tile it are written
          ++n_ready;
          tc_fence_after();
          issue_dq(h);
          umma_commit_warp(&dq_full[h]);
          issue_dkv(h, s, it == 0 && h == 0);
          if (h == 1) umma_commit_warp(&qdo_empty[s]);  // the last readers of stage s are issued
          if (more) {
            if (h == 0 && !(ok = warp_wait_parity(&q_full[s1], par1, abort_flag, p.status))) break;
            tc_fence_after();
            issue_s(h, s1);
            // dQ_h^T of tile i occupies the dP_h^T columns until the drain has read it
            if (!(ok = warp_wait_parity(&dq_empty[h], it & 1, abort_flag, p.status))) break;
            if (h == 0 && !(ok = warp_wait_parity(&do_full[s1], par1, abort_flag, p.status))) break;
            tc_fence_after();
            issue_dp(h, s1);
            umma_commit_warp(&sp_full[h]);
          }
        }
      }
      // After an abort, join the phases not reached, in the order the other side joins them.
      for (; n_ready < 2 * sc.n_iter; ++n_ready) named_bar_sync(kReadyBar + (n_ready & 1), kReadyThreads);
      if (ok && sc.n_iter > 0) umma_commit_warp(dkv_full);
      umma_commit_warp(mma_done);
      volatile int no_abort = 0;
      wait_parity(mma_done, 0, &no_abort, p.status, 200000000ull);
      __syncwarp();
    }
  }
  } else if (warp < kDrainWarp0) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsCompute));
    // ========================== P^T / dS^T (one thread per key) ==========================
    // Key warpgroup c (warps 4c..4c+3) takes queries [32c, 32c+32) of every half.
    const int c = warp / 4;
    const int j = threadIdx.x % 128;  // key row == TMEM lane
    const int kj = sc.k0 + j;
    const uint32_t lane_base = (uint32_t)((warp % 4) * 32) << 16;
    uint8_t* ds_row = smem + C::kDSOff + j * 128;
    bool ok = true;
    for (int it = 0; it < sc.n_iter; ++it) {
      const int s = it & 1;
      const int q0 = (sc.i_lo + it % nt) * kBM;
      const bool need_mask = bwd_tile_needs_mask(a, sc.k0, q0);
      const float* l2s = reinterpret_cast<const float*>(smem + C::kRowOff + s * 1024);
      const float* dds = l2s + kBM;
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        // S_h^T, dP_h^T of this tile; this also means every MMA issued before
        // them (the previous readers of the dS^T half and of P_h^T) has completed
        if (ok) ok = warp_wait_parity(&sp_full[h], it & 1, abort_flag, p.status);
        if (!ok) {
          named_bar_sync(kReadyBar + h, kReadyThreads);  // aborted: keep the phases matched
          continue;
        }
        tc_fence_after();
        const uint32_t slot = tmem + lane_base + 128u * h;
        uint32_t sv[32], pv[32];
        tmem_ld32(slot + 32 * c, sv);
        tmem_ld32(slot + T_DP + 32 * c, pv);
        tmem_wait_ld();
        reg_fence<32>(sv);
        reg_fence<32>(pv);
        if (need_mask)
          bwd_chunk<D, true>(sv, pv, l2s, dds, 2 * h + c, a, kj, q0, scale_log2, slot + 32 * c, ds_row, j);
        else
          bwd_chunk<D, false>(sv, pv, l2s, dds, 2 * h + c, a, kj, q0, scale_log2, slot + 32 * c, ds_row, j);
        tmem_wait_st();
        tc_fence_before();
        fence_proxy_async_smem();
        named_bar_sync(kReadyBar + h, kReadyThreads);
      }
    }
    // ---- dK / dV epilogue: key warpgroup 0 writes dV, warpgroup 1 writes dK ----
    // Through shared memory: each key thread writes 128 bytes of its row (32 fp32 values, or 64
    // converted to bf16; the 16-byte pieces of row j rotated by j & 7) into a staging chunk. With
    // accumulate, TMA adds the staged rows to dK / dV element by element at L2 (the 128-byte
    // swizzle of the gradient's tensor map); otherwise the warpgroup's 128 threads store the
    // chunk as 16-byte pieces, 8 threads per 128-byte row segment. The staging buffers are the Q
    // (dV) and dO (dK) stages, free once dkv_full says every MMA has completed (never loaded when
    // the CTA saw no query tile).
    if (ok && sc.n_iter > 0) ok = warp_wait_parity(dkv_full, 0, abort_flag, p.status);
    // a dependent launch (the next ring step) adds into dK / dV only after the launch before it is done
    grid_dependency_wait();
    {
      tc_fence_after();
      const bool have = sc.n_iter > 0;
      const float mul = c ? a.scale : 1.f;
      const bool f32 = c ? p.dk_is_f32 : p.dv_is_f32;
      const CUtensorMap* tmap = c ? &tdk : &tdv;
      const Seq4 dst = c ? p.dk : p.dv;
      const int piece = j & 7;
      uint8_t* stage = smem + (c ? C::kDOOff : C::kQOff);
      const uint32_t src_t = tmem + lane_base + (c ? T_DK : T_DV);
      const uint32_t ep_id = kEpiBar + c;
      if (f32 && p.accumulate) {
        // fp32 added to (a ring step after the first): D / 32 boxes of 32 columns staged, then
        // added element by element at L2 by TMA (no read of the old values here)
        if (ok) {
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t src[32];
            if (have) {
              tmem_ld32(src_t + c0, src);
              tmem_wait_ld();
              reg_fence<32>(src);
            } else {
#pragma unroll
              for (int e = 0; e < 32; ++e) src[e] = 0u;
            }
#pragma unroll
            for (int k = 0; k < 8; ++k)
              *reinterpret_cast<float4*>(stage + (c0 / 32) * 16384 + j * 128 + ((k ^ (j & 7)) * 16)) =
                  make_float4(__uint_as_float(src[4 * k]) * mul, __uint_as_float(src[4 * k + 1]) * mul,
                              __uint_as_float(src[4 * k + 2]) * mul, __uint_as_float(src[4 * k + 3]) * mul);
          }
          fence_proxy_async_smem();  // these writes are read by the TMA reductions below
        }
        named_bar_sync(ep_id, 128);
        if (ok && j == 0) {
          // (rows past the last key are not touched)
          for (int x = 0; x < D / 32; ++x) tma_reduce_add_4d(tmap, stage + x * 16384, 32 * x, kvh, sc.k0, b);
          bulk_commit_group();
          // (a launch that depends on this one programmatically also needs the additions done)
          if (p.pdl_next) bulk_wait_group_all();
          else bulk_wait_group_read_all();
        }
      } else if (f32) {
        // fp32 gradients written: 32 columns per pass
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          if (ok) {
            uint32_t src[32];
            if (have) {
              tmem_ld32(src_t + c0, src);
              tmem_wait_ld();
              reg_fence<32>(src);
            } else {
#pragma unroll
              for (int e = 0; e < 32; ++e) src[e] = 0u;
            }
#pragma unroll
            for (int k = 0; k < 8; ++k)
              *reinterpret_cast<float4*>(stage + j * 128 + ((k ^ (j & 7)) * 16)) =
                  make_float4(__uint_as_float(src[4 * k]) * mul, __uint_as_float(src[4 * k + 1]) * mul,
                              __uint_as_float(src[4 * k + 2]) * mul, __uint_as_float(src[4 * k + 3]) * mul);
          }
          named_bar_sync(ep_id, 128);
          if (ok) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const int row = (j >> 3) + 16 * k;
              const int key = sc.k0 + row;
              if (key >= a.lk) continue;  // ragged last key block
              const float4 v4 = *reinterpret_cast<const float4*>(stage + row * 128 + ((piece ^ (row & 7)) * 16));
              *reinterpret_cast<float4*>(reinterpret_cast<float*>(dst.ptr) + b * dst.sn + (int64_t)key * dst.sl +
                                         kvh * dst.sh + c0 + 4 * piece) = v4;
            }
          }
          named_bar_sync(ep_id, 128);
        }
      } else {
        // bf16 gradients: the row threads convert, 64 columns (128 bytes) per pass
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 64) {
          if (ok) {
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              uint32_t src[32];
              if (have) {
                tmem_ld32(src_t + c0 + 32 * hf, src);
                tmem_wait_ld();
                reg_fence<32>(src);
              } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) src[e] = 0u;
              }
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const int e = 8 * k;
                uint4 v4;
                v4.x = pack_bf16x2(__uint_as_float(src[e]) * mul, __uint_as_float(src[e + 1]) * mul);
                v4.y = pack_bf16x2(__uint_as_float(src[e + 2]) * mul, __uint_as_float(src[e + 3]) * mul);
                v4.z = pack_bf16x2(__uint_as_float(src[e + 4]) * mul, __uint_as_float(src[e + 5]) * mul);
                v4.w = pack_bf16x2(__uint_as_float(src[e + 6]) * mul, __uint_as_float(src[e + 7]) * mul);
                const int kk = 4 * hf + k;
                *reinterpret_cast<uint4*>(stage + j * 128 + ((kk ^ (j & 7)) * 16)) = v4;
              }
            }
          }
          named_bar_sync(ep_id, 128);
          if (ok) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const int row = (j >> 3) + 16 * k;
              const int key = sc.k0 + row;
              if (key >= a.lk) continue;
              *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(dst.ptr) + b * dst.sn +
                                        (int64_t)key * dst.sl + kvh * dst.sh + c0 + 8 * piece) =
                  *reinterpret_cast<const uint4*>(stage + row * 128 + ((piece ^ (row & 7)) * 16));
            }
          }
          named_bar_sync(ep_id, 128);
        }
      }
    }
  } else {
    static_assert(kRegsDrain <= kRegsLaunch, "the drain warpgroup gives registers back");
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsDrain));
    // ========================== dQ drain (one thread per head-dim index) ==========================
    const int dd = threadIdx.x - 32 * kDrainWarp0;  // dQ^T row == head-dim index == TMEM lane
    const uint32_t lane_base = (uint32_t)((warp % 4) * 32) << 16;
    const bool live = dd < D;  // for d = 64 the upper 64 lanes hold padding rows
    bool ok = true;
    for (int it = 0; ok && it < sc.n_iter; ++it) {
      const int hq = kvh * sc.g + it / nt;
      const int q0 = (sc.i_lo + it % nt) * kBM;
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        // accumulator layout [n h][lq_pad / 4][D][4]: four consecutive query rows per head-dim index
        float* dst = p.dq_acc + (((size_t)(b * a.h + hq) * p.lq_pad + q0 + 64 * h) / 4 * D + dd) * 4;
        if (ok) ok = warp_wait_parity(&dq_full[h], it & 1, abort_flag, p.status);
        if (!ok) break;
        tc_fence_after();
        uint32_t v[64];
        const uint32_t dq_t = tmem + lane_base + 128u * h + T_DP;
        tmem_ld32(dq_t, v);
        tmem_ld32(dq_t + 32, v + 32);
        tmem_wait_ld();
        reg_fence<64>(v);
        tc_fence_before();
        mbar_arrive(&dq_empty[h]);  // the slot is free for the next tile's dP_h^T
        if (live) {
          // a thread adds four query rows of its head-dim entry per instruction; the 32 lanes
          // of a warp cover 32 consecutive entries, one contiguous 512-byte span
#pragma unroll
          for (int u = 0; u < 16; ++u)
            red_add_v4(dst + (size_t)u * D * 4, __uint_as_float(v[4 * u]), __uint_as_float(v[4 * u + 1]),
                       __uint_as_float(v[4 * u + 2]), __uint_as_float(v[4 * u + 3]));
        }
      }
    }
  }

  // ---- teardown ----
  __syncwarp();  // lane-0-only roles rejoin their warp before the CTA barrier
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
cudaError_t launch_bwd_main_d(const BwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv, cudaStream_t s,
                              int* nlaunch) {
  using C = BwdCfg<D>;
  const AttnDims& a = p.a;
  const int nkb = (a.lk + kBN - 1) / kBN;
  const long long blocks = (long long)nkb * a.n * a.hkv;
  if (blocks == 0) return cudaSuccess;
  // Once per device context: allow the dynamic shared memory and read the
  // register count. The register split is only sound at exactly kRegsLaunch
  // registers per thread; refuse to launch otherwise (setmaxnreg.inc would
  // never return).
  static PerContext<int> regs_cache;
  int regs = 0;
  cudaError_t e = regs_cache.get(
      [](int* v) {
        cudaError_t r =
            cudaFuncSetAttribute(bwd_bf16_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (r != cudaSuccess) return r;
        cudaFuncAttributes fa;
        r = cudaFuncGetAttributes(&fa, bwd_bf16_kernel<D>);
        *v = fa.numRegs;
        return r;
      },
      &regs);
  if (e != cudaSuccess) return e;
  if (regs != kRegsLaunch) return cudaErrorInvalidConfiguration;
  const float scale_log2 = a.scale * 1.4426950408889634f;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.pdl ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, bwd_bf16_kernel<D>, tq, tk, tv, tdo, tdk, tdv, p, scale_log2);
  if (e != cudaSuccess) return e;
  *nlaunch += 1;
  return cudaGetLastError();
}

}  // namespace

// One wave of resident CTAs of a row kernel over `rows` rows of D values
// (`cache`: the kernel's wave size, looked up once per device context).
template <typename K>
cudaError_t row_grid(PerContext<int>& cache, K kern, int64_t rows, int d, unsigned* grid) {
  int cap = 0;
  cudaError_t e = wave_cap(cache, kern, kRowThreads, 0, &cap);
  if (e != cudaSuccess) return e;
  const int64_t rows_per_block = (int64_t)kRowThreads / (d / 8) * 2;
  const int64_t blocks = (rows + rows_per_block - 1) / rows_per_block;
  *grid = (unsigned)(blocks < cap ? blocks : cap);
  return cudaSuccess;
}

cudaError_t launch_bwd_prepare(const BwdParams& p, cudaStream_t s, int* nlaunch) {
  const int64_t rows = (int64_t)p.a.n * p.a.h * p.lq_pad;
  if (rows == 0) return cudaSuccess;
  static PerContext<int> cap128, cap64;
  const bool d128 = p.a.d == 128;
  auto kern = d128 ? bwd_preprocess_kernel<128> : bwd_preprocess_kernel<64>;
  unsigned grid = 0;
  cudaError_t e = row_grid(d128 ? cap128 : cap64, kern, rows, p.a.d, &grid);
  if (e != cudaSuccess) return e;
  kern<<<grid, kRowThreads, 0, s>>>(p);
  *nlaunch += 1;
  return cudaGetLastError();
}

cudaError_t launch_bwd_main(const BwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv, cudaStream_t s,
                            int* nlaunch) {
  if (p.a.d == 128) return launch_bwd_main_d<128>(p, tq, tk, tv, tdo, tdk, tdv, s, nlaunch);
  if (p.a.d == 64) return launch_bwd_main_d<64>(p, tq, tk, tv, tdo, tdk, tdv, s, nlaunch);
  return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_finish(const BwdParams& p, cudaStream_t s, int* nlaunch) {
  const int64_t groups = (int64_t)p.a.n * p.a.h * ((p.a.lq + 3) / 4);
  if (groups == 0) return cudaSuccess;
  static PerContext<int> cap128, cap64;
  const bool d128 = p.a.d == 128;
  auto kern = d128 ? bwd_convert_dq_kernel<128> : bwd_convert_dq_kernel<64>;
  unsigned grid = 0;
  // row_grid sizes a block for 2 x 256 / (d / 8) rows; a block of the convert takes 2 x 512 / d
  // groups of four rows per pass, a quarter as many
  cudaError_t e = row_grid(d128 ? cap128 : cap64, kern, 4 * groups, p.a.d, &grid);
  if (e != cudaSuccess) return e;
  kern<<<grid, kRowThreads, 0, s>>>(p);
  *nlaunch += 1;
  return cudaGetLastError();
}

cudaError_t launch_bwd_bf16(const BwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv, cudaStream_t s,
                            int* nlaunch) {
  if (p.a.d != 64 && p.a.d != 128) return cudaErrorInvalidValue;
  cudaError_t e;
  if ((e = launch_bwd_prepare(p, s, nlaunch)) != cudaSuccess) return e;
  if ((e = launch_bwd_main(p, tq, tk, tv, tdo, tdk, tdv, s, nlaunch)) != cudaSuccess) return e;
  return launch_bwd_finish(p, s, nlaunch);
}

}  // namespace bea
