// Parameter blocks shared by the host dispatch (api.cu) and the kernels, and
// the kernel launchers each translation unit exports.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace bea {

// A [n, l, h, d] tensor with a contiguous last dimension (strides in elements).
struct Seq4 {
  void* ptr;
  int64_t sn, sl, sh;
};

// A [n, h, l] fp32 tensor with a contiguous last dimension.
struct Lse3 {
  float* ptr;
  int64_t sn, sh;
};

// Bound of the visible band meaning "no limit"; sequence lengths stay below it.
constexpr int kUnbounded = 1 << 30;

struct AttnDims {
  int n, lq, lk, h, hkv, d;
  // Visible band, in key indices relative to the query index: key j is visible
  // to query i iff i - wl <= j <= i + wr. The host folds the caller's window,
  // the causal flag and the key position offset into these signed bounds
  // (kUnbounded: no limit on that side).
  int wl, wr;
  float scale;
};

__host__ __device__ __forceinline__ bool key_visible(int i, int j, int wl, int wr) {
  return j >= i - wl && j <= i + wr;
}

// ---- ring merge --------------------------------------------------------------
struct MergeParams {
  int n, l, h, d;
  Seq4 acc;  // f32
  Lse3 lse_acc;
  Seq4 blk;  // bf16 or f32
  int blk_is_f32;
  Lse3 lse_blk;
  Seq4 fin;  // bf16, ptr may be null
};
cudaError_t launch_ring_merge(const MergeParams& p, cudaStream_t s, int* nlaunch);

// ---- fp32 SIMT path ------------------------------------------------------------
struct F32FwdParams {
  AttnDims a;
  Seq4 q, k, v, out;  // all f32
  Lse3 lse;
};
cudaError_t launch_fwd_f32(const F32FwdParams& p, cudaStream_t s, int* nlaunch);

struct F32BwdParams {
  AttnDims a;
  Seq4 dout, q, k, v, out, dq, dk, dv;  // all f32
  Lse3 lse;
  float* D;  // workspace [n, h, lq]
  int accumulate;
};
cudaError_t launch_bwd_f32(const F32BwdParams& p, cudaStream_t s, int* nlaunch);

// ---- bf16 tensor-core path -------------------------------------------------------
struct FwdParams {
  AttnDims a;
  Seq4 out;  // merge: the fp32 accumulator (read and written)
  int out_is_f32;
  Lse3 lse;  // merge: the accumulator's log-sum-exp (read and written)
  int merge;  // fold the block into (out, lse) instead of writing it
  int merge_init;  // merge only: the accumulator holds nothing yet ((0, -inf)): write the block, read nothing
  Seq4 fin;   // merge only: bf16 copy of the merged rows, ptr may be null
  int fin_b0, fin_b1;  // merge only: fin is written for batch indices [fin_b0, fin_b1) only
  int pdl;    // launch with programmatic stream serialisation (see grid_dependency_wait)
  int pdl_next;  // the next launch on the stream depends on this one programmatically
  uint32_t* status;
  int inject_abort;  // test hook, 0 = off: CTA 0's MMA warp aborts at tile inject_abort - 1
};
// Tensor maps are built by the caller (api.cu) over q, k, v; for the fused ring step (merge) also
// over the fp32 accumulator (tacc, 32-column boxes) and, when fin is set, the bf16 final copy
// (tfin, 64-column boxes). The plain forward takes no tacc, and tfin over its output when that
// is bf16.
cudaError_t launch_fwd_bf16(const FwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap* tacc, const CUtensorMap* tfin, cudaStream_t s,
                            int* nlaunch);

struct BwdParams {
  AttnDims a;
  Seq4 dout, out, dq, dk, dv;
  int out_is_f32, dq_is_f32, dk_is_f32, dv_is_f32;
  Lse3 lse;
  int accumulate;
  float* dq_acc;  // workspace: fp32 dQ partial sums, [n h][lq_pad / 4][d][4] (four query rows interleaved)
  float* d_row;   // workspace: [n, h, lq_pad] D = rowsum(dO * O)
  float* lse2;    // workspace: [n, h, lq_pad] lse * log2(e), +inf for rows without keys / padding
  int lq_pad;
  int pdl;        // launch with programmatic stream serialisation (see grid_dependency_wait)
  int pdl_next;   // the next launch on the stream depends on this one programmatically
  uint32_t* status;
  int inject_abort;  // test hook, 0 = off: CTA 0's MMA warp aborts at iteration inject_abort - 1
};
// Tensor maps over q, k, v, dout and the gradients dk, dv (make_grad_map: bf16 64-column or fp32
// 32-column boxes of 128 rows) are built by the caller (api.cu).
// launch_bwd_bf16 = prepare (D, lse*log2e, zeroed dQ accumulator) + main
// (dK, dV, dQ accumulation) + finish (dQ = scale * accumulator); the stages
// are also exported separately for callers that accumulate dQ over several
// K/V blocks.
cudaError_t launch_bwd_bf16(const BwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdk,
                            const CUtensorMap& tdv, cudaStream_t s, int* nlaunch);
cudaError_t launch_bwd_prepare(const BwdParams& p, cudaStream_t s, int* nlaunch);
cudaError_t launch_bwd_main(const BwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdk,
                            const CUtensorMap& tdv, cudaStream_t s, int* nlaunch);
cudaError_t launch_bwd_finish(const BwdParams& p, cudaStream_t s, int* nlaunch);

cudaError_t launch_selftest_wait_timeout(uint32_t* status, uint64_t limit_ns, cudaStream_t s);

}  // namespace bea
