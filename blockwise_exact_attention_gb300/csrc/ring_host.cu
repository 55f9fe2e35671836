// Ring attention replayed on one GPU, driven from the host in one call.
//
// flash_attn_jax flash_sharding.py, "Ring Forward": the sequence is split
// into C chunks; at ring step t the device holding query chunk i works on the
// K/V chunk that started on device i - t (ppermute sends i -> i+1), computes
// that block's (out, lse) and folds it into a running fp32 (out, lse) by the
// log-sum-exp merge; under a causal mask a block above the diagonal is
// skipped. "Ring Backward": every visible chunk pair is differentiated with
// the final out/lse of its query rows and the partial gradients are summed in
// fp32 (picotron context_parallel.py, RingAttentionFunc.backward, sends dK/dV
// around with K/V; on one GPU each pair is computed once and dK/dV of key
// chunk j simply accumulate in place).
//
// On one GPU the K/V rotation is a zero-copy chunk view, and the query chunks
// are independent: all chunk pairs of one ring step (query chunk i with key
// chunk (i - t) mod C, for every i) run as ONE launch over a batch of chunk
// views whose batch stride is one chunk. Pairs with i >= t share the key
// offset -t c, the wrapped ones (i < t) (C - t) c; a run whose key band is
// empty (under a causal mask every wrapped pair, under a window the pairs
// beyond it) is skipped. Consecutive launches are chained by programmatic
// dependent launch: step t+1's CTAs start on SMs that step t's tail leaves
// idle and run their main loop at once; each touches the accumulator (or dK,
// dV) only after the launch before it has completed.
#include <algorithm>
#include <cstring>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/bea.h"
#include "abi_internal.h"
#include "common.cuh"

namespace {

using bea::AttnDims;
using namespace bea::abi;

struct Run {
  int t;        // ring step
  int i0, j0;   // first query chunk, first key chunk
  int cnt;      // consecutive chunk pairs
  int64_t koff; // position of the key chunk's key 0 relative to the query chunk's query 0
};

// Whether any of c query rows sees any of c keys whose key 0 sits at query
// position koff: key j is visible to query r iff r - left <= j + koff <= r + right
// (an unbounded side is -1; causal forces right = 0), i.e. j - r lies in
// [-left - koff, right - koff], while j - r ranges over [-(c-1), c-1].
bool band_has_keys(int64_t c, int is_causal, int wl, int wr, int64_t koff) {
  const int right = is_causal ? 0 : wr;
  const int64_t lo = std::max<int64_t>(wl < 0 ? INT64_MIN / 4 : -(int64_t)wl - koff, -(c - 1));
  const int64_t hi = std::min<int64_t>(right < 0 ? INT64_MAX / 4 : (int64_t)right - koff, c - 1);
  return lo <= hi;
}

// The live runs of every ring step, in step order.
std::vector<Run> ring_runs(int C, int64_t c, int is_causal, int wl, int wr) {
  std::vector<Run> runs;
  for (int t = 0; t < C; ++t) {
    const Run cand[2] = {{t, t, 0, C - t, -(int64_t)t * c}, {t, 0, C - t, t, (int64_t)(C - t) * c}};
    for (const Run& r : cand)
      if (r.cnt > 0 && band_has_keys(c, is_causal, wl, wr, r.koff)) runs.push_back(r);
  }
  return runs;
}

// Chunks [f, f + cnt) of batch b of a [n, l, h, d] tensor as a [cnt, c, h, d] view.
bea_tensor seq_view(const bea_tensor* t, int64_t b, int64_t f, int64_t cnt, int64_t c) {
  bea_tensor v = *t;
  const int64_t es = t->dtype == BEA_BF16 ? 2 : 4;
  v.data = static_cast<char*>(t->data) + (b * t->stride[0] + f * c * t->stride[1]) * es;
  v.shape[0] = cnt;
  v.shape[1] = c;
  v.stride[0] = c * t->stride[1];
  return v;
}

// Chunks [f, f + cnt) of batch b of a [n, h, l] fp32 tensor as a [cnt, h, c] view.
bea_tensor lse_view(const bea_tensor* t, int64_t b, int64_t f, int64_t cnt, int64_t c) {
  bea_tensor v = *t;
  v.data = static_cast<float*>(t->data) + b * t->stride[0] + f * c;
  v.shape[0] = cnt;
  v.shape[2] = c;
  v.stride[0] = c;
  return v;
}

// Shared checks of the ring calls: bf16 q, k, v of one length l = C c.
int check_ring_qkv(const bea_tensor* q, const bea_tensor* k, const bea_tensor* v, float scale, int is_causal,
                   int wl, int wr, int n_chunks, AttnDims* a, int64_t* c) {
  int rc;
  const int64_t zero = 0;
  if ((rc = check_qkv(q, k, v, scale, is_causal, wl, wr, &zero, a))) return rc;
  if (q->dtype != BEA_BF16) return BEA_ERR_UNSUPPORTED;
  if (a->lq != a->lk) return BEA_ERR_SHAPE;
  if (n_chunks < 1 || a->lq % n_chunks != 0) return BEA_ERR_ARG;
  *c = a->lq / n_chunks;
  return BEA_OK;
}

}  // namespace

extern "C" {

int bea_ring_attention_fwd(const bea_tensor* q, const bea_tensor* k, const bea_tensor* v, const bea_tensor* out_acc,
                           const bea_tensor* lse, const bea_tensor* out_final, int n_chunks, float softmax_scale,
                           int is_causal, int window_left, int window_right, void* stream) {
  AttnDims a;
  int64_t c = 0;
  int rc;
  if ((rc = check_ring_qkv(q, k, v, softmax_scale, is_causal, window_left, window_right, n_chunks, &a, &c)))
    return rc;
  if ((rc = check_tensor(out_acc, 4))) return rc;
  if (!same_shape(out_acc, q)) return BEA_ERR_SHAPE;
  if (out_acc->dtype != BEA_F32) return BEA_ERR_DTYPE;
  if ((rc = check_lse(lse, a))) return rc;
  if (out_final != nullptr) {
    if ((rc = check_tensor(out_final, 4))) return rc;
    if (!same_shape(out_final, q)) return BEA_ERR_SHAPE;
    if (out_final->dtype != BEA_BF16) return BEA_ERR_DTYPE;
  }
  uint32_t* status = nullptr;
  if (a.n == 0 || a.h == 0 || a.lq == 0) return finish(cudaSuccess, 0);
  if ((rc = status_ptr_for_current_device(&status))) return rc;
  const int C = n_chunks;
  const std::vector<Run> runs = ring_runs(C, c, is_causal, window_left, window_right);
  // each query chunk's last live step: there its merged rows are also cast to bf16
  std::vector<int> last(C, -1);
  for (const Run& r : runs)
    for (int i = r.i0; i < r.i0 + r.cnt; ++i) last[i] = std::max(last[i], r.t);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int launches = 0;
  for (int64_t b = 0; b < a.n; ++b) {
    for (const Run& r : runs) {
      // split the run where needed so that each launch's final chunks form one range
      int u = 0;
      while (u < r.cnt) {
        int w = u;
        while (w < r.cnt && last[r.i0 + w] != r.t) ++w;  // non-final prefix
        const int f0 = w;
        while (w < r.cnt && last[r.i0 + w] == r.t) ++w;  // final range
        const int f1 = w;
        // extend with the non-final chunks that follow, up to the next final one
        while (w < r.cnt && last[r.i0 + w] != r.t) ++w;
        const int cnt = w - u;
        bea_tensor qv = seq_view(q, b, r.i0 + u, cnt, c), kv = seq_view(k, b, r.j0 + u, cnt, c),
                   vv = seq_view(v, b, r.j0 + u, cnt, c), av = seq_view(out_acc, b, r.i0 + u, cnt, c),
                   lv = lse_view(lse, b, r.i0 + u, cnt, c);
        bea_tensor fv{};
        if (out_final) fv = seq_view(out_final, b, r.i0 + u, cnt, c);
        AttnDims da;
        if ((rc = check_qkv(&qv, &kv, &vv, softmax_scale, is_causal, window_left, window_right, &r.koff, &da)))
          return rc;
        bea::FwdParams p;
        std::memset(&p, 0, sizeof(p));
        p.a = da;
        p.out = seq4(&av);
        p.out_is_f32 = 1;
        p.lse = lse3(&lv);
        p.merge = 1;
        p.merge_init = r.t == 0;
        p.fin = (out_final && f1 > f0) ? seq4(&fv) : bea::Seq4{nullptr, 0, 0, 0};
        p.fin_b0 = f0 - u;
        p.fin_b1 = f1 - u;
        p.pdl = launches > 0;  // the first launch waits for whatever came before it on the stream
        p.pdl_next = 1;
        p.status = status;
        p.inject_abort = take_inject_abort();
        CUtensorMap tq, tk, tv, tacc, tfin;
        if ((rc = make_seq_map(&qv, &tq)) || (rc = make_seq_map(&kv, &tk)) || (rc = make_seq_map(&vv, &tv)) ||
            (rc = make_acc_map(&av, &tacc)))
          return rc;
        if (p.fin.ptr != nullptr && (rc = make_seq_map(&fv, &tfin))) return rc;
        const cudaError_t e =
            bea::launch_fwd_bf16(p, tq, tk, tv, &tacc, p.fin.ptr != nullptr ? &tfin : nullptr, s, &launches);
        if (e != cudaSuccess) return finish(e, launches);
        u = w;
      }
    }
  }
  return finish(cudaSuccess, launches);
}

size_t bea_ring_attention_bwd_workspace_size(int64_t n, int64_t l, int64_t h, int64_t d, int n_chunks) {
  if (n < 0 || l < 0 || h < 0 || d < 0 || n_chunks < 1 || l % n_chunks != 0) return 0;
  (void)n;  // the batches run one after another and share the workspace
  return bwd_workspace_layout(n_chunks, l / n_chunks, h, d).total;
}

int bea_ring_attention_bwd(const bea_tensor* dout, const bea_tensor* q, const bea_tensor* k, const bea_tensor* v,
                           const bea_tensor* out, const bea_tensor* lse, const bea_tensor* dq, const bea_tensor* dk,
                           const bea_tensor* dv, int n_chunks, float softmax_scale, int is_causal, int window_left,
                           int window_right, void* workspace, size_t workspace_bytes, void* stream) {
  AttnDims a;
  int64_t c = 0;
  int rc;
  if ((rc = check_ring_qkv(q, k, v, softmax_scale, is_causal, window_left, window_right, n_chunks, &a, &c)))
    return rc;
  if ((rc = check_tensor(dout, 4)) || (rc = check_tensor(out, 4)) || (rc = check_tensor(dq, 4)) ||
      (rc = check_tensor(dk, 4)) || (rc = check_tensor(dv, 4)))
    return rc;
  if (!same_shape(dout, q) || !same_shape(out, q) || !same_shape(dq, q) || !same_shape(dk, k) ||
      !same_shape(dv, k))
    return BEA_ERR_SHAPE;
  if ((rc = check_lse(lse, a))) return rc;
  if (dout->dtype != BEA_BF16) return BEA_ERR_DTYPE;
  if (out->dtype != BEA_BF16 && out->dtype != BEA_F32) return BEA_ERR_DTYPE;
  if (dq->dtype != BEA_F32 || dk->dtype != BEA_F32 || dv->dtype != BEA_F32) return BEA_ERR_DTYPE;
  const int C = n_chunks;
  const BwdWorkspace w = bwd_workspace_layout(C, c, a.h, a.d);
  if ((rc = check_workspace(workspace, workspace_bytes, w))) return rc;
  if (a.n == 0 || a.h == 0 || a.lq == 0) return finish(cudaSuccess, 0);
  uint32_t* status = nullptr;
  if ((rc = status_ptr_for_current_device(&status))) return rc;
  const std::vector<Run> runs = ring_runs(C, c, is_causal, window_left, window_right);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int launches = 0;
  for (int64_t b = 0; b < a.n; ++b) {
    // D and L log2 e of every query row of batch b, its dQ accumulator zeroed
    bea_tensor dov = seq_view(dout, b, 0, C, c), ov = seq_view(out, b, 0, C, c), lv = lse_view(lse, b, 0, C, c);
    bea::BwdParams base;
    std::memset(&base, 0, sizeof(base));
    base.a = a;
    base.a.n = C;
    base.a.lq = base.a.lk = (int)c;
    base.dout = seq4(&dov);
    base.out = seq4(&ov);
    base.out_is_f32 = out->dtype == BEA_F32;
    base.lse = lse3(&lv);
    set_workspace(&base, workspace, w);
    base.status = status;
    cudaError_t e = bea::launch_bwd_prepare(base, s, &launches);
    if (e != cudaSuccess) return finish(e, launches);
    const size_t rows_per_chunk = (size_t)a.h * base.lq_pad;
    for (const Run& r : runs) {
      bea_tensor qv = seq_view(q, b, r.i0, r.cnt, c), kv = seq_view(k, b, r.j0, r.cnt, c),
                 vv = seq_view(v, b, r.j0, r.cnt, c), dov_r = seq_view(dout, b, r.i0, r.cnt, c),
                 dkv = seq_view(dk, b, r.j0, r.cnt, c), dvv = seq_view(dv, b, r.j0, r.cnt, c);
      bea::BwdParams p = base;
      if ((rc = check_qkv(&qv, &kv, &vv, softmax_scale, is_causal, window_left, window_right, &r.koff, &p.a)))
        return rc;
      p.dk = seq4(&dkv);
      p.dv = seq4(&dvv);
      p.dk_is_f32 = p.dv_is_f32 = 1;
      // step 0 is the diagonal, live for every chunk: it writes dK / dV, later steps add
      p.accumulate = r.t > 0;
      // this run's query chunks start i0 chunks into the workspace regions
      p.dq_acc = base.dq_acc + (size_t)r.i0 * rows_per_chunk * a.d;
      p.d_row = base.d_row + (size_t)r.i0 * rows_per_chunk;
      p.lse2 = base.lse2 + (size_t)r.i0 * rows_per_chunk;
      p.pdl = r.t > 0;  // step 0 follows the preprocess, whose results it reads at once
      p.pdl_next = 1;   // the next step adds into the same dK / dV as soon as this one is done
      p.inject_abort = take_inject_abort();
      CUtensorMap tq, tk, tv, tdo, tdk, tdv;
      if ((rc = make_seq_map(&qv, &tq)) || (rc = make_seq_map(&kv, &tk)) || (rc = make_seq_map(&vv, &tv)) ||
          (rc = make_seq_map(&dov_r, &tdo)) || (rc = make_grad_map(&dkv, &tdk)) || (rc = make_grad_map(&dvv, &tdv)))
        return rc;
      e = bea::launch_bwd_main(p, tq, tk, tv, tdo, tdk, tdv, s, &launches);
      if (e != cudaSuccess) return finish(e, launches);
    }
    // dQ = scale x accumulator for every query row of batch b
    bea_tensor dqv = seq_view(dq, b, 0, C, c);
    bea::BwdParams fp = base;
    fp.a.scale = softmax_scale;
    fp.dq = seq4(&dqv);
    fp.dq_is_f32 = 1;
    fp.accumulate = 0;
    e = bea::launch_bwd_finish(fp, s, &launches);
    if (e != cudaSuccess) return finish(e, launches);
  }
  return finish(cudaSuccess, launches);
}

}  // extern "C"
