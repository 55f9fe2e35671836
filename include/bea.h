/*
 * bea.h — C ABI of the blockwise exact attention library (libbea.so).
 *
 * Exact softmax attention computed block by block with an online softmax on
 * one GB300 (sm_103a), its backward pass recomputed from the per-row
 * log-sum-exp, and the log-sum-exp merge that folds a partial (out, lse) from
 * one K/V block into a running (out, lse) — the step ring attention repeats
 * once per K/V rotation.
 *
 * Tensors.
 *   Every tensor is described by a bea_tensor: a DEVICE pointer, a dtype, a
 *   rank, a shape and strides in ELEMENTS. The caller owns every buffer; the
 *   library never allocates, frees or keeps a pointer after a call returns.
 *   Sequence tensors are [n, l, h, d] (batch, sequence, heads, head dim) with
 *   the last dimension contiguous (stride 1), the base pointer 16-byte
 *   aligned and the other strides multiples of 16 bytes, so that chunk views
 *   of a longer sequence (an offset base pointer with the parent's strides)
 *   are accepted without a copy. The log-sum-exp is [n, h, l] fp32, natural
 *   log, softmax_scale included, with a contiguous last dimension and
 *   4-byte alignment
 *   (flash_attn_jax flash_sharding.py, sections "Sharding" and "Ring
 *   Forward": out [n,l,h,d], lse [n,h,l]).
 *
 * Grouped-query attention.
 *   q has h heads, k and v have h_kv heads with h % h_kv == 0; query head i
 *   reads K/V head i / (h / h_kv) (picotron context_parallel.py,
 *   RingAttention._repeat_kv), without expanding K/V in memory.
 *
 * Masks.
 *   is_causal: query i sees key j only if j <= i (picotron
 *   ring_attention_forward: the upper triangle is masked).
 *   window (left, right), -1 meaning unbounded: key j is visible to query i
 *   iff (left < 0 || j >= i - left) && (right < 0 || j <= i + right). The
 *   pages only ever pass (-1, -1); this inclusive reading is the library's.
 *   is_causal forces right = 0; right > 0 together with is_causal is an
 *   argument error.
 *   Positions: the window compares sequence positions, with key j at position
 *   j + key_offset relative to query i at position i. bea_flash_mha_fwd and
 *   bea_flash_mha_bwd use key_offset = lq - lk, which aligns the last query
 *   with the last key (bottom-right; 0 when lq == lk, the only case the pages
 *   use); the fused ring step and the K/V-block stage take it explicitly (a
 *   ring chunk pair passes the distance between its key and query chunks).
 *   Sequence lengths must be below 2^30.
 *   A query row that sees no key gets out = 0 and lse = -inf.
 *
 * Streams and errors.
 *   `stream` is a cudaStream_t (NULL = legacy default stream) of the current
 *   device. Every call validates all arguments on the host first and
 *   launches nothing when a check fails. Launches are asynchronous. Return
 *   values: BEA_OK or one of the negative BEA_ERR_* codes. No kernel traps:
 *   a kernel whose internal wait runs past its time limit ORs a flag into a
 *   per-device status word, which bea_get_device_status() reads.
 *
 * Thread safety: calls may come from several host threads; the library's
 * host state is a per-device cache filled on first use and the one-shot test
 * hook armed by bea_selftest_inject_abort (process-wide: the next launch from
 * any thread takes it).
 */
#ifndef BEA_H_
#define BEA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define BEA_VERSION 1

typedef enum bea_dtype {
  BEA_BF16 = 0, /* bfloat16 */
  BEA_F32 = 1   /* float32 */
} bea_dtype;

typedef enum bea_status {
  BEA_OK = 0,
  BEA_ERR_ARG = -1,         /* null pointer, bad scalar (scale, window, flags) */
  BEA_ERR_SHAPE = -2,       /* shapes inconsistent with each other */
  BEA_ERR_DTYPE = -3,       /* dtype not allowed for this argument */
  BEA_ERR_ALIGN = -4,       /* pointer or stride not 16-byte aligned, last dim not contiguous */
  BEA_ERR_UNSUPPORTED = -5, /* valid request this build does not implement (e.g. head dim) */
  BEA_ERR_CUDA = -6,        /* a CUDA runtime/driver call failed */
  BEA_ERR_TIMEOUT = -7,     /* a kernel wait ran past its limit (from bea_get_device_status) */
  BEA_ERR_WORKSPACE = -8    /* workspace missing, misaligned or too small */
} bea_status;

typedef struct bea_tensor {
  void* data;        /* device pointer to element [0,0,0,0] */
  int32_t dtype;     /* bea_dtype */
  int32_t ndim;      /* 4 for [n,l,h,d] tensors, 3 for [n,h,l] lse tensors */
  int64_t shape[4];  /* first ndim entries used */
  int64_t stride[4]; /* in elements; first ndim entries used */
} bea_tensor;

/*
 * Forward: out = softmax(softmax_scale * q k^T + mask) v and
 * lse = log(sum_j exp(softmax_scale * q.k_j + mask_j)) per query row
 * (picotron context_parallel.py, ring_attention_forward; flash_attn_jax
 * flash_sharding.py, the local fwd(q, k, v) of partition_fwd).
 *
 *   q    [n, lq, h, d]     bf16 or f32
 *   k, v [n, lk, h_kv, d]  same dtype as q
 *   out  [n, lq, h, d]     bf16 q: bf16 or f32; f32 q: f32 (written)
 *   lse  [n, h, lq]        f32 (written)
 *   softmax_scale must be finite and > 0.
 *   bf16: d must be 64 or 128; runs on the tcgen05 tensor cores with fp32
 *   accumulation (P is rounded to bf16 before P v).
 *   f32: 4 <= d <= 128, d % 4 == 0; runs an exact fp32 SIMT kernel.
 */
int bea_flash_mha_fwd(const bea_tensor* q, const bea_tensor* k, const bea_tensor* v, const bea_tensor* out,
                      const bea_tensor* lse, float softmax_scale, int is_causal, int window_left,
                      int window_right, void* stream);

/*
 * Fused ring step: the forward of one K/V block, folded straight into a
 * running fp32 accumulator by the log-sum-exp merge (flash_attn_jax
 * flash_sharding.py, "Ring Forward": the block's (out, lse) merged into the
 * carried (o, lse) once per ring step). Equal to bea_flash_mha_fwd into a
 * temporary followed by bea_ring_merge, without writing the block's output
 * to memory and without its rounding to bf16.
 *
 *   q, k, v    as for the forward, bf16 only (f32: BEA_ERR_UNSUPPORTED)
 *   out_acc    [n, lq, h, d] f32, read and written
 *   lse_acc    [n, h, lq]    f32, read and written
 *   out_final  NULL, or [n, lq, h, d] bf16: also receives the merged rows cast
 *              to bf16 (the last step of a ring)
 *   key_offset position of key 0 relative to query 0 (see Masks); |key_offset|
 *              <= 2^30
 * Per row, with La the accumulator's and L the block's log-sum-exp:
 * M = max(La, L); if M == -inf the row is left unchanged; otherwise
 * L' = M + log1p(exp(min(La, L) - M)), out_acc <- exp(La - L') out_acc +
 * exp(L - L') O_block, lse_acc <- L'.
 */
int bea_flash_mha_fwd_merge(const bea_tensor* q, const bea_tensor* k, const bea_tensor* v, const bea_tensor* out_acc,
                            const bea_tensor* lse_acc, const bea_tensor* out_final, float softmax_scale, int is_causal,
                            int window_left, int window_right, int64_t key_offset, void* stream);

/*
 * Bytes of device workspace bea_flash_mha_bwd needs for q of shape
 * [n, lq, h, d] (an fp32 dQ accumulator plus two fp32 values per row).
 */
size_t bea_flash_mha_bwd_workspace_size(int64_t n, int64_t lq, int64_t h, int64_t d);

/*
 * Backward from the GIVEN out and lse (picotron context_parallel.py,
 * ring_attention_backward, Steps 1-6):
 *   P = exp(softmax_scale * q k^T - lse) (masked entries 0), dV = P^T dO,
 *   dP = dO v^T, D = rowsum(dO * out), dS = P * (dP - D),
 *   dQ = softmax_scale * dS k, dK = softmax_scale * dS^T q,
 * with dK, dV summed over the query heads of each K/V head. Using the final
 * out/lse of the full row (not a chunk's) is what lets ring chunk pairs add
 * their partial gradients (flash_sharding.py, "Ring Backward").
 *
 *   dout        [n, lq, h, d]    q's dtype
 *   q, k, v     as for the forward
 *   out         [n, lq, h, d]    q's dtype, or f32
 *   lse         [n, h, lq]       f32
 *   dq          [n, lq, h, d]    q's dtype or f32 (written)
 *   dk, dv      [n, lk, h_kv, d] q's dtype or f32 (written)
 *   accumulate  0: dq/dk/dv are overwritten; 1: the gradients are ADDED to
 *               dq/dk/dv, which must then all be f32 (ring chunk pairs).
 *   workspace   device buffer of at least bea_flash_mha_bwd_workspace_size()
 *               bytes, 256-byte aligned, owned by the caller, contents on
 *               entry irrelevant; calls that may run concurrently need
 *               separate workspaces.
 */
int bea_flash_mha_bwd(const bea_tensor* dout, const bea_tensor* q, const bea_tensor* k, const bea_tensor* v,
                      const bea_tensor* out, const bea_tensor* lse, const bea_tensor* dq, const bea_tensor* dk,
                      const bea_tensor* dv, float softmax_scale, int is_causal, int window_left,
                      int window_right, int accumulate, void* workspace, size_t workspace_bytes,
                      void* stream);

/*
 * The bf16 backward in its three stages, for a caller that accumulates the dQ
 * of one set of query rows over several K/V blocks: the backward of ring
 * attention, where each query chunk meets every visible K/V chunk once
 * (flash_attn_jax flash_sharding.py, "Ring Backward": dq accumulates over the
 * steps; picotron context_parallel.py, RingAttentionFunc.backward). Running
 * prepare once, kv_block once per K/V block, then finish once keeps dQ in
 * fp32 in the workspace across blocks and computes D once per query chunk.
 * bea_flash_mha_bwd on bf16 inputs is exactly prepare + kv_block + finish.
 *
 * All three take the same workspace, sized by
 * bea_flash_mha_bwd_workspace_size(n, lq, h, d) of the query-side tensors,
 * 256-byte aligned. Between prepare and finish it holds the state of the
 * accumulation; calls on it must be ordered on one stream. Only bf16 q/k/v
 * are supported (f32 inputs: BEA_ERR_UNSUPPORTED; use bea_flash_mha_bwd).
 *
 * prepare  (Step "D = rowsum(dO * O)"): dout [n, lq, h, d] bf16;
 *          out same shape, bf16 or f32; lse [n, h, lq] f32. Writes D and
 *          lse * log2(e) per row and zeroes the fp32 dQ accumulator.
 * kv_block (Steps P, dV, dP, dS, dK, and dQ's sum over these keys): dout,
 *          q [n, lq, h, d] bf16, k, v [n, lk, h_kv, d] bf16; dk, dv
 *          [n, lk, h_kv, d] bf16 or f32, written (accumulate 0) or added to
 *          (accumulate 1, both f32). Adds this block's dS k into the
 *          accumulator. The mask arguments are those of bea_flash_mha_bwd,
 *          with key_offset the position of this block's key 0 relative to
 *          query 0 (see Masks).
 * finish   dq [n, lq, h, d] bf16 or f32: dq = softmax_scale * accumulator,
 *          written (accumulate 0) or added to an f32 dq (accumulate 1).
 */
int bea_flash_mha_bwd_prepare(const bea_tensor* dout, const bea_tensor* out, const bea_tensor* lse,
                              void* workspace, size_t workspace_bytes, void* stream);
int bea_flash_mha_bwd_kv_block(const bea_tensor* dout, const bea_tensor* q, const bea_tensor* k,
                               const bea_tensor* v, const bea_tensor* dk, const bea_tensor* dv,
                               float softmax_scale, int is_causal, int window_left, int window_right,
                               int64_t key_offset, int accumulate, void* workspace, size_t workspace_bytes,
                               void* stream);
int bea_flash_mha_bwd_finish(const bea_tensor* dq, float softmax_scale, int accumulate, void* workspace,
                             size_t workspace_bytes, void* stream);

/*
 * Ring attention replayed on one GPU in one call (flash_attn_jax
 * flash_sharding.py, "Ring Forward"): the sequence is split into n_chunks
 * equal chunks; at ring step t query chunk i meets the K/V chunk
 * (i - t) mod n_chunks (the chunk that started on device i - t when K/V move
 * i -> i+1), and every live pair's (out, lse) is folded into the running
 * fp32 (out_acc, lse) by the log-sum-exp merge of bea_flash_mha_fwd_merge.
 * Pairs whose keys are all masked (under is_causal every pair above the
 * diagonal; under a window every pair beyond it) are skipped; the window
 * compares sequence positions, so a chunk pair sees exactly the keys the
 * single call would. All pairs of one ring step run as one launch over chunk
 * views; the launches of one call are chained on `stream` by programmatic
 * dependent launch (a step starts computing while the step before finishes
 * and merges only after it has).
 *
 *   q          [n, l, h, d] bf16; k, v [n, l, h_kv, d] bf16 (same l)
 *   out_acc    [n, l, h, d] f32, written: the result (the ring's accumulator)
 *   lse        [n, h, l] f32, written
 *   out_final  NULL, or [n, l, h, d] bf16: also receives the result cast to
 *              bf16, written at each query chunk's last live step
 *   n_chunks   >= 1, dividing l
 * Errors as for bea_flash_mha_fwd; l % n_chunks != 0 is BEA_ERR_ARG, f32
 * inputs BEA_ERR_UNSUPPORTED.
 */
int bea_ring_attention_fwd(const bea_tensor* q, const bea_tensor* k, const bea_tensor* v, const bea_tensor* out_acc,
                           const bea_tensor* lse, const bea_tensor* out_final, int n_chunks, float softmax_scale,
                           int is_causal, int window_left, int window_right, void* stream);

/*
 * Workspace bytes of bea_ring_attention_bwd for q [n, l, h, d] split into
 * n_chunks chunks (0 when n_chunks does not divide l).
 */
size_t bea_ring_attention_bwd_workspace_size(int64_t n, int64_t l, int64_t h, int64_t d, int n_chunks);

/*
 * Backward of ring attention on one GPU in one call (flash_attn_jax
 * flash_sharding.py, "Ring Backward"; picotron context_parallel.py,
 * RingAttentionFunc.backward): every live chunk pair (same schedule and masks
 * as bea_ring_attention_fwd) is differentiated once with the FINAL out/lse of
 * its query rows, and the partial gradients are summed in fp32: dQ of a query
 * chunk in the workspace accumulator, dK/dV of a key chunk in place. All
 * pairs of one ring step run as one launch; per batch row: one preprocess,
 * one launch per live step, one dQ conversion.
 *
 *   dout, q    [n, l, h, d] bf16; k, v [n, l, h_kv, d] bf16
 *   out        [n, l, h, d] bf16 or f32; lse [n, h, l] f32
 *   dq         [n, l, h, d] f32, written; dk, dv [n, l, h_kv, d] f32, written
 *   workspace  >= bea_ring_attention_bwd_workspace_size() bytes, 256-byte
 *              aligned, caller-owned, contents on entry irrelevant
 */
int bea_ring_attention_bwd(const bea_tensor* dout, const bea_tensor* q, const bea_tensor* k, const bea_tensor* v,
                           const bea_tensor* out, const bea_tensor* lse, const bea_tensor* dq, const bea_tensor* dk,
                           const bea_tensor* dv, int n_chunks, float softmax_scale, int is_causal, int window_left,
                           int window_right, void* workspace, size_t workspace_bytes, void* stream);

/*
 * bea_flash_mha_bwd without a caller-supplied workspace. (The pages have no
 * counterpart; this is a library convenience.)
 *
 * For callers that cannot allocate device memory: code that reaches the
 * library only through a C function pointer from another language or plugin
 * host that hands over just the tensors it owns, or a long-running serving
 * loop that must not call cudaMalloc (which can synchronise the device). The
 * workspace comes from a fixed array of BEA_NOALLOC_BWD_SCRATCH_BYTES in the
 * library's own device memory; every GPU that loads the library holds that
 * array until the process exits. This call allocates nothing.
 *
 * Arguments and results are those of bea_flash_mha_bwd, checked in the same
 * order and with the same error codes. Only a call that passes those checks
 * and whose workspace (bea_flash_mha_bwd_workspace_size, computed without
 * overflow) exceeds the array returns BEA_ERR_WORKSPACE, before anything is
 * launched.
 *
 * The first call in a device's context looks up the array's device address
 * (cudaGetSymbolAddress) with that device current and caches it for that
 * context; a new context on the device (e.g. after cudaDeviceReset) looks it
 * up again on its first call. Make that first call before any stream
 * capture. All calls on a device share the one
 * array, so two calls whose kernels may overlap on the GPU (different
 * streams, or several host threads) race on it: order them on one stream.
 * The array keeps the last call's contents; each call rewrites all of it
 * that it reads, so nothing needs clearing between calls.
 */
#define BEA_NOALLOC_BWD_SCRATCH_BYTES (64u * 1024u * 1024u)
int bea_flash_mha_bwd_noalloc(const bea_tensor* dout, const bea_tensor* q, const bea_tensor* k,
                              const bea_tensor* v, const bea_tensor* out, const bea_tensor* lse,
                              const bea_tensor* dq, const bea_tensor* dk, const bea_tensor* dv,
                              float softmax_scale, int is_causal, int window_left, int window_right,
                              int accumulate, void* stream);

/*
 * Log-sum-exp merge, in place on the accumulator (flash_attn_jax
 * flash_sharding.py, "Ring Forward"; the same fold as picotron
 * update_out_and_lse in its sigmoid form). Per row r = (b, i, head):
 *   M = max(La, Lb); if M == -inf the row is left unchanged; otherwise
 *   L = M + log1p(exp(min(La, Lb) - M)), Oa <- exp(La - L) Oa + exp(Lb - L) Ob,
 *   La <- L.
 *
 *   out_acc   [n, l, h, d] f32 (read and written)
 *   lse_acc   [n, h, l]    f32 (read and written)
 *   out_blk   [n, l, h, d] bf16 or f32
 *   lse_blk   [n, h, l]    f32
 *   out_final NULL, or [n, l, h, d] bf16: also receives the merged rows cast
 *             to bf16 (the last step of a ring).
 *   d must be 16, 32, 64 or 128.
 */
int bea_ring_merge(const bea_tensor* out_acc, const bea_tensor* lse_acc, const bea_tensor* out_blk,
                   const bea_tensor* lse_blk, const bea_tensor* out_final, void* stream);

/*
 * Synchronises `stream`, reads the device status word of the current device
 * and clears it. Returns BEA_OK, BEA_ERR_TIMEOUT if any kernel since the last
 * read gave up a wait, BEA_ERR_UNSUPPORTED if a kernel met a configuration it
 * cannot run, or BEA_ERR_CUDA.
 */
int bea_get_device_status(void* stream);

/* Static English text for a status code. */
const char* bea_status_string(int code);

/* BEA_VERSION of the built library. */
int bea_version(void);

/*
 * Failure-detection self test: launches one CTA whose thread waits on an
 * mbarrier that nothing arrives on, with a limit of `limit_us` microseconds
 * (1..2000000). The wait gives up, the kernel returns normally and the
 * status word reads BEA_ERR_TIMEOUT afterwards. No trap, no fault.
 */
int bea_selftest_wait_timeout(int limit_us, void* stream);

/*
 * Failure-detection self test of the attention kernels. Arms a one-shot
 * injection: the next bf16 forward or backward main-kernel launch of this
 * process (bea_flash_mha_fwd, _fwd_merge, _bwd, _bwd_kv_block, _bwd_noalloc)
 * behaves in its first CTA as if a wait of the MMA-issuing warp had run out of
 * time at tile (forward) or iteration (backward) `tile`. That CTA raises its
 * abort flag and records BEA_STATUS_TIMEOUT. Every other role of the CTA then
 * leaves its loop on its next wait, in-flight copies land, TMEM is freed and
 * the kernel returns normally. The outputs of that launch are undefined; the
 * status word reads BEA_ERR_TIMEOUT afterwards. `tile` = -1 disarms.
 * Returns BEA_ERR_ARG for tile < -1. Nothing traps or faults.
 */
int bea_selftest_inject_abort(int tile);

/* Number of kernels the last successful call on this host thread launched. */
int bea_last_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* BEA_H_ */
