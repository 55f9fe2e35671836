// Blockwise exact attention forward on sm_103a tensor cores (bf16 in, fp32
// accumulation), emitting O and the per-row log-sum-exp L.
//
// What it computes is picotron context_parallel.py, ring_attention_forward
// (S = scale Q K^T, causal/window mask, softmax, L, P V), reorganised as the
// blockwise online softmax: K/V are visited one 128-key tile at a time and
// each query row keeps a running max m and running sum l, so S never leaves
// the SM. The result is the same up to rounding order; P is rounded to bf16
// before the P V product.
//
// One CTA owns 256 query rows (two 128-row subtiles) of one (batch, head):
//   warp 8      TMA producer: Q once, then K_j into an NS-stage ring;
//   warp 10     TMA producer of V_j, on its own ring (V_j is released after
//               P V, K_j after the S of tile j);
//   warp 9      MMA issuer (the whole warp runs the loop, one elected lane
//               issues): S_t = Q_t K_j^T into TMEM (both operands in
//               shared memory), O_t += P_t V_j with P_t read from TMEM;
//   warps 0-3   softmax for subtile 0, warps 4-7 for subtile 1: one thread
//               per query row (TMEM lane), online softmax, P written back to
//               TMEM over S as packed bf16, O rescaled in TMEM only when the
//               row max grows by more than 2^8, and the final epilogue.
//   warp 11     idle.
// The epilogue stages O in shared memory and writes it out (TMA tensor stores
// for a bf16 result). The fused ring step (kMerge) stages the caller's fp32
// accumulator rows by TMA in the K/V stages as the last tiles free them,
// folds the block into them in place by the log-sum-exp merge, and writes
// them back by TMA.
// The MMA issue order S_0(j), S_1(j), PV_0(j), S_0(j+1), PV_1(j), S_1(j+1),
// ... lets each softmax group work while the tensor core serves the other
// subtile. Tiles outside the causal/window band are never loaded or computed;
// only tiles that straddle the band edge (or the ragged end of K) are masked
// element by element.
//
// TMEM (512 columns): S_0 [0,128), S_1 [128,256), O_0 [256,256+D),
// O_1 [384,384+D); P_t occupies the first 64 columns of S_t. S_t(j+1)
// overwrites P_t(j) only after PV_t(j), which the single issuing thread
// placed before it in the MMA pipeline.
#include <cuda_bf16.h>

#include <cstring>

#include "common.cuh"
#include "launch_cache.cuh"
#include "ptx.cuh"

namespace bea {
namespace {

constexpr int kBlockM = 128;  // rows per subtile (= TMEM lanes)
constexpr int kBlockN = 128;  // keys per tile
constexpr int kSub = 2;       // subtiles per CTA
constexpr int kThreads = 384;  // 3 warpgroups
// Register split: launched at kRegsLaunch per thread (65536 / 384 rounded
// down to 8); the softmax warpgroups raise to kRegsSoftmax and the
// producer/MMA warpgroup lowers to kRegsOther, which sums to the launch:
// 256 * 200 + 128 * 104 = 384 * 168.
constexpr int kRegsLaunch = 168;
constexpr int kRegsSoftmax = 200;
constexpr int kRegsOther = 104;
static_assert(256 * kRegsSoftmax + 128 * kRegsOther == kThreads * kRegsLaunch, "register split");
constexpr int kProducerWarp = 8;  // Q and K loads
constexpr int kMmaWarp = 9;
constexpr int kVLoadWarp = 10;    // V loads
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when the max grows by > 2^8
// "P_t of tile j is in TMEM" goes from softmax warpgroup t to the MMA warp over
// hardware named barrier kPReadyBar + t: one phase per tile, 128 softmax threads
// plus the MMA warp. A named barrier has no time limit, so the phases are kept
// matched on every path:
//  * the MMA warp joins once per tile of subtile t; after an abort it still
//    joins, without work, for each tile it has not reached;
//  * each softmax warp joins once per tile of its range, with or without work.
//  * Every join waits for the phase to complete (barrier.sync, never a bare
//    arrive), so no warp can join phase j+1 while phase j is still open: a
//    bare arrive followed by an aborting warp's next join could land both in
//    one phase and leave a later phase short of arrivals. The wait costs the
//    softmax nothing, as its next step waits for S_t(j+1), which the MMA warp
//    issues only after phase j.
constexpr uint32_t kPReadyBar = 1;
constexpr uint32_t kPReadyThreads = 128 + 32;
// Epilogue of subtile t: its 128 softmax threads hand the staged O chunk to one
// another over named barrier kEpiBar + t (every thread of the subtile joins
// every phase, with or without work).
constexpr uint32_t kEpiBar = 3;

template <int D>
struct FwdCfg {
  static constexpr int kBoxes = D / 64;          // 64-column (128-byte) TMA boxes per row
  static constexpr int kTileBytes = 128 * D * 2;  // one 128-row bf16 tile
  static constexpr int kStages = (D == 128) ? 2 : 4;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kSub * kTileBytes;
  static constexpr int kVOff = kKOff + kStages * kTileBytes;
  static constexpr int kBarOff = kVOff + kStages * kTileBytes;
  static constexpr int kNumBars = 1 + 4 * kStages + 2 * kSub + 1 + kSub * 2;
  static constexpr int kSmemBytes = kBarOff + kNumBars * 8 + 16 /*tmem slot + abort*/ + 1024 /*align slack*/;
  // Fused ring step: subtile t's fp32 accumulator rows (128 x D, as D/32 swizzled 32-column
  // boxes of 16 KB) are staged in the K stages (t = 0) or the V stages (t = 1) once those are
  // free; the bf16 final copy in the subtile's Q tile.
  static constexpr int kBox = 16384;
  static constexpr int kAccBoxes = D / 32;
  static constexpr int kBoxesPerStage = kTileBytes / kBox;
  static constexpr int kAccStages = kAccBoxes / kBoxesPerStage;  // stages one subtile's accumulator takes
  static_assert(kAccStages * kBoxesPerStage == kAccBoxes && kAccStages <= kStages && kAccStages <= 2,
                "a subtile's accumulator fills whole K (V) stages");
  static constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false, false);
  static constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, false, true);
  static constexpr uint32_t kVLbo = 64 * 128 * 2;  // byte distance of 64-column V blocks
};

struct Sched {
  int lo[kSub], hi[kSub];  // K tile range per subtile (empty if lo >= hi)
  int lo_all, hi_all;
  int q0;
};

__device__ __forceinline__ void tile_range(const AttnDims& a, int qs, int& lo, int& hi) {
  lo = hi = 0;
  if (qs >= a.lq) return;
  const int qe = min(qs + kBlockM, a.lq);
  const int kmin = (int)max(0LL, (long long)qs - a.wl);
  const int kmax = (int)min((long long)a.lk, (long long)qe + a.wr);
  if (kmax <= kmin) return;
  lo = kmin / kBlockN;
  hi = (kmax + kBlockN - 1) / kBlockN;
}

// Does tile j need per-element masking for subtile rows [qs, qs+128)?
__device__ __forceinline__ bool tile_needs_mask(const AttnDims& a, int qs, int j) {
  const int k0 = j * kBlockN, k1 = k0 + kBlockN - 1;
  if (k1 >= a.lk) return true;
  const int q1 = qs + kBlockM - 1;
  if ((long long)k0 < (long long)q1 - a.wl) return true;
  if ((long long)k1 > (long long)qs + a.wr) return true;
  return false;
}

template <int D, bool kMerge>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_bf16_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tacc,
                    const __grid_constant__ CUtensorMap tfin, const FwdParams p, float scale_log2) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* v_full = k_full + C::kStages;
  uint64_t* k_empty = v_full + C::kStages;  // K and V rings are released separately:
  uint64_t* v_empty = k_empty + C::kStages; // K_j after the S of tile j, V_j after its P V
  uint64_t* s_full = v_empty + C::kStages;
  uint64_t* o_full = s_full + kSub;
  uint64_t* mma_done = o_full + kSub;
  // fused ring step: [t * kAccStages + i]: stage i of subtile t's accumulator has landed
  uint64_t* acc_full = mma_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const AttnDims& a = p.a;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  // ---- work decomposition: longest (latest) query blocks first ----
  const int nqb = (a.lq + kSub * kBlockM - 1) / (kSub * kBlockM);
  const int bh_count = a.n * a.h;
  // When the band covers every (query, key) pair (no mask, or a ring step's chunk pair that
  // lies wholly inside it) every CTA has the same work. With one query head per K/V head the
  // CTAs are then taken head by head, so that the ones running together stream one head's K/V
  // tiles from L2 (measured: 32k d=64 full attention -2%; the 16k ring's full chunk pairs, run
  // as a batch of 7 chunks x 16 heads, would otherwise spread ~150 heads' K/V over L2).
  // Under a causal or window band the batches go one after another and, within one, the
  // latest (longest) query blocks first, the heads fastest.
  const bool full_band = a.wl >= a.lq - 1 && a.wr >= a.lk - 1;
  const bool head_major = full_band && a.h == a.hkv;
  const int per_batch = nqb * a.h;
  const int qb = head_major ? nqb - 1 - (int)(blockIdx.x % nqb)
                            : nqb - 1 - (int)((blockIdx.x % per_batch) / a.h);
  const int bh = head_major ? (int)(blockIdx.x / nqb)
                            : (int)(blockIdx.x / per_batch) * a.h + (int)(blockIdx.x % a.h);
  (void)bh_count;
  const int b = bh / a.h, hq = bh % a.h, kvh = hq / (a.h / a.hkv);
  Sched sc;
  sc.q0 = qb * kSub * kBlockM;
  sc.lo_all = 1 << 30;
  sc.hi_all = -1;
#pragma unroll
  for (int t = 0; t < kSub; ++t) {
    tile_range(a, sc.q0 + t * kBlockM, sc.lo[t], sc.hi[t]);
    if (sc.lo[t] < sc.hi[t]) {
      sc.lo_all = min(sc.lo_all, sc.lo[t]);
      sc.hi_all = max(sc.hi_all, sc.hi[t]);
    }
  }
  if (sc.hi_all < 0) sc.lo_all = sc.hi_all = 0;

  // ---- setup ----
  // The producer's lane initialises the barriers of the first loads (q_full, k_full) and sends
  // those loads (Q and the first K tiles, which wait on nothing) before the CTA-wide barrier, so
  // that they are in flight while TMEM is allocated and the other warps arrive; meanwhile the
  // warp's other lanes initialise the remaining barriers, one each (every barrier counts one
  // arrival).
  uint32_t qbytes = 0;        // producer lane: Q bytes in flight on q_full
  int k_early = 0;            // producer lane: K tiles already issued
  const uint64_t pol = l2_policy_evict_last();
  constexpr int kFirstBars = 1 + C::kStages;  // q_full, k_full[0, kStages): bars[0, kFirstBars)
  static_assert(C::kNumBars - kFirstBars <= 31, "one remaining barrier per lane");
  if (warp == kProducerWarp && lane > 0 && lane <= C::kNumBars - kFirstBars) {
    mbar_init(&bars[kFirstBars + lane - 1], 1);
    fence_mbar_init();
  }
  if (threadIdx.x == kProducerWarp * 32) {
    *abort_flag = 0;
    for (int i = 0; i < kFirstBars; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
    if (sc.hi_all > sc.lo_all) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
    }
    if (kMerge) prefetch_tmap(&tacc);
    if (kMerge ? p.fin.ptr != nullptr : !p.out_is_f32) prefetch_tmap(&tfin);
    for (int t = 0; t < kSub; ++t)
      if (sc.lo[t] < sc.hi[t]) qbytes += C::kTileBytes;
    if (qbytes) {
      mbar_arrive_expect_tx(q_full, qbytes);
      for (int t = 0; t < kSub; ++t) {
        if (sc.lo[t] >= sc.hi[t]) continue;
        uint8_t* dst = smem + C::kQOff + t * C::kTileBytes;
        for (int x = 0; x < C::kBoxes; ++x)
          tma_load_4d(dst + x * 16384, &tq, q_full, x * 64, hq, sc.q0 + t * kBlockM, b);
      }
    }
    for (; k_early < C::kStages && sc.lo_all + k_early < sc.hi_all; ++k_early) {
      uint8_t* kd = smem + C::kKOff + k_early * C::kTileBytes;
      mbar_arrive_expect_tx(&k_full[k_early], C::kTileBytes);
      for (int x = 0; x < C::kBoxes; ++x)
        tma_load_4d_hint(kd + x * 16384, &tk, &k_full[k_early], x * 64, kvh, (sc.lo_all + k_early) * kBlockN, b, pol);
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
  // Fused ring step: subtile t's accumulator rows are staged in the K (t = 0) or V (t = 1)
  // stages, taken in the order their last tiles release them: stage i of the accumulator (boxes
  // [i, i + 1) x kBoxesPerStage) goes where tile ntiles - kStages + i was (a stage no tile used
  // when that index is negative). acc_stage gives that stage; stage_acc, run by the lane that
  // fed the ring after its last load, waits for each release (the ring's next phases) and loads
  // the boxes, once the launch this one depends on (the previous ring step) is done. The first
  // step of a ring reads no accumulator and only says, once all of them are free, that the
  // stages may be written. Returns whether loads went out.
  const int ntiles = sc.hi_all - sc.lo_all;
  auto acc_stage = [&](int i) { return ((ntiles - C::kStages + i) % C::kStages + C::kStages) % C::kStages; };
  auto stage_acc = [&](int t, uint64_t* empty, uint8_t* area) -> int {
    const int qs = sc.q0 + t * kBlockM;
    if (qs >= a.lq) return 0;
    int loaded = 0;  // stages whose loads went out
    for (int i = 0; i < C::kAccStages; ++i) {
      const int x = ntiles - C::kStages + i;  // the tile whose release frees this stage
      if (x >= 0 && !wait_parity(&empty[x % C::kStages], (x / C::kStages) & 1, abort_flag, p.status)) break;
      if (i == 0) grid_dependency_wait();
      uint64_t* bar = &acc_full[t * C::kAccStages + i];
      if (p.merge_init) {
        mbar_arrive(bar);
        continue;
      }
      mbar_arrive_expect_tx(bar, C::kBoxesPerStage * C::kBox);
      uint8_t* dst = area + acc_stage(i) * C::kTileBytes;
      for (int u = 0; u < C::kBoxesPerStage; ++u) {
        const int c = i * C::kBoxesPerStage + u;
        tma_load_4d(dst + u * C::kBox, &tacc, bar, 32 * c, hq, qs, b);
      }
      ++loaded;
    }
    return loaded;
  };
  if (warp >= 8) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOther));
  if (warp == kProducerWarp) {
    // ========================== TMA producer ==========================
    if (lane == 0) {
      // (Q and the first K tiles went out during the setup)
      int it = k_early;
      for (int j = sc.lo_all + k_early; j < sc.hi_all; ++j, ++it) {
        const int s = it % C::kStages;
        if (it >= C::kStages) {
          if (!wait_parity(&k_empty[s], ((it / C::kStages) & 1) ^ 1, abort_flag, p.status)) break;
        }
        uint8_t* kd = smem + C::kKOff + s * C::kTileBytes;
        mbar_arrive_expect_tx(&k_full[s], C::kTileBytes);
        for (int x = 0; x < C::kBoxes; ++x)
          tma_load_4d_hint(kd + x * 16384, &tk, &k_full[s], x * 64, kvh, j * kBlockN, b, pol);
      }
      // Loads still in flight must land before the CTA's shared memory goes away.
      const int issued = it;
      for (int k = max(0, issued - C::kStages); k < issued; ++k) {
        volatile int no_abort = 0;
        wait_parity(&k_full[k % C::kStages], (k / C::kStages) & 1, &no_abort, p.status, 200000000ull);
      }
      if (qbytes) {
        volatile int no_abort = 0;
        wait_parity(q_full, 0, &no_abort, p.status, 200000000ull);
      }
      if constexpr (kMerge) {
        const int loaded = issued == ntiles ? stage_acc(0, k_empty, smem + C::kKOff) : 0;
        for (int i = 0; i < loaded; ++i) {
          volatile int no_abort = 0;
          wait_parity(&acc_full[i], 0, &no_abort, p.status, 200000000ull);
        }
      }
    }
  } else if (warp == kVLoadWarp) {
    // ========================== V loads (own ring, own release) ==========================
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_last();
      int it = 0;
      for (int j = sc.lo_all; j < sc.hi_all; ++j, ++it) {
        const int s = it % C::kStages;
        if (it >= C::kStages) {
          if (!wait_parity(&v_empty[s], ((it / C::kStages) & 1) ^ 1, abort_flag, p.status)) break;
        }
        uint8_t* vd = smem + C::kVOff + s * C::kTileBytes;
        mbar_arrive_expect_tx(&v_full[s], C::kTileBytes);
        for (int x = 0; x < C::kBoxes; ++x)
          tma_load_4d_hint(vd + x * 16384, &tv, &v_full[s], x * 64, kvh, j * kBlockN, b, pol);
      }
      const int issued = it;
      for (int k = max(0, issued - C::kStages); k < issued; ++k) {
        volatile int no_abort = 0;
        wait_parity(&v_full[k % C::kStages], (k / C::kStages) & 1, &no_abort, p.status, 200000000ull);
      }
      if constexpr (kMerge) {
        const int loaded = issued == ntiles ? stage_acc(1, v_empty, smem + C::kVOff) : 0;
        for (int i = 0; i < loaded; ++i) {
          volatile int no_abort = 0;
          wait_parity(&acc_full[C::kAccStages + i], 0, &no_abort, p.status, 200000000ull);
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ========================== MMA issuer ==========================
    // All 32 lanes run the loop and wait together; the issue calls elect one
    // lane. (With lane 0 alone in the loop, the busy softmax warps on the
    // same scheduler starve it of issue slots and the tensor core idles.)
    {
      // base descriptors; every operand below is an offset from one of them
      const uint64_t q_desc = sdesc_sw128(smem_u32(smem + C::kQOff), 16, 1024);
      const uint64_t k_desc = sdesc_sw128(smem_u32(smem + C::kKOff), 16, 1024);
      const uint64_t v_desc = sdesc_sw128(smem_u32(smem + C::kVOff), C::kVLbo, 1024);
      const int lo0 = sc.lo[0], hi0 = sc.hi[0], lo1 = sc.lo[1], hi1 = sc.hi[1];
      const int lo_all = sc.lo_all, hi_all = sc.hi_all;
      int pv0 = 0, pv1 = 0;  // P V products issued per subtile
      bool ok = true;
// S_t = Q_t K^T from K stage `stg` (one 16-wide K step per MMA)
#define BEA_ISSUE_S(t, stg)                                                                          \
  do {                                                                                               \
    const uint64_t qd_ = sdesc_add(q_desc, (t) * C::kTileBytes);                                     \
    const uint64_t kd_ = sdesc_add(k_desc, (stg) * C::kTileBytes);                                   \
    _Pragma("unroll") for (int k_ = 0; k_ < D / 16; ++k_) {                                          \
      const uint32_t off_ = (k_ / 4) * 16384 + (k_ % 4) * 32;                                        \
      umma_ss_warp(tmem + (t) * 128, sdesc_add(qd_, off_), sdesc_add(kd_, off_), C::kIdescS, k_ > 0 ? 1u : 0u); \
    }                                                                                                \
    umma_commit_warp(&s_full[t]);                                                                         \
  } while (0)
// O_t (+)= P_t V from V stage `stg`; P_t is read from TMEM over S_t
#define BEA_ISSUE_PV(t, stg, first)                                                                  \
  do {                                                                                               \
    const uint64_t vd_ = sdesc_add(v_desc, (stg) * C::kTileBytes);                                   \
    _Pragma("unroll") for (int k_ = 0; k_ < kBlockN / 16; ++k_)                                      \
      umma_ts_warp(tmem + 256 + (t) * 128, tmem + (t) * 128 + k_ * 8, sdesc_add(vd_, k_ * 2048), C::kIdescPV, \
              (k_ > 0 || !(first)) ? 1u : 0u);                                                       \
  } while (0)

      if (hi_all > lo_all) {
        ok = warp_wait_parity(q_full, 0, abort_flag, p.status);
        if (ok) ok = warp_wait_parity(&k_full[0], 0, abort_flag, p.status);
        if (ok) {
          tc_fence_after();
          if (lo0 == lo_all && hi0 > lo0) BEA_ISSUE_S(0, 0);
          if (lo1 == lo_all && hi1 > lo1) BEA_ISSUE_S(1, 0);
          umma_commit_warp(&k_empty[0]);  // K of the first tile is read by nothing else
        }
        int it = 0;
        for (int j = lo_all; ok && j < hi_all; ++j, ++it) {
          if (p.inject_abort == it + 1 && blockIdx.x == 0) {
            // test hook: behave exactly as if a wait of this warp had run out of time here
            if (lane == 0) {
              *abort_flag = 1;
              report_status(p.status, BEA_STATUS_TIMEOUT);
            }
            ok = false;
            break;
          }
          const int s = it % C::kStages;
          const uint32_t par = (it / C::kStages) & 1;
          const int s1 = (it + 1) % C::kStages;
          const uint32_t par1 = ((it + 1) / C::kStages) & 1;
          const bool a0 = j >= lo0 && j < hi0, a1 = j >= lo1 && j < hi1;
          const bool n0 = j + 1 >= lo0 && j + 1 < hi0, n1 = j + 1 >= lo1 && j + 1 < hi1;
          bool k_next_ready = false;
          if (!(ok = warp_wait_parity(&v_full[s], par, abort_flag, p.status))) break;
          if (a0) {
            named_bar_sync(kPReadyBar + 0, kPReadyThreads);  // P_0 of tile j is in TMEM
            tc_fence_after();
            BEA_ISSUE_PV(0, s, pv0 == 0);
            ++pv0;
            // O_0 is final once its last P V completes: subtile 0's epilogue need not wait for
            // subtile 1's last softmax and P V
            if (j == hi0 - 1) umma_commit_warp(&o_full[0]);
          }
          if (n0) {
            if (!(ok = warp_wait_parity(&k_full[s1], par1, abort_flag, p.status))) break;
            tc_fence_after();
            k_next_ready = true;
            BEA_ISSUE_S(0, s1);
          }
          if (a1) {
            named_bar_sync(kPReadyBar + 1, kPReadyThreads);  // P_1 of tile j is in TMEM
            tc_fence_after();
            BEA_ISSUE_PV(1, s, pv1 == 0);
            ++pv1;
          }
          if (n1) {
            if (!k_next_ready) {
              if (!(ok = warp_wait_parity(&k_full[s1], par1, abort_flag, p.status))) break;
              tc_fence_after();
            }
            BEA_ISSUE_S(1, s1);
          }
          if (j + 1 < hi_all) umma_commit_warp(&k_empty[s1]);  // every S of tile j+1 is issued
          umma_commit_warp(&v_empty[s]);                       // every P V of tile j is issued
          if (j == hi1 - 1) umma_commit_warp(&o_full[1]);
        }
      }
#undef BEA_ISSUE_S
#undef BEA_ISSUE_PV
      // After an abort, join the P-ready phases of the tiles not reached (a no-op otherwise).
      for (; pv0 < hi0 - lo0; ++pv0) named_bar_sync(kPReadyBar + 0, kPReadyThreads);
      for (; pv1 < hi1 - lo1; ++pv1) named_bar_sync(kPReadyBar + 1, kPReadyThreads);
      // Everything issued must finish before TMEM is released.
      umma_commit_warp(mma_done);
      volatile int no_abort = 0;
      wait_parity(mma_done, 0, &no_abort, p.status, 200000000ull);
      __syncwarp();
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    // ========================== softmax groups ==========================
    const int t = warp / 4;           // subtile
    const int r = threadIdx.x % 128;  // row within subtile == TMEM lane
    const uint32_t lane_base = (uint32_t)((warp % 4) * 32) << 16;
    const uint32_t s_tmem = tmem + lane_base + t * 128;
    const uint32_t o_tmem = tmem + lane_base + 256 + t * 128;
    const int qs = sc.q0 + t * kBlockM;
    const int qi = qs + r;
    float m_ref = -INFINITY;  // running max, log2 domain
    float l_sum = 0.f;
    bool ok = true;
    int it = 0;
    const int my_lo = t ? sc.lo[1] : sc.lo[0], my_hi = t ? sc.hi[1] : sc.hi[0];  // no dynamic indexing
    for (int j = my_lo; j < my_hi; ++j, ++it) {
      if (ok) ok = warp_wait_parity(&s_full[t], it & 1, abort_flag, p.status);
      if (!ok) {
        named_bar_sync(kPReadyBar + t, kPReadyThreads);  // aborted: keep the P-ready phases matched
        continue;
      }
      tc_fence_after();
      uint32_t sr[128];
      tmem_ld32(s_tmem + 0, sr);
      tmem_ld32(s_tmem + 32, sr + 32);
      tmem_ld32(s_tmem + 64, sr + 64);
      tmem_ld32(s_tmem + 96, sr + 96);
      tmem_wait_ld();
      reg_fence<128>(sr);
      if (tile_needs_mask(a, qs, j)) {
        const int k0 = j * kBlockN;
#pragma unroll
        for (int c = 0; c < 128; ++c) {
          const int kj = k0 + c;
          if (!(kj < a.lk && key_visible(qi, kj, a.wl, a.wr))) sr[c] = __float_as_uint(-INFINITY);
        }
      }
      // softmax_scale > 0, so the max commutes with the scaling. Eight
      // independent partial maxima keep the dependent chain short; the
      // three-input max takes two new values per instruction.
      // Partial maximum u covers columns u + 8k, k = 0..15.
      float m8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        float m = fmax3(__uint_as_float(sr[u]), __uint_as_float(sr[u + 8]), __uint_as_float(sr[u + 16]));
#pragma unroll
        for (int k = 3; k < 15; k += 2) m = fmax3(m, __uint_as_float(sr[u + 8 * k]), __uint_as_float(sr[u + 8 * k + 8]));
        m8[u] = fmaxf(m, __uint_as_float(sr[u + 120]));
      }
      float mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
      mx *= scale_log2;
      const float m_new = fmaxf(m_ref, mx);
      const bool grow = m_new > m_ref + kRescaleThreshold;  // also true when m_ref = -inf, m_new finite
      float f = 1.f;
      bool rescale = false;
      if (it == 0) {
        m_ref = m_new;  // the first P V overwrites O, nothing to rescale
      } else {
        rescale = __any_sync(0xffffffffu, grow);
        if (grow) {
          f = ex2_approx(m_ref - m_new);
          m_ref = m_new;
          l_sum *= f;
        }
      }
      const float neg_m = (m_ref == -INFINITY) ? 0.f : -m_ref;
      uint32_t pk[64];
      // exponent arguments and the row sum on packed fp32 pairs; eight independent partial sums
      const uint64_t sl2 = f2(scale_log2, scale_log2), nm2 = f2(neg_m, neg_m);
      uint64_t ps[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const uint64_t x = f2_fma(f2(__uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1])), sl2, nm2);
        const float p0 = ex2_approx(f2_lo(x));
        const float p1 = ex2_approx(f2_hi(x));
        ps[c & 3] = f2_add(ps[c & 3], f2(p0, p1));
        pk[c] = pack_bf16x2(p0, p1);
      }
      const uint64_t s2 = f2_add(f2_add(ps[0], ps[1]), f2_add(ps[2], ps[3]));
      l_sum += f2_lo(s2) + f2_hi(s2);
      tmem_st32(s_tmem + 0, pk);
      tmem_st32(s_tmem + 32, pk + 32);
      if (rescale) {
        // PV_t(j-1) has completed: s_full for tile j was committed after it. Rare (the row max
        // grew by more than 2^8): a rolled loop, which keeps the register demand of the tile
        // loop down (unrolled, it makes the compiler spill around it on every tile).
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t orow[32];
          tmem_ld32(o_tmem + c0, orow);
          tmem_wait_ld();
          reg_fence<32>(orow);
#pragma unroll
          for (int c = 0; c < 32; ++c) orow[c] = __float_as_uint(__uint_as_float(orow[c]) * f);
          tmem_st32(o_tmem + c0, orow);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      named_bar_sync(kPReadyBar + t, kPReadyThreads);
    }
    // ---- epilogue ----
    // O leaves TMEM through shared memory so that global memory sees whole
    // 128-byte row segments: each row's thread writes a chunk of its row (32
    // fp32 or 64 bf16 values, 128 bytes) into a staging buffer with the 16-byte
    // pieces of row r rotated by r & 7 (bank-conflict free both ways), then the
    // subtile's 128 threads move the chunk as 16-byte pieces, 8 threads per
    // row segment. The staging buffer is this subtile's Q tile, free once every
    // S_t has completed, which o_full[t] implies (for a subtile without tiles Q_t
    // was never loaded).
    const bool have_o = my_lo < my_hi;
    const bool row_ok = qi < a.lq;
    float* lse_p = p.lse.ptr + b * p.lse.sn + hq * p.lse.sh + qi;
    // the coalesced phase: thread u of the subtile takes 16-byte piece u % 8 of rows u / 8 + 16 k
    const int u = r;
    const int piece = u & 7;
    const bool init = kMerge && p.merge_init != 0;
    float la = -INFINITY;
    if constexpr (kMerge) {
      if (qs < a.lq && !init) {
        // Once the launch this one depends on (the previous ring step) is done, this row's
        // accumulator log-sum-exp is read while the last P V completes (L2-only: the previous
        // step wrote it from another SM).
        grid_dependency_wait();
        if (row_ok) la = __ldcg(lse_p);
      }
    }
    if (ok && have_o) ok = warp_wait_parity(&o_full[t], 0, abort_flag, p.status);
    if (qs < a.lq) {  // uniform over the subtile: all 128 threads join the barriers below
      // a dependent launch (the next ring step) touches out/lse only after the launch before it is done
      grid_dependency_wait();
      tc_fence_after();
      const float inv = (l_sum > 0.f) ? 1.f / l_sum : 0.f;
      const float L = (l_sum > 0.f) ? (m_ref + lg2_approx(l_sum)) * 0.69314718055994531f : -INFINITY;
      uint8_t* stage = smem + C::kQOff + t * C::kTileBytes;
      const int ep_id = kEpiBar + t;
      if constexpr (kMerge) {
        // Fused ring step: fold this block's (O, L) into the fp32 accumulator (out, lse) by the
        // log-sum-exp merge of flash_attn_jax flash_sharding.py, "Ring Forward":
        //   L' = max + log1p(exp(min - max)), acc <- acc exp(La - L') + O exp(L - L'),
        // leaving a row whose two log-sum-exps are both -inf unchanged. The first step of a ring
        // (merge_init) has nothing to fold into: acc <- O / l, lse <- L.
        float wa = 0.f, wb = inv, l_new = L;
        bool keep = false;
        if (!init) {
          const float mx = fmaxf(la, L);
          if (mx == -INFINITY) {
            keep = true;
          } else {
            const float mn = fminf(la, L);
            l_new = mx + log1pf(expf(mn - mx));
            wa = expf(la - l_new);
            wb = expf(L - l_new) * inv;
          }
        }
        if (ok && row_ok && !keep) *lse_p = l_new;
        const bool fin_on = p.fin.ptr != nullptr && b >= p.fin_b0 && b < p.fin_b1;
        // The accumulator rows are staged in shared memory as 32-column boxes, 128-byte
        // swizzled (16-byte piece k of row r at k ^ (r & 7)), so that each row's thread reads and
        // writes its own row without bank conflicts. The merged box goes back by a TMA store;
        // the bf16 copy is assembled in the Q tile (64-column boxes) and stored the same way.
        uint8_t* acc_area = smem + (t == 0 ? C::kKOff : C::kVOff);
        auto acc_box = [&](int c) {
          return acc_area + acc_stage(c / C::kBoxesPerStage) * C::kTileBytes + (c % C::kBoxesPerStage) * C::kBox;
        };
        uint8_t* fin_s = stage;
        // O_t leaves TMEM one 32-column chunk ahead of the merge: chunk c + 1 loads while chunk c is
        // merged (two register buffers; the chunk loop is unrolled so that they stay registers)
        uint32_t oa[32], ob[32];
        bool pend = false;
        if (ok && have_o) {
          tmem_ld32(o_tmem, oa);
          pend = true;
        }
#pragma unroll
        for (int c = 0; c < C::kAccBoxes; ++c) {
          uint32_t* cur = (c & 1) ? ob : oa;
          uint32_t* nxt = (c & 1) ? oa : ob;
          if (ok && c % C::kBoxesPerStage == 0)  // this stage of the accumulator has landed
            ok = warp_wait_parity(&acc_full[t * C::kAccStages + c / C::kBoxesPerStage], 0, abort_flag, p.status);
          if (pend) {
            tmem_wait_ld();
            reg_fence<32>(cur);
            pend = false;
          }
          if (ok) {
            if (have_o) {
              if (c + 1 < C::kAccBoxes) {
                tmem_ld32(o_tmem + 32 * (c + 1), nxt);
                pend = true;
              }
            } else {
#pragma unroll
              for (int e = 0; e < 32; ++e) cur[e] = 0u;
            }
            uint8_t* row_s = acc_box(c) + r * 128;
            uint8_t* fin_row = fin_s + (c / 2) * 16384 + r * 128;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              float4* pa = reinterpret_cast<float4*>(row_s + ((k ^ (r & 7)) * 16));
              const float o0 = __uint_as_float(cur[4 * k]), o1 = __uint_as_float(cur[4 * k + 1]);
              const float o2 = __uint_as_float(cur[4 * k + 2]), o3 = __uint_as_float(cur[4 * k + 3]);
              float4 m;
              if (init) {
                m = make_float4(o0 * wb, o1 * wb, o2 * wb, o3 * wb);
                *pa = m;
              } else if (keep) {
                m = *pa;
              } else {
                const float4 av = *pa;
                m = make_float4(fmaf(o0, wb, av.x * wa), fmaf(o1, wb, av.y * wa), fmaf(o2, wb, av.z * wa),
                                fmaf(o3, wb, av.w * wa));
                *pa = m;
              }
              if (fin_on) {
                // columns 32c + 4k .. +3 of the 64-column bf16 box c / 2: byte (c % 2) * 64 + 8k of the row
                const int pf = (c % 2) * 4 + k / 2;
                *reinterpret_cast<uint2*>(fin_row + ((pf ^ (r & 7)) * 16) + (k % 2) * 8) =
                    make_uint2(pack_bf16x2(m.x, m.y), pack_bf16x2(m.z, m.w));
              }
            }
            fence_proxy_async_smem();  // these writes are read by the TMA store below
          }
          named_bar_sync(ep_id, 128);
          if (ok && r == 0) {
            tma_store_4d(&tacc, acc_box(c), 32 * c, hq, qs, b);
            if (fin_on && (c % 2 == 1)) tma_store_4d(&tfin, fin_s + (c / 2) * 16384, 64 * (c / 2), hq, qs, b);
            bulk_commit_group();
          }
        }
        if (pend) tmem_wait_ld();  // a load still in flight after an abort
        // the stores read shared memory until they complete; the CTA's exit waits for them
        if (r == 0) bulk_wait_group_all();
      } else {
        if (ok && row_ok) *lse_p = L;
        if (p.out_is_f32) {
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 32) {
            if (ok) {
              uint32_t orow[32];
              if (have_o) {
                tmem_ld32(o_tmem + c0, orow);
                tmem_wait_ld();
                reg_fence<32>(orow);
              } else {
#pragma unroll
                for (int c = 0; c < 32; ++c) orow[c] = 0u;
              }
#pragma unroll
              for (int k = 0; k < 8; ++k)
                *reinterpret_cast<float4*>(stage + r * 128 + ((k ^ (r & 7)) * 16)) =
                    make_float4(__uint_as_float(orow[4 * k]) * inv, __uint_as_float(orow[4 * k + 1]) * inv,
                                __uint_as_float(orow[4 * k + 2]) * inv, __uint_as_float(orow[4 * k + 3]) * inv);
            }
            named_bar_sync(ep_id, 128);
            if (ok) {
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const int row = (u >> 3) + 16 * k;
                const int qrow = qs + row;
                if (qrow >= a.lq) continue;
                *reinterpret_cast<uint4*>(reinterpret_cast<float*>(p.out.ptr) + b * p.out.sn +
                                          (int64_t)qrow * p.out.sl + hq * p.out.sh + c0 + 4 * piece) =
                    *reinterpret_cast<const uint4*>(stage + row * 128 + ((piece ^ (row & 7)) * 16));
              }
            }
            named_bar_sync(ep_id, 128);
          }
        } else {
          // bf16 O_t / l: both (all) 64-column boxes staged in the subtile's Q tile, 128-byte
          // swizzled, then written by TMA stores (tfin is the output's map here)
          if (ok) {
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 64) {
#pragma unroll
              for (int hf = 0; hf < 2; ++hf) {
                uint32_t orow[32];
                if (have_o) {
                  tmem_ld32(o_tmem + c0 + 32 * hf, orow);
                  tmem_wait_ld();
                  reg_fence<32>(orow);
                } else {
#pragma unroll
                  for (int c = 0; c < 32; ++c) orow[c] = 0u;
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const int e = 8 * k;
                  uint4 v4;
                  v4.x = pack_bf16x2(__uint_as_float(orow[e]) * inv, __uint_as_float(orow[e + 1]) * inv);
                  v4.y = pack_bf16x2(__uint_as_float(orow[e + 2]) * inv, __uint_as_float(orow[e + 3]) * inv);
                  v4.z = pack_bf16x2(__uint_as_float(orow[e + 4]) * inv, __uint_as_float(orow[e + 5]) * inv);
                  v4.w = pack_bf16x2(__uint_as_float(orow[e + 6]) * inv, __uint_as_float(orow[e + 7]) * inv);
                  const int kk = 4 * hf + k;
                  *reinterpret_cast<uint4*>(stage + (c0 / 64) * 16384 + r * 128 + ((kk ^ (r & 7)) * 16)) = v4;
                }
              }
            }
            fence_proxy_async_smem();  // these writes are read by the TMA stores below
          }
          named_bar_sync(ep_id, 128);
          if (ok && r == 0) {
            for (int c = 0; c < D / 64; ++c) tma_store_4d(&tfin, stage + c * 16384, 64 * c, hq, qs, b);
            bulk_commit_group();
            // (a launch that depends on this one programmatically also needs the writes done)
            if (p.pdl_next) bulk_wait_group_all();
            else bulk_wait_group_read_all();
          }
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

template <int D, bool kMerge>
cudaError_t launch_fwd_d(const FwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& tacc, const CUtensorMap& tfin, cudaStream_t s, int* nlaunch) {
  using C = FwdCfg<D>;
  // Once per device context: allow the kernel's dynamic shared memory and read
  // its register count. The register split above is only sound at exactly
  // kRegsLaunch registers per thread; refuse to launch otherwise
  // (setmaxnreg.inc would never return).
  static PerContext<int> regs_cache;
  int regs = 0;
  cudaError_t e = regs_cache.get(
      [](int* v) {
        cudaError_t r = cudaFuncSetAttribute(fwd_bf16_kernel<D, kMerge>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (r != cudaSuccess) return r;
        cudaFuncAttributes fa;
        r = cudaFuncGetAttributes(&fa, fwd_bf16_kernel<D, kMerge>);
        *v = fa.numRegs;
        return r;
      },
      &regs);
  if (e != cudaSuccess) return e;
  if (regs != kRegsLaunch) return cudaErrorInvalidConfiguration;
  const int nqb = (p.a.lq + kSub * kBlockM - 1) / (kSub * kBlockM);
  const long long blocks = (long long)nqb * p.a.n * p.a.h;
  if (blocks == 0) return cudaSuccess;
  const float scale_log2 = p.a.scale * 1.4426950408889634f;
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
  e = cudaLaunchKernelEx(&cfg, fwd_bf16_kernel<D, kMerge>, tq, tk, tv, tacc, tfin, p, scale_log2);
  if (e != cudaSuccess) return e;
  *nlaunch += 1;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_bf16(const FwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap* tacc, const CUtensorMap* tfin, cudaStream_t s, int* nlaunch) {
  CUtensorMap none;
  std::memset(&none, 0, sizeof(none));
  if (p.merge && tacc == nullptr) return cudaErrorInvalidValue;
  // tfin: the merge's bf16 final copy, or the plain forward's bf16 output
  if ((p.merge ? p.fin.ptr != nullptr : !p.out_is_f32) && tfin == nullptr) return cudaErrorInvalidValue;
  const CUtensorMap& ta = tacc ? *tacc : none;
  const CUtensorMap& tf = tfin ? *tfin : none;
  if (p.a.d == 128) return p.merge ? launch_fwd_d<128, true>(p, tq, tk, tv, ta, tf, s, nlaunch)
                                   : launch_fwd_d<128, false>(p, tq, tk, tv, ta, tf, s, nlaunch);
  if (p.a.d == 64) return p.merge ? launch_fwd_d<64, true>(p, tq, tk, tv, ta, tf, s, nlaunch)
                                  : launch_fwd_d<64, false>(p, tq, tk, tv, ta, tf, s, nlaunch);
  return cudaErrorInvalidValue;
}

}  // namespace bea
