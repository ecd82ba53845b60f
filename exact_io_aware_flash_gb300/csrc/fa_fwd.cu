// Forward kernel: exact attention with online softmax on tcgen05 tensor cores.
//
// What it computes ("FlashAttention Primer: IO-Aware Attention, from FA1 to FA4",
// sections "Why attention is quadratic" and "FlashAttention-1"; "Flash Attention"
// (aiwiki.ai), section "Online softmax"): for every query row i,
//     O_i = sum_k softmax_k(scale * q_i . k_k) v_k,   LSE_i = ln sum_k exp(scale * q_i . k_k)
// by streaming key/value tiles through shared memory and carrying a running row
// maximum m, running sum l and an unnormalised accumulator O (the FA2 form: P is
// exponentiated against the running maximum and O is divided by l once at the
// end, "Flash Attention", section "Online softmax").
//
// GB300 design.  A work item is a pair of 128-row query tiles (A, B) of one
// head; the grid has one CTA per item, and a running CTA takes over the items
// of CTAs that have not started (cluster launch control), so each CTA runs
// items back to back with its pipelines running on across item boundaries.
//   warp 8      TMA producer and scheduler: claims and publishes the next item;
//               Q tiles per item, then K_j through a 3-stage and V_j through a
//               2-stage shared-memory ring (128-byte swizzle, 3-D tensor maps
//               over [B*H, N, d] so ragged tails are zero-filled).
//   warps 9-10  MMA issuers, one thread per query tile X: S_X = Q_X K_j^T into
//               Tensor Memory, O_X += P_X V_j with P_X read from Tensor Memory
//               (A operand) and V_j from shared memory as an MN-major B operand.
//   warp 11     idle (completes the control warpgroup for register reallocation).
//   warps 0-3   softmax for query tile A, warps 4-7 for tile B: thread t owns
//               row t (TMEM lane t); exp2 with the scale folded in; P written
//               back to TMEM as 16-bit pairs over the first half of S.
// Instantiations: 16-bit (fp16/bf16), causal sliding window (WIN), and e4m3
// inputs (F8) -- see the kernel's comment.
// The two tiles ping-pong: while one softmax group works, the tensor core runs
// the other tile's MMAs ("FlashAttention Primer", section "FlashAttention-3":
// softmax of one block overlaps the matmuls of another; Figure 7).
//
// Conditional rescaling ("Flash Attention", section "FlashAttention-4": skip the
// O rescale unless the running maximum grows by more than log2(256) = 8 in the
// exp2 domain): exact, since O and l always share the same reference maximum.
//
// Causal ("FlashAttention Primer", section "FlashAttention-1", causal
// paragraph): key tiles above the diagonal are never loaded or computed; only
// the diagonal tile and the ragged last tile are masked element-wise.
#include "fa_internal.h"
#include "ptx.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

namespace fa {
namespace {

constexpr int kBM = 128;           // query rows per tile
constexpr int kBN = 128;           // keys per tile
constexpr int kAtomBytes = 16384;  // 128 rows x 128 bytes: 64 columns of one 16-bit tile
constexpr int kThreads = 384;      // 12 warps: two softmax warpgroups, one control warpgroup
// Registers per thread: the launch gives every thread 168 (65,536 / 384, in
// steps of 8); the control warpgroup (producer, two MMA issuers, one idle warp)
// gives registers back so that each softmax thread can hold a whole row of S.
// 128 x 64 + 256 x 216 = 63,488 <= 384 x 168 = 64,512.
constexpr uint32_t kRegsControl = 64;
constexpr uint32_t kRegsSoftmax = 216;
static_assert(128 * kRegsControl + 256 * kRegsSoftmax <= kThreads * 168, "register split");
// The two query tiles run half a period apart, so K_j is released by the
// later tile; a third K stage lets K_{j+2} load while that tile finishes.
constexpr int kKStages = 3;
constexpr int kVStages = 2;
constexpr int kConsumerWarps = 10;  // 8 softmax warps + 2 MMA issuer warps read each item

template <int D, int ELT>
struct FwdSmem {
  static constexpr int kTile = kBM * D * ELT;  // bytes of one 128 x D tile of ELT-byte elements
  static constexpr int kQ = 0;               // 2 query tiles
  static constexpr int kK = kQ + 2 * kTile;  // K ring, kKStages
  static constexpr int kV = kK + kKStages * kTile;  // V ring, kVStages
  static constexpr int kBar = kV + kVStages * kTile;
  static constexpr int kMisc = kBar + 256;   // scheduler response and item slots
  static constexpr int kBytes = kMisc + 64;
  static constexpr int kAlloc = kBytes + 1024;  // slack for 1024-byte alignment
};

enum Bars {
  BQFULL = 0,    // +tile
  BQEMPTY = 2,   // +tile: the tile's last S MMA of an item has completed
  BKFULL = 4,    // +stage (3)
  BKEMPTY = 7,   // +stage (3), one arrival per MMA issuer
  BVFULL = 10,   // +stage (2)
  BVEMPTY = 12,  // +stage (2), one arrival per MMA issuer
  BSFULL = 14,   // +tile
  BPFULL = 16,   // +tile
  BODONE = 18,   // +tile
  BFINAL = 20,   // +tile
  BITEMFULL = 22,   // +slot (2): next work item published
  BITEMEMPTY = 24,  // +slot (2): read by every consumer warp
  BCLC = 26,        // scheduler response landed
  BTOKEN = 27,      // +tile: the softmax turn handed to tile X (4 arrivals)
  NBARS = 29
};

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

// Bounded wait used only while tearing down after an abort: ignores the abort
// flag so that copies already in flight land before the CTA exits.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > 200000000ull) break;
  }
}

// One work item: a pair of 128-row query tiles (A = 2p, B = 2p + 1) of one head.
// The item streams key tiles loA .. loA + nKV - 1; tile X visits nX of them,
// starting at key tile loX.
struct FwdItem {
  int bh, kvh, tA, tB, nA, nB, nKV, loA, loB;
};

// First key tile a causal sliding window of `window` keys exposes to query
// tile t: its first row, t*128, sees keys t*128 - window + 1 .. t*128.
__device__ __forceinline__ int window_first_tile(int t, int window) {
  const int first_key = t * kBM - window + 1;
  return first_key > 0 ? first_key / kBN : 0;
}

// per: query tiles per item, 2 (tiles 2p and 2p + 1) or 1 (tile p alone, no
// tile B), the latter when pairs would leave SMs idle.
template <bool WIN>
__device__ __forceinline__ FwdItem decode_item(int item, int heads, int head_group, int Hq,
                                               int Hkv, int T, int causal, int window, int per) {
  const int pairs = (T + per - 1) / per;
  // Groups of heads whose K and V stay in L2; heaviest causal pairs first.
  const WorkItem wi = grouped_heavy_first(item, heads, pairs, head_group);
  const int pair = pairs - 1 - wi.rank;
  FwdItem it;
  it.bh = wi.head;  // b * Hq + h
  const int h = it.bh % Hq;
  const int b = it.bh / Hq;
  it.kvh = b * Hkv + h / (Hq / Hkv);
  it.tA = per * pair;
  it.tB = per == 2 ? per * pair + 1 : T;
  const bool hasB = it.tB < T;
  it.loA = WIN ? window_first_tile(it.tA, window) : 0;
  it.loB = (WIN && hasB) ? window_first_tile(it.tB, window) : it.loA;
  it.nA = causal ? it.tA + 1 - it.loA : T;
  it.nB = hasB ? (causal ? it.tB + 1 - it.loB : T) : 0;
  const int endB = it.loB - it.loA + it.nB;  // stream tiles tile B needs
  it.nKV = it.nA > endB ? it.nA : endB;
  return it;
}

// Persistent over work items: the grid has one CTA per item, and a running CTA
// takes over the items of CTAs that have not started yet (cluster launch
// control), so one CTA runs many items back to back and the next item's Q
// loads and first S MMA overlap the current item's last softmax and epilogue.
// WIN: causal sliding window of `window` keys (key k visible to query i iff
// i - window < k <= i): each query tile visits only the key tiles its window
// reaches, and the window's lower edge is masked element-wise ("Flash
// Attention" (aiwiki.ai), sections "Features" and "Block-sparse
// FlashAttention": blocks a mask leaves empty are skipped).
// F8: e4m3 inputs ("FlashAttention Primer", section "FlashAttention-3: Hopper
// asynchrony and FP8": block-quantized FP8 operands).  Q and K arrive as codes
// with one scale per 128-row block (q_scale, k_scale), V as transposed codes
// [d][keys] with one scale per channel (v_scale); both products run as
// kind::f8f6f4 MMAs (twice the 16-bit rate), P is rounded to e4m3 for P V, the
// block scales enter each round's exponent factor and the channel scales the
// epilogue.  O is written in bfloat16.
template <int D, bool BF16, bool WIN, bool F8>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, void* __restrict__ out,
                  float* __restrict__ lse_out, int heads, int head_group, int Hq, int Hkv, int N,
                  int causal, int window, int per, float scale_log2, const float* __restrict__ q_scale,
                  const float* __restrict__ k_scale, const float* __restrict__ v_scale, int* err) {
  static_assert(!F8 || (D == 128 && BF16 && !WIN), "e4m3 path: d = 128, bfloat16 output, no window");
  constexpr int kElt = F8 ? 1 : 2;
  using L = FwdSmem<D, kElt>;
  constexpr int kAtoms = D * kElt / 128;  // 128-byte-wide atoms per tile row
  constexpr int kAtomCols = 128 / kElt;   // elements per atom row
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  void* clc_resp = smem + L::kMisc;                                   // 16 bytes
  volatile int* item_slot = reinterpret_cast<volatile int*>(smem + L::kMisc + 16);  // 2 ints

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int T = (N + kBM - 1) / kBM;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NBARS; ++i) {
      uint32_t cnt = 1;
      if (i == BPFULL || i == BPFULL + 1 || i == BTOKEN || i == BTOKEN + 1) cnt = 4;
      if ((i >= BKEMPTY && i < BKEMPTY + kKStages) || (i >= BVEMPTY && i < BVEMPTY + kVStages)) cnt = 2;
      if (i == BITEMEMPTY || i == BITEMEMPTY + 1) cnt = kConsumerWarps;
      mbar_init(&bar[i], cnt);
    }
    *abort_flag = (*reinterpret_cast<volatile int*>(err) != kDevErrNone) ? 1 : 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool run = (*abort_flag == 0);

  // Every role walks the same item sequence, published by the producer one
  // item at a time through a two-slot ring; -1 ends it.  Returns false on abort.
  auto next_item = [&](int count, int& item) -> bool {
    const int slot = count & 1;
    if (!mbar_wait(&bar[BITEMFULL + slot], (count >> 1) & 1, abort_flag, err)) return false;
    item = item_slot[slot];
    return true;
  };

  if (warp >= 8) {
  // Control warpgroup.  Register reallocation sits inside each role's branch so
  // that no softmax code is reachable under the control warpgroup's limit.
  setmaxnreg_dec<kRegsControl>();
  if (run && warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      const uint64_t pol_q = l2_policy_evict_first();
      const uint64_t pol_kv = l2_policy_evict_last();
      int item = blockIdx.x;
      int kv = 0;                  // key tiles loaded so far, over all items (ring position)
      int kdone = 0, vdone = 0;    // K and V loads issued (differ only after an abort)
      int quse[2] = {0, 0};        // items so far that used query buffer X
      int qpend[2] = {-1, -1};     // parity of the last Q load per buffer, -1 if none
      bool clc_pending = false;    // a scheduler request is in flight
      bool clc_open = true;        // no request has failed yet
      int clc_count = 0;
      bool ok = true;
      for (int count = 0; ok; ++count) {
        const int slot = count & 1;
        if (!(ok = mbar_wait(&bar[BITEMEMPTY + slot], ((count >> 1) & 1) ^ 1, abort_flag, err))) break;
        item_slot[slot] = item;
        mbar_arrive(&bar[BITEMFULL + slot]);  // release: the slot write is visible to waiters
        if (item < 0) break;
        const FwdItem it = decode_item<WIN>(item, heads, head_group, Hq, Hkv, T, causal, window, per);
        // Query tiles: buffer X is free once the previous item's last S_X has completed.
        for (int X = 0; X < 2 && ok; ++X) {
          const int nX = X ? it.nB : it.nA;
          if (nX == 0) continue;
          if (quse[X] > 0 && !(ok = mbar_wait(&bar[BQEMPTY + X], (quse[X] - 1) & 1, abort_flag, err)))
            break;
          mbar_expect_tx(&bar[BQFULL + X], L::kTile);
          for (int a = 0; a < kAtoms; ++a)
            tma_load_3d(smem + L::kQ + X * L::kTile + a * kAtomBytes, &tm_q, &bar[BQFULL + X],
                        a * kAtomCols, (X ? it.tB : it.tA) * kBM, it.bh, pol_q);
          qpend[X] = quse[X] & 1;
          ++quse[X];
        }
        for (int j = 0; ok && j < it.nKV; ++j, ++kv) {
          const int sk = kv % kKStages;
          const int sv = kv % kVStages;
          if (!(ok = mbar_wait(&bar[BKEMPTY + sk], ((kv / kKStages) & 1) ^ 1, abort_flag, err))) break;
          mbar_expect_tx(&bar[BKFULL + sk], L::kTile);
          for (int a = 0; a < kAtoms; ++a)
            tma_load_3d(smem + L::kK + sk * L::kTile + a * kAtomBytes, &tm_k, &bar[BKFULL + sk],
                        a * kAtomCols, (it.loA + j) * kBN, it.kvh, pol_kv);
          kdone = kv + 1;
          if (!(ok = mbar_wait(&bar[BVEMPTY + sv], ((kv / kVStages) & 1) ^ 1, abort_flag, err))) break;
          mbar_expect_tx(&bar[BVFULL + sv], L::kTile);
          if constexpr (F8) {  // transposed codes: box of d rows x 128 keys
            tma_load_3d(smem + L::kV + sv * L::kTile, &tm_v, &bar[BVFULL + sv], (it.loA + j) * kBN, 0,
                        it.kvh, pol_kv);
          } else {
            for (int a = 0; a < kAtoms; ++a)
              tma_load_3d(smem + L::kV + sv * L::kTile + a * kAtomBytes, &tm_v, &bar[BVFULL + sv],
                          a * 64, (it.loA + j) * kBN, it.kvh, pol_kv);
          }
          vdone = kv + 1;
        }
        if (!ok) break;
        // Claim the next item only now that this one's loads are all issued, so
        // that a claimed item waits as little as possible behind this one.
        int next = -1;
        if (clc_open) {
          mbar_expect_tx(&bar[BCLC], 16);
          clc_try_cancel(clc_resp, &bar[BCLC]);
          clc_pending = true;
          if (!(ok = mbar_wait(&bar[BCLC], clc_count & 1, abort_flag, err))) break;
          clc_pending = false;
          ++clc_count;
          next = clc_cancelled_block_x(clc_resp);
          if (next >= static_cast<int>(gridDim.x)) next = -1;
          if (next < 0) clc_open = false;
        }
        item = next;
      }
      if (*abort_flag) {
        // Let every copy already issued land before shared memory is released.
        for (int X = 0; X < 2; ++X)
          if (qpend[X] >= 0) drain_wait(&bar[BQFULL + X], static_cast<uint32_t>(qpend[X]));
        for (int u = (kdone > kKStages ? kdone - kKStages : 0); u < kdone; ++u)
          drain_wait(&bar[BKFULL + u % kKStages], (u / kKStages) & 1);
        for (int u = (vdone > kVStages ? vdone - kVStages : 0); u < vdone; ++u)
          drain_wait(&bar[BVFULL + u % kVStages], (u / kVStages) & 1);
        if (clc_pending) drain_wait(&bar[BCLC], clc_count & 1);
      }
    }
  } else if (run && (warp == 9 || warp == 10)) {
    // ------------------------------------------------------------ MMA issuers
    // One issuing thread per query tile: a thread blocks while the tensor core
    // accepts its MMAs, and with one issuer per tile that blocking never holds
    // up the other tile's chain.  Each tile runs S(j), softmax(j), PV(j),
    // S(j+1), ...; S(j+1) overwrites the columns PV(j) reads P from, so it is
    // issued once PV(j) has completed (tcgen05 orders MMAs only for the same
    // accumulator).  K_j and V_j are released when both tiles are done with
    // them: the empty barriers count one arrival per issuer.
    const int X = warp - 9;
    constexpr uint32_t kIdS = F8 ? idesc_e4m3(kBM, kBN) : idesc_f16(kBM, kBN, BF16, false, false);
    constexpr uint32_t kIdO = F8 ? idesc_e4m3(kBM, D) : idesc_f16(kBM, D, BF16, false, true);
    const uint32_t qa = smem_u32(smem + L::kQ) + X * L::kTile;
    const uint32_t sk = smem_u32(smem + L::kK);
    const uint32_t sv = smem_u32(smem + L::kV);
    const uint32_t tS = tmem + X * 128;
    const uint32_t tO = tmem + 256 + X * 128;

    // Descriptors: the k-step-0 encoding of each tile plus a compile-time
    // offset of the start-address field (bits 0-13, address >> 4; shared
    // addresses stay below 2^18), which keeps the issuing thread's per-MMA
    // instruction count low.
    constexpr uint64_t kStageStep = L::kTile >> 4;
    const uint64_t dq0 = sdesc_sw128(qa, 16, 1024);
    const uint64_t dk0 = sdesc_sw128(sk, 16, 1024);
    const uint64_t dv0 = F8 ? sdesc_sw128(sv, 16, 1024) : sdesc_sw128(sv, kAtomBytes, 1024);
    auto issue_s = [&](int stk) {  // S_X = Q_X K_j^T
      const uint64_t kd = dk0 + stk * kStageStep;
#pragma unroll
      for (int ks = 0; ks < D * kElt / 32; ++ks) {  // 32 bytes of K per instruction
        const uint64_t off = static_cast<uint64_t>(((ks >> 2) * kAtomBytes + (ks & 3) * 32) >> 4);
        if constexpr (F8)
          mma_ss_e4m3(tS, dq0 + off, kd + off, kIdS, ks > 0);
        else
          mma_ss(tS, dq0 + off, kd + off, kIdS, ks > 0);
      }
      mma_commit(&bar[BSFULL + X]);
      mma_commit(&bar[BKEMPTY + stk]);
    };
    auto issue_pv = [&](int stv, bool first) {
      const uint64_t vd = dv0 + stv * kStageStep;
#pragma unroll
      for (int ks = 0; ks < kBN * kElt / 32; ++ks) {
        // P: 32 bytes of keys = 8 TMEM columns per instruction.  V: MN-major
        // 16-bit tile, or (e4m3) the transposed codes as a K-major operand.
        if constexpr (F8)
          mma_ts_e4m3(tO, tS + ks * 8, vd + static_cast<uint64_t>((ks * 32) >> 4), kIdO,
                      (!first || ks > 0) ? 1u : 0u);
        else
          mma_ts(tO, tS + ks * 8, vd + static_cast<uint64_t>((ks * 2048) >> 4), kIdO,
                 (!first || ks > 0) ? 1u : 0u);
      }
      mma_commit(&bar[BODONE + X]);
      mma_commit(&bar[BVEMPTY + stv]);
    };

    int kv = 0;     // key tiles consumed so far over all items (ring position)
    int xs = 0;     // S/softmax/PV rounds of this tile so far over all items
    int quse = 0;   // items so far in which this tile existed
    bool ok = true;
    for (int count = 0; ok; ++count) {
      int item = -1;
      bool got = true;
      if (lane == 0) got = next_item(count, item);
      ok = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
      item = __shfl_sync(0xffffffffu, item, 0);
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[BITEMEMPTY + (count & 1)]);
      if (item < 0) break;
      if (lane == 0) {
        const FwdItem it = decode_item<WIN>(item, heads, head_group, Hq, Hkv, T, causal, window, per);
        const int nX = X ? it.nB : it.nA;
        // Key tiles of the item's stream this query tile does not visit (under
        // a sliding window, tile B skips the first one; under causal masking
        // tile A skips the last) still need this issuer's release.  It consumes
        // them like the others -- waits until the tile has landed, then
        // releases it -- so that its view of each ring stays in step: every
        // wait on a full barrier is then for the phase right after the last
        // one it observed, which a parity wait can tell apart.
        auto skip_tile = [&](int u) -> bool {
          const int stk = u % kKStages;
          const int stv = u % kVStages;
          if (!mbar_wait(&bar[BKFULL + stk], (u / kKStages) & 1, abort_flag, err)) return false;
          if (!mbar_wait(&bar[BVFULL + stv], (u / kVStages) & 1, abort_flag, err)) return false;
          mbar_arrive(&bar[BKEMPTY + stk]);
          mbar_arrive(&bar[BVEMPTY + stv]);
          return true;
        };
        const int lead = (WIN && X) ? it.loB - it.loA : 0;
        for (int j = 0; ok && j < lead; ++j) ok = skip_tile(kv + j);
        const int base = kv + lead;  // ring position of this tile's first key tile
        if (ok && nX > 0) {
          const int stk0 = base % kKStages;
          ok = mbar_wait(&bar[BQFULL + X], quse & 1, abort_flag, err) &&
               mbar_wait(&bar[BKFULL + stk0], (base / kKStages) & 1, abort_flag, err);
          // The previous item's last PV reads P from the S columns.
          if (ok && xs > 0) ok = mbar_wait(&bar[BODONE + X], (xs - 1) & 1, abort_flag, err);
          if (ok) {
            tc_fence_after();
            issue_s(stk0);
            if (nX == 1) mma_commit(&bar[BQEMPTY + X]);
          }
          for (int j = 0; ok && j < nX; ++j) {
            const int u = base + j;
            const int stv = u % kVStages;
            if (!(ok = mbar_wait(&bar[BVFULL + stv], (u / kVStages) & 1, abort_flag, err))) break;
            if (!(ok = mbar_wait(&bar[BPFULL + X], (xs + j) & 1, abort_flag, err))) break;
            tc_fence_after();
            issue_pv(stv, j == 0);
            if (j + 1 < nX) {
              const int stk1 = (u + 1) % kKStages;
              if (!(ok = mbar_wait(&bar[BKFULL + stk1], ((u + 1) / kKStages) & 1, abort_flag, err))) break;
              if (!(ok = mbar_wait(&bar[BODONE + X], (xs + j) & 1, abort_flag, err))) break;
              tc_fence_after();
              issue_s(stk1);
              if (j + 2 == nX) mma_commit(&bar[BQEMPTY + X]);  // last S of the item: Q_X free after it
            }
          }
          xs += nX;
          ++quse;
        }
        for (int j = lead + nX; ok && j < it.nKV; ++j) ok = skip_tile(kv + j);
        kv += it.nKV;
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    }
    if (lane == 0) {
      // Every MMA this thread issued has completed before TMEM is released.
      mma_commit(&bar[BFINAL + X]);
      drain_wait(&bar[BFINAL + X], 0);
    }
  }
  } else {
  setmaxnreg_inc<kRegsSoftmax>();
  if (run) {
    // ------------------------------------------------------------ softmax + epilogue
    const int X = warp >> 2;
    const int r = threadIdx.x & 127;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + X * 128;
    const uint32_t tO = tmem + lane_off + 256 + X * 128;
    const bool pos_scale = scale_log2 > 0.f;
    int xs = 0;           // softmax rounds of this tile so far over all items
    int tokens = 0;       // turns handed to this tile so far
    int prev_nA = 0, prev_nB = 0;  // rounds of each tile in the previous item (0: none yet)
    bool ok = true;
    for (int count = 0; ok; ++count) {
      int item = -1;
      bool got = true;
      if (lane == 0) got = next_item(count, item);
      ok = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
      item = __shfl_sync(0xffffffffu, item, 0);
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[BITEMEMPTY + (count & 1)]);
      if (item < 0) break;
      const FwdItem it = decode_item<WIN>(item, heads, head_group, Hq, Hkv, T, causal, window, per);
      const int t = X ? it.tB : it.tA;
      const int nX = X ? it.nB : it.nA;
      const int loX = X ? it.loB : it.loA;  // key tile of round 0
      const float qsc = F8 ? q_scale[static_cast<size_t>(it.bh) * T + t] : 1.f;
      const int m = it.nA < it.nB ? it.nA : it.nB;  // rounds both tiles have
      const int q = t * kBM + r;
      float m_run = -INFINITY;
      float l_run = 0.f;
      for (int j = 0; j < nX; ++j) {
        // The two tiles' softmaxes take turns, so that each runs alone on the
        // SM's ALUs while the tensor core works on the other tile.  Over all
        // items the rounds run in one sequence: per item A(0), B(0), A(1),
        // B(1), ..., then the rounds only one tile has (B's last round under
        // causal masking; every round of A when the item has no tile B).  A
        // tile waits for the turn where the round before its own in that
        // sequence is the other tile's, and hands the turn over where the
        // round after its own is the other tile's.  Every item starts with
        // A(0).  Hand-overs to one tile alternate with hand-overs back, so
        // each wait is for the phase right after the last one this tile saw.
        bool wait_turn, pass_turn;
        if (X == 0) {
          wait_turn = (j == 0) ? (prev_nA > 0 && prev_nB >= prev_nA) : (j <= m);
          pass_turn = j < m;
        } else {
          wait_turn = j < m;
          pass_turn = (j < m - 1) || (j == m - 1 && it.nA >= it.nB) || (j >= m && j == it.nB - 1);
        }
        bool turn = true;
        if (wait_turn) {
          turn = mbar_wait(&bar[BTOKEN + X], tokens & 1, abort_flag, err);
          ++tokens;
        }
        ok = __all_sync(0xffffffffu, turn && mbar_wait(&bar[BSFULL + X], (xs + j) & 1, abort_flag, err));
        if (!ok) break;
        tc_fence_after();
        // x holds the scores as raw bits: s * scale * log2(e) after the first pass.
        uint32_t x[kBN];
#pragma unroll
        for (int c = 0; c < kBN; c += 32) tmem_ld32(tS + c, x + c);
        tmem_ld_wait();
        reg_fence<kBN>(x);
        const int kbase = (loX + j) * kBN;
        const bool diag = causal && (loX + j == t);
        // The factor from raw scores to the exp2 domain: scale*log2(e), times the
        // query and key blocks' dequantization scales for e4m3 inputs.
        float fac = scale_log2;
        bool pos = pos_scale;
        if constexpr (F8) {
          fac = scale_log2 * (qsc * k_scale[static_cast<size_t>(it.kvh) * T + loX + j]);
          pos = fac > 0.f;
        }
        const float sfac_r = pos ? fac : 1.0f;
        // Scores stay raw when the factor is positive (the exponent is then one
        // FFMA, s * factor - m, and the row maximum of raw scores times the
        // positive factor is the maximum of the scaled scores); otherwise they
        // are scaled first and the factor below is 1.
        if (!pos) {
#pragma unroll
          for (int c = 0; c < kBN; ++c) x[c] = __float_as_uint(__uint_as_float(x[c]) * fac);
        }
        if (diag || kbase + kBN > N) {
          int lim = N - kbase;
          if (diag && r + 1 < lim) lim = r + 1;  // key kbase + c visible iff c <= r
#pragma unroll
          for (int c = 0; c < kBN; ++c)
            if (c >= lim) x[c] = __float_as_uint(-INFINITY);
        }
        if (WIN && kbase + window <= t * kBM + kBM - 1) {
          // The window's lower edge crosses this tile: key kbase + c is visible
          // to query q iff kbase + c > q - window.  A row can be left with no
          // visible key here (only in its first round); see m_use below.
          const int lo_c = q - window + 1 - kbase;
#pragma unroll
          for (int c = 0; c < kBN; ++c)
            if (c < lo_c) x[c] = __float_as_uint(-INFINITY);
        }
        // row maximum: eight independent chains (chain u: scores u, u+8, ...,
        // u+120) of three-input maxima, then a tree
        float m8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          float m = fmax3(__uint_as_float(x[u]), __uint_as_float(x[u + 8]), __uint_as_float(x[u + 16]));
#pragma unroll
          for (int k = 3; k < 15; k += 2)
            m = fmax3(m, __uint_as_float(x[u + 8 * k]), __uint_as_float(x[u + 8 * k + 8]));
          m8[u] = fmaxf(m, __uint_as_float(x[u + 120]));
        }
        const float mx =
            fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7])) * sfac_r;
        // Conditional rescale: keep the stale maximum unless it grew by more than 8
        // (p <= 2^8 then); the decision is warp-uniform because TMEM access is.
        float alpha = 1.0f;
        bool rescale = false;
        if (j == 0) {
          m_run = mx;
        } else {
          const bool need = mx > m_run + 8.0f;
          rescale = __any_sync(0xffffffffu, need);
          if (need) {
            alpha = ex2_approx(m_run - mx);
            m_run = mx;
          }
        }
        // exponent arguments and row sums two at a time (packed fp32).  A row
        // whose keys so far are all masked has m_run = -inf; its exponents are
        // taken against 0 (all p = 0), and its next round rescales by 0.
        const float m_use = (WIN && m_run == -INFINITY) ? 0.f : m_run;
        const uint64_t sfac2 = f2_pack(sfac_r, sfac_r);
        const uint64_t negm2 = f2_pack(-m_use, -m_use);
        uint64_t rs2[2] = {0ull, 0ull};
#pragma unroll
        for (int c = 0; c < kBN; c += 32) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float a0, a1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(x[c + 2 * e]), __uint_as_float(x[c + 2 * e + 1])),
                             sfac2, negm2),
                      a0, a1);
            const float p0 = ex2_approx(a0);
            const float p1 = ex2_approx(a1);
            rs2[e & 1] = f2_add(rs2[e & 1], f2_pack(p0, p1));
            if constexpr (F8) {  // four e4m3 per column, the lowest key in the lowest byte
              const uint32_t h2 = __nv_cvt_float2_to_fp8x2(make_float2(p0, p1), __NV_SATFINITE, __NV_E4M3);
              pk[e >> 1] = (e & 1) ? (pk[e >> 1] | (h2 << 16)) : h2;
            } else {
              pk[e] = pack2<BF16>(p0, p1);
            }
          }
          if constexpr (F8)
            tmem_st8(tS + c / 4, pk);
          else
            tmem_st16(tS + c / 2, pk);
        }
        float r0, r1, r2, r3;
        f2_unpack(rs2[0], r0, r1);
        f2_unpack(rs2[1], r2, r3);
        l_run = l_run * alpha + ((r0 + r1) + (r2 + r3));
        if (rescale) {
          // O_X was last written by PV_X(j-1), which completed before S_X(j) was issued.
#pragma unroll
          for (int c = 0; c < D; c += 32) {
            uint32_t o[32];
            tmem_ld32(tO + c, o);
            tmem_ld_wait();
            reg_fence<32>(o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(tO + c, o);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bar[BPFULL + X]);
          if (pass_turn) mbar_arrive(&bar[BTOKEN + (X ^ 1)]);
        }
      }
      if (ok && nX > 0)
        ok = __all_sync(0xffffffffu, mbar_wait(&bar[BODONE + X], (xs + nX - 1) & 1, abort_flag, err));
      if (ok && nX > 0) {
        // Epilogue.  The next item's first PV overwrites O_X; it is issued only
        // after this warp's next P arrival, which follows these loads.
        tc_fence_after();
        const float inv_l = 1.0f / l_run;
        const bool valid = q < N;
        // Rows are 128 or 256 bytes, so 32-byte alignment of O's base (the ABI
        // guarantees 16) makes every 32-column chunk 32-byte aligned.
        const bool out32 = (reinterpret_cast<uintptr_t>(out) & 31) == 0;
        uint16_t* orow = reinterpret_cast<uint16_t*>(out) + (static_cast<size_t>(it.bh) * N + q) * D;
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          uint32_t o[32];
          tmem_ld32(tO + c, o);
          tmem_ld_wait();
          reg_fence<32>(o);
          uint32_t pk[16];
          if constexpr (F8) {  // V's channel scales
            const float* vsc = v_scale + static_cast<size_t>(it.kvh) * D + c;
#pragma unroll
            for (int e = 0; e < 16; ++e)
              pk[e] = pack2<BF16>(__uint_as_float(o[2 * e]) * (inv_l * vsc[2 * e]),
                                  __uint_as_float(o[2 * e + 1]) * (inv_l * vsc[2 * e + 1]));
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e)
              pk[e] = pack2<BF16>(__uint_as_float(o[2 * e]) * inv_l, __uint_as_float(o[2 * e + 1]) * inv_l);
          }
          if (valid) {
            if (out32) {  // whole 32-byte sectors: half the store instructions
              st_global_v8(orow + c, pk);
              st_global_v8(orow + c + 16, pk + 8);
            } else {
              uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
              for (int v4 = 0; v4 < 4; ++v4)
                dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
            }
          }
        }
        if (valid)
          lse_out[static_cast<size_t>(it.bh) * N + q] = (m_run + log2f(l_run)) * 0.69314718055994530942f;
      }
      xs += nX;
      prev_nA = it.nA;
      prev_nB = it.nB;
    }
  }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool BF16, bool WIN, bool F8 = false>
cudaError_t launch_fwd_t(const AttnShape& s, const FwdArgs& a, cudaStream_t stream) {
  auto kern = fa_fwd_kernel<D, BF16, WIN, F8>;
  constexpr int smem = FwdSmem<D, F8 ? 1 : 2>::kAlloc;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), smem,
                                F8 ? 28 : (WIN ? 4 : 0) + (D == 64 ? 0 : 2) + (BF16 ? 1 : 0));
  if (e != cudaSuccess) return e;
  const int T = (s.N + kBM - 1) / kBM;
  // Work items of two query tiles, or of one when pairs would not fill the SMs.
  const int per = (static_cast<long>((T + 1) / 2) * s.B * s.Hq < sm_count()) ? 1 : 2;
  const int items_per_head = (T + per - 1) / per;
  dim3 grid(static_cast<unsigned>(items_per_head * s.B * s.Hq));  // (head, item) work items
  const float scale_log2 = s.scale * 1.4426950408889634f;
  // Heads side by side so that their K and V (4*N*d bytes per KV head, shared
  // by Hq/Hkv query heads) stay within about a quarter of the L2.
  const long kv_bytes_per_head = 4L * s.N * D / (s.Hq / s.Hkv);
  long hg = (32L << 20) / (kv_bytes_per_head > 0 ? kv_bytes_per_head : 1);
  hg = hg < 1 ? 1 : (hg > 64 ? 64 : hg);
  kern<<<grid, kThreads, smem, stream>>>(a.tm_q, a.tm_k, a.tm_v, a.o, a.lse, s.B * s.Hq,
                                         static_cast<int>(hg), s.Hq, s.Hkv, s.N, s.causal,
                                         s.window, per, scale_log2, a.q_scale, a.k_scale, a.v_scale,
                                         a.err);
  return cudaGetLastError();
}

}  // namespace

size_t forward_smem_bytes(int d) {
  return d == 64 ? FwdSmem<64, 2>::kAlloc : FwdSmem<128, 2>::kAlloc;
}

cudaError_t launch_forward_fp8(const AttnShape& s, const FwdArgs& a, cudaStream_t stream) {
  return launch_fwd_t<128, true, false, true>(s, a, stream);
}

cudaError_t launch_forward(const AttnShape& s, const FwdArgs& a, cudaStream_t stream) {
  if (s.window > 0) {  // causal sliding window
    if (s.d == 64)
      return s.bf16 ? launch_fwd_t<64, true, true>(s, a, stream) : launch_fwd_t<64, false, true>(s, a, stream);
    return s.bf16 ? launch_fwd_t<128, true, true>(s, a, stream) : launch_fwd_t<128, false, true>(s, a, stream);
  }
  if (s.d == 64)
    return s.bf16 ? launch_fwd_t<64, true, false>(s, a, stream) : launch_fwd_t<64, false, false>(s, a, stream);
  return s.bf16 ? launch_fwd_t<128, true, false>(s, a, stream) : launch_fwd_t<128, false, false>(s, a, stream);
}

}  // namespace fa
