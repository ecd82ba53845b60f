// Backward kernels: recompute P block by block from the saved log-sum-exp and
// produce dQ, dK, dV without ever storing an N x N matrix.
//
// Math ("FlashAttention Primer: IO-Aware Attention, from FA1 to FA4", section
// "Backward pass: recomputation instead of storage", Figure 5; the gradient of
// O = softmax(scale Q K^T) V, with the softmax-Jacobian term D that the printed
// formula leaves out):
//     P    = exp(scale * Q K^T - LSE)           (recomputed, never stored)
//     dV   = P^T dO
//     dP   = dO V^T
//     D_i  = sum_c dO_ic O_ic
//     dS   = P o (dP - D)
//     dQ   = scale * dS K,   dK = scale * dS^T Q
//
// Kernels, in launch order on the caller's stream:
//   fa_bwd_dq_kernel     one CTA per (query head, 128-query tile i), looping over
//                        key tiles j (causal: j <= i), dQ accumulating in TMEM:
//                          D_i (rows of O and dO, while the first S is computed)
//                          S = Q_i K_j^T,  dP = dO_i V_j^T        (SMEM x SMEM)
//                          P, dS                               (compute warps)
//                          dQ += dS K_j                        (TMEM A operand)
//                        It also writes D for the next kernel.
//   fa_bwd_dkdv_kernel   one CTA per (KV head, 128-key tile j), looping over the
//                        KV head's query heads and query tiles i (causal: i >= j),
//                        in the transposed orientation so the key tile owns the
//                        TMEM lanes and dK, dV accumulate in Tensor Memory:
//                          S^T  = K_j Q_i^T,  dP^T = V_j dO_i^T   (SMEM x SMEM)
//                          P^T, dS^T                           (compute warps)
//                          dV  += P^T dO_i,   dK  += dS^T Q_i     (TMEM A operand)
//                        Its body (dkdv_body.cuh) is shared with the one-pass
//                        backward of fa_bwd_atomic.cu.
// Outputs leave as 16-bit tiles staged in idle shared memory and written by
// TMA stores (a thread-per-row global store pattern costs a whole iteration).
// dQ is therefore summed over key tiles inside one CTA rather than with atomic
// adds across CTAs (the primer notes the default backward uses atomic adds and
// is nondeterministic, section "Backward pass: recomputation instead of
// storage").  Every gradient is summed in a fixed order, so the backward is
// bitwise deterministic; the price is recomputing S and dP in both kernels
// (7 instead of 5 N x N x d products).
//
// Both kernels use 6 warps: warps 0-3 compute (thread t owns row t of the
// tile, TMEM lane t), warp 4 is the TMA producer, warp 5 the single-thread MMA
// issuer and TMEM allocator.
#include "dkdv_body.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

using namespace bwd;

constexpr int kThreads = 192;  // dQ kernel: 4 compute warps, producer, MMA issuer

// ------------------------------------------------------------------ dK, dV
// The key-tile pass (dkdv_body.cuh) without the one-pass dQ share.
template <int D, bool BF16, bool WIN>
__global__ void __launch_bounds__(kDkdvThreads, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                       const float* __restrict__ lse, const float* __restrict__ Drow, int heads,
                       int head_group, int Hq, int Hkv, int N, int causal, int window, float scale,
                       int* err) {
  dkdv_body<D, BF16, WIN, false>(&tm_q, &tm_k, &tm_v, &tm_do, &tm_dk, &tm_dv, lse, Drow, nullptr, heads,
                                 head_group, Hq, Hkv, N, causal, window, scale, err);
}

// ------------------------------------------------------------------ dQ
// K_j is read by S(j) and by dQ(j), the last MMA of an iteration, so its stage
// frees late; three stages let the load of K_{j+2} overlap dQ(j).  V_j is read
// only by dP(j) and frees early: two stages.
constexpr int kDqKStages = 3;

template <int D>
struct DqSmem {
  static constexpr int kTile = kBlk * D * 2;
  static constexpr int kQ = 0;
  static constexpr int kdO = kQ + kTile;
  static constexpr int kK = kdO + kTile;                 // kDqKStages stages
  static constexpr int kV = kK + kDqKStages * kTile;     // 2 stages
  static constexpr int kBar = kV + 2 * kTile;
  static constexpr int kBytes = kBar + 256;
  static constexpr int kAlloc = kBytes + 1024;
};

enum DqBars {
  QB_Q = 0,       // Q_i, dO_i
  QB_KFULL = 1,   // +stage (3)
  QB_KEMPTY = 4,  // +stage (3)
  QB_VFULL = 7,   // +stage (2)
  QB_VEMPTY = 9,  // +stage (2)
  QB_SFULL = 11,
  QB_DPFULL = 12,
  QB_SFREE = 13,   // S read into registers (4 warps)
  QB_DPFREE = 14,  // dP read (4 warps)
  QB_DSREADY = 15, // dS written to TMEM (4 warps)
  QB_DQDONE = 16,  // dQ MMA done: dS columns free
  QB_FINAL = 17,
  QB_OFREE = 18,   // O_i read (4 warps): K stage 2 may be loaded
  QB_O = 19,       // O_i landed (in K stage 2)
  QB_N = 20
};

// WIN: causal sliding window (see the dK/dV kernel): query tile i meets only
// the key tiles its window reaches.
template <int D, bool BF16, bool WIN>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                     const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_o,
                     const float* __restrict__ lse, float* __restrict__ Drow, int heads,
                     int head_group, int Hq, int Hkv, int N,
                     int causal, int window, float scale, int* err) {
  using L = DqSmem<D>;
  constexpr int kAtoms = D / 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + QB_N);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int T = (N + kBlk - 1) / kBlk;
  // Groups of query heads whose K and V stay in L2; within a group the query
  // tiles with the most key tiles under causal masking (large i) first.
  const WorkItem wi = grouped_heavy_first(blockIdx.x, heads, T, head_group);
  const int i = T - 1 - wi.rank;
  const int bhq = wi.head;  // b * Hq + hq
  const int b = bhq / Hq;
  const int hq = bhq % Hq;
  const int kvh = b * Hkv + hq / (Hq / Hkv);
  const int j_lo = WIN ? window_first_tile(i, window) : 0;  // first key tile visited
  const int n_j = causal ? i + 1 - j_lo : T;
  constexpr uint32_t kColDQ = 0, kColS = 128, kColDP = 256, kColDS = 384;

  if (threadIdx.x == 0) {
    for (int k = 0; k < QB_N; ++k) {
      uint32_t cnt = 1;
      if (k == QB_SFREE || k == QB_DPFREE || k == QB_DSREADY || k == QB_OFREE) cnt = 4;
      mbar_init(&bar[k], cnt);
    }
    *abort_flag = 0;  // the producer checks the error word once its first loads are issued
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      tma_prefetch_desc(&tm_o);
      const uint64_t pol_q = l2_policy_evict_first();
      const uint64_t pol_kv = l2_policy_evict_last();
      mbar_expect_tx(&bar[QB_Q], 2 * L::kTile);
      for (int a = 0; a < kAtoms; ++a) {
        tma_load_3d(smem + L::kQ + a * kAtomBytes, &tm_q, &bar[QB_Q], a * 64, i * kBlk, bhq, pol_q);
        tma_load_3d(smem + L::kdO + a * kAtomBytes, &tm_do, &bar[QB_Q], a * 64, i * kBlk, bhq, pol_q);
      }
      int kissued = 0, vissued = 0;
      bool o_issued = false;
      for (int jj = 0; jj < n_j; ++jj) {
        const int sk = jj % kDqKStages;
        const uint32_t pk = (jj / kDqKStages) & 1;
        const int sv = jj & 1;
        const uint32_t pv = (jj >> 1) & 1;
        if (jj == 2 && !mbar_wait(&bar[QB_OFREE], 0, abort_flag, err)) break;
        if (!mbar_wait(&bar[QB_KEMPTY + sk], pk ^ 1, abort_flag, err)) break;
        mbar_expect_tx(&bar[QB_KFULL + sk], L::kTile);
        for (int a = 0; a < kAtoms; ++a)
          tma_load_3d(smem + L::kK + sk * L::kTile + a * kAtomBytes, &tm_k, &bar[QB_KFULL + sk],
                      a * 64, (j_lo + jj) * kBlk, kvh, pol_kv);
        kissued = jj + 1;
        if (!mbar_wait(&bar[QB_VEMPTY + sv], pv ^ 1, abort_flag, err)) break;
        mbar_expect_tx(&bar[QB_VFULL + sv], L::kTile);
        for (int a = 0; a < kAtoms; ++a)
          tma_load_3d(smem + L::kV + sv * L::kTile + a * kAtomBytes, &tm_v, &bar[QB_VFULL + sv],
                      a * 64, (j_lo + jj) * kBlk, kvh, pol_kv);
        vissued = jj + 1;
        if (jj == 0) {
          // O_i goes to K stage 2, idle until K_2: the compute warps read it
          // (for D) before that stage is loaded.
          mbar_expect_tx(&bar[QB_O], L::kTile);
          for (int a = 0; a < kAtoms; ++a)
            tma_load_3d(smem + L::kK + 2 * L::kTile + a * kAtomBytes, &tm_o, &bar[QB_O], a * 64,
                        i * kBlk, bhq, pol_q);
          o_issued = true;
          // Read only now, off the path to the first MMA (see the dK/dV kernel).
          if (*reinterpret_cast<volatile int*>(err) != kDevErrNone) *abort_flag = 1;
        }
      }
      if (*abort_flag) {
        drain_wait(&bar[QB_Q], 0);
        if (o_issued) drain_wait(&bar[QB_O], 0);
        for (int jj = (kissued > kDqKStages ? kissued - kDqKStages : 0); jj < kissued; ++jj)
          drain_wait(&bar[QB_KFULL + jj % kDqKStages], (jj / kDqKStages) & 1);
        for (int jj = (vissued > 2 ? vissued - 2 : 0); jj < vissued; ++jj)
          drain_wait(&bar[QB_VFULL + (jj & 1)], (jj >> 1) & 1);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_f16(kBlk, kBlk, BF16, false, false);  // S, dP
      constexpr uint32_t kIdQ = idesc_f16(kBlk, D, BF16, false, true);      // dQ
      constexpr uint64_t kStageStep = L::kTile >> 4;  // one stage further, in descriptor units
      const uint64_t dq0 = kmajor_desc(smem_u32(smem + L::kQ), 0);
      const uint64_t ddo0 = kmajor_desc(smem_u32(smem + L::kdO), 0);
      const uint64_t dk0 = kmajor_desc(smem_u32(smem + L::kK), 0);
      const uint64_t dv0 = kmajor_desc(smem_u32(smem + L::kV), 0);
      const uint64_t mk0 = mnmajor_desc(smem_u32(smem + L::kK), 0);
      auto issue_s = [&](int stk) {  // S = Q_i K_j^T
        const uint64_t kd = dk0 + stk * kStageStep;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          mma_ss(tmem + kColS, kmajor_step(dq0, ks), kmajor_step(kd, ks), kIdS, ks > 0);
        mma_commit(&bar[QB_SFULL]);
      };
      auto issue_dp = [&](int stv) {  // dP = dO_i V_j^T; V_j is free again once this completes
        const uint64_t vd = dv0 + stv * kStageStep;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          mma_ss(tmem + kColDP, kmajor_step(ddo0, ks), kmajor_step(vd, ks), kIdS, ks > 0);
        mma_commit(&bar[QB_DPFULL]);
        mma_commit(&bar[QB_VEMPTY + stv]);
      };
      bool ok = mbar_wait(&bar[QB_Q], 0, abort_flag, err) &&
                mbar_wait(&bar[QB_KFULL], 0, abort_flag, err);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        ok = mbar_wait(&bar[QB_VFULL], 0, abort_flag, err);
        if (ok) {
          tc_fence_after();
          issue_dp(0);
        }
      }
      for (int jj = 0; ok && jj < n_j; ++jj) {
        const int stk = jj % kDqKStages;
        if (jj + 1 < n_j) {
          const int stk1 = (jj + 1) % kDqKStages;
          const uint32_t phk1 = ((jj + 1) / kDqKStages) & 1;
          const int stv1 = (jj + 1) & 1;
          const uint32_t phv1 = ((jj + 1) >> 1) & 1;
          // S(j+1) may start once S(j) has been read out of TMEM; dP(j+1) once dP(j) has.
          if (!(ok = mbar_wait(&bar[QB_KFULL + stk1], phk1, abort_flag, err))) break;
          if (!(ok = mbar_wait(&bar[QB_SFREE], jj & 1, abort_flag, err))) break;
          tc_fence_after();
          issue_s(stk1);
          if (!(ok = mbar_wait(&bar[QB_VFULL + stv1], phv1, abort_flag, err))) break;
          if (!(ok = mbar_wait(&bar[QB_DPFREE], jj & 1, abort_flag, err))) break;
          tc_fence_after();
          issue_dp(stv1);
        }
        // dQ += dS K_j   (dS: 16-bit pairs in its own TMEM columns; K_j as an MN-major B)
        if (!(ok = mbar_wait(&bar[QB_DSREADY], jj & 1, abort_flag, err))) break;
        tc_fence_after();
        const uint64_t km = mk0 + stk * kStageStep;
#pragma unroll
        for (int ks = 0; ks < kBlk / 16; ++ks)
          mma_ts(tmem + kColDQ, tmem + kColDS + ks * 8, mnmajor_step(km, ks), kIdQ,
                 (jj > 0 || ks > 0) ? 1u : 0u);
        mma_commit(&bar[QB_DQDONE]);
        mma_commit(&bar[QB_KEMPTY + stk]);
      }
      mma_commit(&bar[QB_FINAL]);
      drain_wait(&bar[QB_FINAL], 0);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ compute: P, dS
    const int t = threadIdx.x;  // query row within the tile
    const int q = i * kBlk + t;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tS = tmem + lane_off + kColS;
    const uint32_t tP = tmem + lane_off + kColDP;
    const uint32_t tDS = tmem + lane_off + kColDS;
    const float sl2 = scale * kLog2e;
    const size_t g = static_cast<size_t>(bhq) * N + q;
    // Padding rows (q >= N) get LSE = +inf: P and dS are exactly 0 there.
    const float lse2 = (q < N) ? lse[g] * kLog2e : INFINITY;
    // D_q = sum_c dO_qc O_qc from the O_i and dO_i tiles the producer staged,
    // computed once the first P is done (while the first dP MMA runs) and
    // written out for the dK/dV kernel, which runs after this one.
    auto row_d = [&]() -> float {
      float dq_d = 0.f;
      if (q < N) {
        const uint8_t* dorow = smem + L::kdO + t * 128;
        const uint8_t* orow = smem + L::kK + 2 * L::kTile + t * 128;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {  // 16-byte chunk c of the row (128-byte swizzle)
          const int off = (c / 8) * kAtomBytes + (((c % 8) ^ (t & 7)) * 16);
          const uint4 w = *reinterpret_cast<const uint4*>(dorow + off);
          const uint4 ov = *reinterpret_cast<const uint4*>(orow + off);
          const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w};
          const uint32_t dw[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 x = unpack2<BF16>(ow[e]);
            const float2 y = unpack2<BF16>(dw[e]);
            acc[e] = fmaf(x.x, y.x, acc[e]);
            acc[e] = fmaf(x.y, y.y, acc[e]);
          }
        }
        dq_d = (acc[0] + acc[1]) + (acc[2] + acc[3]);
        Drow[g] = dq_d;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[QB_OFREE]);  // generic reads of K stage 2 done
      return dq_d;
    };
    uint64_t negd2 = 0;
    bool ok = true;
    for (int jj = 0; ok && jj < n_j; ++jj) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bar[QB_SFULL], jj & 1, abort_flag, err));
      if (!ok) break;
      tc_fence_after();
      float p[kBlk];
      {
        uint32_t sv[kBlk];
#pragma unroll
        for (int c = 0; c < kBlk; c += 32) tmem_ld32(tS + c, sv + c);
        tmem_ld_wait();
        reg_fence<kBlk>(sv);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[QB_SFREE]);
        const uint64_t sl2x2 = f2_pack(sl2, sl2);
        const uint64_t nl2 = f2_pack(-lse2, -lse2);
#pragma unroll
        for (int c = 0; c < kBlk; c += 2) {
          float a0, a1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sl2x2, nl2),
                    a0, a1);
          p[c] = ex2_approx(a0);
          p[c + 1] = ex2_approx(a1);
        }
      }
      const int kt = j_lo + jj;  // key tile
      if (causal && kt == i) {  // key kt*128 + c after query i*128 + t is masked
#pragma unroll
        for (int c = 0; c < kBlk; ++c)
          if (c > t) p[c] = 0.f;
      }
      if (WIN && kt * kBlk + window <= i * kBlk + kBlk - 1) {
        // The window's edge crosses this tile: key kt*128 + c is visible to
        // query i*128 + t iff it is greater than i*128 + t - window.
        const int lim = (i - kt) * kBlk + t - window;
#pragma unroll
        for (int c = 0; c < kBlk; ++c)
          if (c <= lim) p[c] = 0.f;
      }
      if (jj == 0) {
        // dO_i (with Q_i) and O_i have landed.
        ok = __all_sync(0xffffffffu, mbar_wait(&bar[QB_Q], 0, abort_flag, err) &&
                                         mbar_wait(&bar[QB_O], 0, abort_flag, err));
        if (!ok) break;
        const float dd = row_d();
        negd2 = f2_pack(-dd, -dd);
      }
      ok = __all_sync(0xffffffffu, mbar_wait(&bar[QB_DPFULL], jj & 1, abort_flag, err));
      // dS(j) overwrites the columns dQ(j-1) reads.
      if (ok && jj > 0)
        ok = __all_sync(0xffffffffu, mbar_wait(&bar[QB_DQDONE], (jj - 1) & 1, abort_flag, err));
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int h = 0; h < kBlk; h += 64) {  // two TMEM round trips of 64 columns
        uint32_t dpv[64];
        tmem_ld32(tP + h, dpv);
        tmem_ld32(tP + h + 32, dpv + 32);
        tmem_ld_wait();
        reg_fence<64>(dpv);
        if (h + 64 == kBlk) {  // dP(j) fully read: dP(j+1) may overwrite it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar[QB_DPFREE]);
        }
#pragma unroll
        for (int c = 0; c < 64; c += 32) {
          uint32_t dsw[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float g0, g1;
            f2_unpack(f2_mul(f2_pack(p[h + c + 2 * e], p[h + c + 2 * e + 1]),
                             f2_add(f2_pack(__uint_as_float(dpv[c + 2 * e]),
                                            __uint_as_float(dpv[c + 2 * e + 1])),
                                    negd2)),
                      g0, g1);
            dsw[e] = pack2<BF16>(g0, g1);
          }
          tmem_st16(tDS + (h + c) / 2, dsw);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[QB_DSREADY]);
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bar[QB_FINAL], 0, abort_flag, err));
    if (ok) {
      // Q's last reader, S(n_j - 1), has completed: dQ is staged in its place.
      tc_fence_after();
      uint8_t* st_dq = smem + L::kQ;
      stage_row_from_tmem<D, BF16>(tmem + lane_off + kColDQ, st_dq, t, scale);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && i * kBlk + 32 * warp < N) {
#pragma unroll
        for (int a = 0; a < kAtoms; ++a)
          tma_store_3d(&tm_dq, st_dq + a * kAtomBytes + warp * 4096, a * 64, i * kBlk + 32 * warp, bhq);
        bulk_commit_group();
        bulk_wait_read_all();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool BF16, bool WIN>
cudaError_t launch_bwd_t(const AttnShape& s, const BwdArgs& a, cudaStream_t stream) {
  const int T = (s.N + kBlk - 1) / kBlk;
  auto kdkdv = fa_bwd_dkdv_kernel<D, BF16, WIN>;
  constexpr int smem_kv = DkdvSmem<D, false>::kAlloc;
  const int slot = (WIN ? 4 : 0) + (D == 64 ? 0 : 2) + (BF16 ? 1 : 0);
  cudaError_t e;
  if ((e = set_smem_once(reinterpret_cast<const void*>(kdkdv), smem_kv, 8 + slot)) != cudaSuccess)
    return e;
  auto kdq = fa_bwd_dq_kernel<D, BF16, WIN>;
  constexpr int smem_q = DqSmem<D>::kAlloc;
  if ((e = set_smem_once(reinterpret_cast<const void*>(kdq), smem_q, 16 + slot)) != cudaSuccess)
    return e;

  // The dQ kernel runs first: besides dQ it writes D = rowsum(dO o O), which
  // the dK/dV kernel reads.
  if (a.ev_before_dq && (e = cudaEventRecord(a.ev_before_dq, stream)) != cudaSuccess) return e;
  kdq<<<dim3(static_cast<unsigned>(T * s.B * s.Hq)), kThreads, smem_q, stream>>>(
      a.tm_q, a.tm_k, a.tm_v, a.tm_do, a.tm_dq, a.tm_o, a.lse, a.D,
      s.B * s.Hq, l2_head_group(4L * s.N * D), s.Hq, s.Hkv, s.N, s.causal, s.window, s.scale, a.err);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (a.ev_before_dkdv && (e = cudaEventRecord(a.ev_before_dkdv, stream)) != cudaSuccess) return e;
  kdkdv<<<dim3(static_cast<unsigned>(T * s.B * s.Hkv)), kDkdvThreads, smem_kv, stream>>>(
      a.tm_q, a.tm_k, a.tm_v, a.tm_do, a.tm_dk, a.tm_dv, a.lse, a.D, s.B * s.Hkv,
      l2_head_group(4L * s.N * D * (s.Hq / s.Hkv)), s.Hq, s.Hkv, s.N, s.causal, s.window, s.scale,
      a.err);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (a.ev_after_dkdv && (e = cudaEventRecord(a.ev_after_dkdv, stream)) != cudaSuccess) return e;
  return cudaSuccess;
}

}  // namespace

size_t backward_smem_bytes(int d) {
  return d == 64 ? DkdvSmem<64, false>::kAlloc : DkdvSmem<128, false>::kAlloc;
}

cudaError_t launch_backward(const AttnShape& s, const BwdArgs& a, cudaStream_t stream) {
  if (s.window > 0) {  // causal sliding window
    if (s.d == 64)
      return s.bf16 ? launch_bwd_t<64, true, true>(s, a, stream) : launch_bwd_t<64, false, true>(s, a, stream);
    return s.bf16 ? launch_bwd_t<128, true, true>(s, a, stream) : launch_bwd_t<128, false, true>(s, a, stream);
  }
  if (s.d == 64)
    return s.bf16 ? launch_bwd_t<64, true, false>(s, a, stream) : launch_bwd_t<64, false, false>(s, a, stream);
  return s.bf16 ? launch_bwd_t<128, true, false>(s, a, stream) : launch_bwd_t<128, false, false>(s, a, stream);
}

}  // namespace fa
