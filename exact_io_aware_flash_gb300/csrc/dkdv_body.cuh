// The key-tile pass of the backward, shared by the two backward algorithms:
//
//   ONEPASS = false  (fa_bwd_dkdv_kernel, deterministic two-pass backward)
//     one CTA per (KV head, 128-key tile j), looping over the KV head's query
//     heads and query tiles i (causal: i >= j), in the transposed orientation
//     so the key tile owns the TMEM lanes and dK, dV accumulate in TMEM:
//       S^T  = K_j Q_i^T,  dP^T = V_j dO_i^T           (SMEM x SMEM)
//       P^T, dS^T                                      (compute warps)
//       dV  += P^T dO_i,   dK  += dS^T Q_i             (TMEM A operand)
//     dQ comes from a separate query-tile pass.
//
//   ONEPASS = true   (fa_bwd_onepass_kernel, the atomic backward)
//     the same loop, plus this key tile's share of dQ_i on every iteration:
//       dS^T -> shared memory (one 128 x 128 16-bit tile)
//       dK  += dS^T Q_i                                (SMEM x SMEM, K-major dS^T)
//       dQ_i partial = dS K_j                          (SMEM x SMEM, MN-major dS)
//     four more warps read the dQ partial out of TMEM and add it into an fp32
//     accumulator in global memory (red.global.add), so dQ_i collects the sum
//     over key tiles from many CTAs in no fixed order: 5 instead of 7
//     N x N x d products, and a nondeterministic summation order for dQ.
//     ("FlashAttention Primer: IO-Aware Attention, from FA1 to FA4", section
//     "Backward pass: recomputation instead of storage": the default backward
//     accumulates dQ across thread blocks with atomic adds.)
//
// Warps: 0-3 compute (thread t owns key row t of the tile, TMEM lane t).
//   two-pass (192 threads): 4 the TMA producer, 5 the single-thread MMA issuer
//     and TMEM allocator.
//   one-pass (384 threads, three whole warpgroups so registers can move between
//     them): 4-7 the dQ drain (warp w reads TMEM lanes 32 * (w mod 4) .. + 31),
//     8 the producer, 9 the issuer, 10-11 idle.  Ten warps would cap every
//     thread at 168 registers (three warps share a sub-partition's 16K); with
//     twelve, the compute warpgroup takes 232 from the control warpgroup.
#pragma once

#include "bwd_common.cuh"

namespace fa {
namespace bwd {

constexpr int kDkdvThreads = 192;
constexpr int kOnePassThreads = 384;
// Registers per thread after reallocation.  setmaxnreg.inc draws on the pool
// the CTA was launched with (384 threads x 168), so the shares must fit in it.
constexpr uint32_t kOnePassRegsCompute = 224;  // warps 0-3
constexpr uint32_t kOnePassRegsDrain = 176;    // warps 4-7 (a whole 32 x d fp32 slab in registers)
constexpr uint32_t kOnePassRegsControl = 104;  // warps 8-11
static_assert(128 * (kOnePassRegsCompute + kOnePassRegsDrain + kOnePassRegsControl) <=
                  kOnePassThreads * 168,
              "register split exceeds the launch pool");

template <int D, bool ONEPASS>
struct DkdvSmem {
  static constexpr int kTile = kBlk * D * 2;
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTile;
  static constexpr int kQ = kV + kTile;         // 2 stages
  static constexpr int kdO = kQ + 2 * kTile;    // 2 stages
  // ONEPASS: the 128 x 128 16-bit dS tile of an iteration.  With d = 128 it
  // overwrites that iteration's dO_i stage once dV and dP^T have read it
  // (a separate 32 KB tile would not fit in 227 KB); with d = 64 the dO stage
  // is too small and the tile has its own region.
  static constexpr int kdS = kdO + 2 * kTile;
  static constexpr int kdSBytes = (ONEPASS && D == 64) ? kBlk * kBlk * 2 : 0;
  static constexpr int kLse = kdS + kdSBytes;   // 2 stages x 128 floats: -LSE * log2(e)
  static constexpr int kDrow = kLse + 1024;     // 2 stages x 128 floats: -D
  static constexpr int kBar = kDrow + 1024;
  static constexpr int kBytes = kBar + 256;
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr int ds_tile(int st) { return D == 128 ? kdO + st * kTile : kdS; }
};

enum DkdvBars {
  KB_KV = 0,
  KB_QFULL = 1,   // +stage: Q_i, dO_i (TMA) and LSE_i, D_i (32 producer lanes)
  KB_QEMPTY = 3,  // +stage
  KB_SFULL = 5,   // S^T in TMEM
  KB_DPFULL = 6,  // dP^T in TMEM
  KB_PREADY = 7,  // P^T written to TMEM (4 warps)
  KB_DSREADY = 8, // dS^T written to TMEM (two-pass) or to shared memory (one-pass) (4 warps)
  KB_DVDONE = 9,  // dV MMA done: S^T columns free
  KB_DKDONE = 10, // dK MMA done: dP^T columns free (two-pass)
  KB_FINAL = 11,
  KB_DQFULL = 12, // one-pass: the dQ partial is in the dP^T columns
  KB_DQFREE = 13, // one-pass: the 4 drain warps have read it
  KB_N = 14
};

// WIN: causal sliding window of `window` keys (key k visible to query q iff
// q - window < k <= q): key tile j meets only the query tiles its keys are
// visible to, and the window's edge is masked element-wise.
// dq_acc (ONEPASS only): [B*Hq][N][D] fp32, zero on entry, receives the
// unscaled sum over key tiles of dS K.
template <int D, bool BF16, bool WIN, bool ONEPASS>
__device__ __forceinline__ void dkdv_body(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                                          const CUtensorMap* tm_v, const CUtensorMap* tm_do,
                                          const CUtensorMap* tm_dk, const CUtensorMap* tm_dv,
                                          const float* __restrict__ lse, const float* __restrict__ Drow,
                                          float* __restrict__ dq_acc, int heads, int head_group, int Hq,
                                          int Hkv, int N, int causal, int window, float scale, int* err) {
  using L = DkdvSmem<D, ONEPASS>;
  constexpr int kAtoms = D / 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + KB_N);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int T = (N + kBlk - 1) / kBlk;
  // Groups of KV heads whose Q and dO stay in L2; within a group the key tiles
  // with the most work under causal masking (small j) first.
  const WorkItem wi = grouped_heavy_first(blockIdx.x, heads, T, head_group);
  const int j = wi.rank;
  const int bkv = wi.head;  // b * Hkv + hkv
  const int b = bkv / Hkv;
  const int hkv = bkv % Hkv;
  const int group = Hq / Hkv;
  const int i0 = causal ? j : 0;
  // Last query tile that sees a key of tile j: keys up to j*128 + 127 are
  // visible to queries up to j*128 + 126 + window.
  int i_last = T - 1;
  if (WIN) {
    const int qmax = (j * kBlk + kBlk - 2 + window) / kBlk;
    i_last = qmax < T - 1 ? qmax : T - 1;
  }
  const int n_i = i_last - i0 + 1;
  const int n_it = group * n_i;
  // The one-pass dQ partial reuses the dP^T columns: they are free once the
  // compute warps have turned dP^T into dS^T in shared memory.
  constexpr uint32_t kColDV = 0, kColDK = 128, kColS = 256, kColDP = 384, kColDQ = kColDP;
  constexpr int kProducer = ONEPASS ? 8 : 4;
  constexpr int kIssuer = ONEPASS ? 9 : 5;

  if (threadIdx.x == 0) {
    for (int i = 0; i < KB_N; ++i) {
      uint32_t cnt = 1;
      if (i == KB_QFULL || i == KB_QFULL + 1) cnt = 33;
      if (i == KB_PREADY || i == KB_DSREADY || i == KB_DQFREE) cnt = 4;
      mbar_init(&bar[i], cnt);
    }
    *abort_flag = 0;  // the producer checks the error word once its first loads are issued
    fence_mbar_init();
  }
  if (warp == kIssuer) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // The roles, dispatched below (the lambdas are called once and inlined).
  auto producer = [&]() {
    // ------------------------------------------------------------ producer
    float* s_lse = reinterpret_cast<float*>(smem + L::kLse);
    float* s_d = reinterpret_cast<float*>(smem + L::kDrow);
    int issued = 0;
    if (lane == 0) {
      tma_prefetch_desc(tm_q);
      tma_prefetch_desc(tm_k);
      tma_prefetch_desc(tm_v);
      tma_prefetch_desc(tm_do);
      const uint64_t pol = l2_policy_evict_first();
      mbar_expect_tx(&bar[KB_KV], 2 * L::kTile);
      for (int a = 0; a < kAtoms; ++a) {
        tma_load_3d(smem + L::kK + a * kAtomBytes, tm_k, &bar[KB_KV], a * 64, j * kBlk, bkv, pol);
        tma_load_3d(smem + L::kV + a * kAtomBytes, tm_v, &bar[KB_KV], a * 64, j * kBlk, bkv, pol);
      }
    }
    const uint64_t pol_q = l2_policy_evict_last();
    for (int it = 0; it < n_it; ++it) {
      const int hq = hkv * group + it / n_i;
      const int i = i0 + it % n_i;
      const int bhq = b * Hq + hq;
      const int st = it & 1;
      bool ok = true;
      if (lane == 0) {
        ok = mbar_wait(&bar[KB_QEMPTY + st], ((it >> 1) & 1) ^ 1, abort_flag, err);
        if (ok) {
          mbar_expect_tx(&bar[KB_QFULL + st], 2 * L::kTile);
          for (int a = 0; a < kAtoms; ++a) {
            tma_load_3d(smem + L::kQ + st * L::kTile + a * kAtomBytes, tm_q, &bar[KB_QFULL + st],
                        a * 64, i * kBlk, bhq, pol_q);
            tma_load_3d(smem + L::kdO + st * L::kTile + a * kAtomBytes, tm_do, &bar[KB_QFULL + st],
                        a * 64, i * kBlk, bhq, pol_q);
          }
          issued = it + 1;
          // A CTA that starts after another one raised the error word stops at
          // its next wait; reading the word only now keeps its latency off the
          // path to the first MMA.
          if (it == 0 && *reinterpret_cast<volatile int*>(err) != kDevErrNone) *abort_flag = 1;
        }
      }
      if (__shfl_sync(0xffffffffu, ok ? 1 : 0, 0) == 0) break;  // also orders the stage reuse
      // -LSE (as log2) and -D of the tile's 128 query rows, negated so the
      // compute warps add them; padding rows get LSE = +inf so their recomputed
      // probabilities are exactly 0.
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = lane * 4 + e;
        const int qrow = i * kBlk + r;
        const size_t g = static_cast<size_t>(bhq) * N + qrow;
        const bool in = qrow < N;
        s_lse[st * 128 + r] = in ? -lse[g] * kLog2e : -INFINITY;
        s_d[st * 128 + r] = in ? -Drow[g] : 0.f;
      }
      mbar_arrive(&bar[KB_QFULL + st]);
    }
    if (lane == 0 && *abort_flag) {
      drain_wait(&bar[KB_KV], 0);
      for (int it = (issued > 2 ? issued - 2 : 0); it < issued; ++it)
        drain_wait(&bar[KB_QFULL + (it & 1)], (it >> 1) & 1);
    }
  };
  auto issuer = [&]() {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_f16(kBlk, kBlk, BF16, false, false);  // S^T, dP^T
      constexpr uint32_t kIdKV = idesc_f16(kBlk, D, BF16, false, true);     // dV, dK
      constexpr uint32_t kIdQ = idesc_f16(kBlk, D, BF16, true, true);       // dQ partial
      constexpr uint64_t kStageStep = L::kTile >> 4;  // one stage further, in descriptor units
      const uint64_t dk0 = kmajor_desc(smem_u32(smem + L::kK), 0);
      const uint64_t dv0 = kmajor_desc(smem_u32(smem + L::kV), 0);
      const uint64_t dq0 = kmajor_desc(smem_u32(smem + L::kQ), 0);
      const uint64_t ddo0 = kmajor_desc(smem_u32(smem + L::kdO), 0);
      const uint64_t mq0 = mnmajor_desc(smem_u32(smem + L::kQ), 0);
      const uint64_t mdo0 = mnmajor_desc(smem_u32(smem + L::kdO), 0);
      // one-pass: K_j as the MN-major B of dQ; the dS tile (rows = keys, 64-query
      // atoms) as the MN-major A of dQ = dS K_j and the K-major A of dK += dS^T Q_i
      [[maybe_unused]] const uint64_t mk0 = mnmajor_desc(smem_u32(smem + L::kK), 0);
      [[maybe_unused]] const uint64_t dsm0 = mnmajor_desc(smem_u32(smem + L::ds_tile(0)), 0);
      [[maybe_unused]] const uint64_t dsk0 = kmajor_desc(smem_u32(smem + L::ds_tile(0)), 0);
      constexpr uint64_t kDsStep = D == 128 ? kStageStep : 0;  // d = 64: one tile for both stages
      auto issue_s = [&](int st) {  // S^T = K_j Q_i^T
        const uint64_t qd = dq0 + st * kStageStep;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          mma_ss(tmem + kColS, kmajor_step(dk0, ks), kmajor_step(qd, ks), kIdS, ks > 0);
        mma_commit(&bar[KB_SFULL]);
      };
      auto issue_dp = [&](int st) {  // dP^T = V_j dO_i^T
        const uint64_t dd = ddo0 + st * kStageStep;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          mma_ss(tmem + kColDP, kmajor_step(dv0, ks), kmajor_step(dd, ks), kIdS, ks > 0);
        mma_commit(&bar[KB_DPFULL]);
      };
      bool ok = mbar_wait(&bar[KB_KV], 0, abort_flag, err) &&
                mbar_wait(&bar[KB_QFULL], 0, abort_flag, err);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        issue_dp(0);
      }
      // Issue order per iteration: dV(it), S^T(it+1), then
      //   two-pass: dK(it), dP^T(it+1)
      //   one-pass: dQ(it), dK(it), dP^T(it+1)
      // S^T(it+1) needs only dV(it) finished (it overwrites the P^T columns), so
      // the next P^T phase can start while this iteration's dS^T is still being
      // computed.
      for (int it = 0; ok && it < n_it; ++it) {
        const int st = it & 1;
        const uint64_t qm = mq0 + st * kStageStep;
        const uint64_t dom = mdo0 + st * kStageStep;
        const bool more = it + 1 < n_it;
        const int st1 = (it + 1) & 1;
        // dV += P^T dO_i   (P^T: 16-bit pairs over the first half of the S^T columns)
        if (!(ok = mbar_wait(&bar[KB_PREADY], it & 1, abort_flag, err))) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < kBlk / 16; ++ks)
          mma_ts(tmem + kColDV, tmem + kColS + ks * 8, mnmajor_step(dom, ks), kIdKV,
                 (it > 0 || ks > 0) ? 1u : 0u);
        mma_commit(&bar[KB_DVDONE]);
        if (more) {
          if (!(ok = mbar_wait(&bar[KB_QFULL + st1], ((it + 1) >> 1) & 1, abort_flag, err))) break;
          if (!(ok = mbar_wait(&bar[KB_DVDONE], it & 1, abort_flag, err))) break;
          tc_fence_after();
          issue_s(st1);
        }
        if (!(ok = mbar_wait(&bar[KB_DSREADY], it & 1, abort_flag, err))) break;
        tc_fence_after();
        if constexpr (ONEPASS) {
          const uint64_t dsm = dsm0 + st * kDsStep;
          const uint64_t dsk = dsk0 + st * kDsStep;
#pragma unroll
          for (int ks = 0; ks < kBlk / 16; ++ks)
            mma_ss(tmem + kColDQ, mnmajor_step(dsm, ks), mnmajor_step(mk0, ks), kIdQ, ks > 0);
          mma_commit(&bar[KB_DQFULL]);
#pragma unroll
          for (int ks = 0; ks < kBlk / 16; ++ks)
            mma_ss(tmem + kColDK, kmajor_step(dsk, ks), mnmajor_step(qm, ks), kIdKV,
                   (it > 0 || ks > 0) ? 1u : 0u);
          mma_commit(&bar[KB_QEMPTY + st]);  // Q_i, dO_i and the dS tile over it are read
          if (more) {
            // dP^T(it+1) overwrites the dQ partial the drain warps read.
            if (!(ok = mbar_wait(&bar[KB_DQFREE], it & 1, abort_flag, err))) break;
            tc_fence_after();
            issue_dp(st1);
          }
        } else {
          // dK += dS^T Q_i   (dS^T: 16-bit pairs over the first half of the dP^T columns)
#pragma unroll
          for (int ks = 0; ks < kBlk / 16; ++ks)
            mma_ts(tmem + kColDK, tmem + kColDP + ks * 8, mnmajor_step(qm, ks), kIdKV,
                   (it > 0 || ks > 0) ? 1u : 0u);
          mma_commit(&bar[KB_DKDONE]);
          mma_commit(&bar[KB_QEMPTY + st]);
          if (more) {
            // dP^T(it+1) overwrites the dS^T columns dK(it) reads.
            if (!(ok = mbar_wait(&bar[KB_DKDONE], it & 1, abort_flag, err))) break;
            tc_fence_after();
            issue_dp(st1);
          }
        }
      }
      mma_commit(&bar[KB_FINAL]);
      drain_wait(&bar[KB_FINAL], 0);
    }
  };
  auto compute = [&]() {
    // ------------------------------------------------------------ compute: P^T, dS^T
    const int t = threadIdx.x;  // key row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tS = tmem + lane_off + kColS;
    const uint32_t tP = tmem + lane_off + kColDP;
    const float sl2 = scale * kLog2e;
    const uint64_t sl2x2 = f2_pack(sl2, sl2);
    const float* s_lse = reinterpret_cast<const float*>(smem + L::kLse);
    const float* s_d = reinterpret_cast<const float*>(smem + L::kDrow);
    // One-pass: a key row past N (zero K and V rows from the TMA fill) must
    // contribute nothing to dQ, so its probabilities are zeroed; without a
    // causal mask it meets real queries, whose LSE can make exp(0 - LSE) huge.
    const bool key_pad = ONEPASS && j * kBlk + t >= N;
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int i = i0 + it % n_i;
      const int st = it & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(&bar[KB_SFULL], it & 1, abort_flag, err) &&
                                       mbar_wait(&bar[KB_QFULL + st], (it >> 1) & 1, abort_flag, err));
      if (!ok) break;
      tc_fence_after();
      const bool diag = causal && (i == j);
      const float* lse2 = s_lse + st * 128;
      const float* dd = s_d + st * 128;
      // P^T row t: exp2(s * scale*log2(e) - LSE_q*log2(e)); query q before key t is masked.
      float p[kBlk];
#pragma unroll
      for (int h = 0; h < kBlk; h += 64) {  // two halves keep the live registers below the cap
        uint32_t sv[64];
        tmem_ld32(tS + h, sv);
        tmem_ld32(tS + h + 32, sv + 32);
        tmem_ld_wait();
        reg_fence<64>(sv);
#pragma unroll
        for (int c = 0; c < 64; c += 4) {
          const float4 l4 = lds128_ordered(lse2 + h + c);  // -LSE_q * log2(e)
          float a0, a1, a2, a3;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sl2x2,
                           f2_pack(l4.x, l4.y)),
                    a0, a1);
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[c + 2]), __uint_as_float(sv[c + 3])), sl2x2,
                           f2_pack(l4.z, l4.w)),
                    a2, a3);
          p[h + c] = ex2_approx(a0);
          p[h + c + 1] = ex2_approx(a1);
          p[h + c + 2] = ex2_approx(a2);
          p[h + c + 3] = ex2_approx(a3);
        }
      }
      if (diag) {
#pragma unroll
        for (int c = 0; c < kBlk; ++c)
          if (c < t) p[c] = 0.f;
      }
      if (WIN && (i - j) * kBlk + kBlk - 1 >= window) {
        // The window's edge crosses this tile: query i*128 + c sees key
        // j*128 + t iff i*128 + c - window < j*128 + t.
        const int lim_c = (j - i) * kBlk + t + window;
#pragma unroll
        for (int c = 0; c < kBlk; ++c)
          if (c >= lim_c) p[c] = 0.f;
      }
      if (key_pad) {
#pragma unroll
        for (int c = 0; c < kBlk; ++c) p[c] = 0.f;
      }
#pragma unroll
      for (int c = 0; c < kBlk; c += 32) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) pk[e] = pack2<BF16>(p[c + 2 * e], p[c + 2 * e + 1]);
        tmem_st16(tS + c / 2, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[KB_PREADY]);
      // dS^T = P^T o (dP^T - D_q), chunk by chunk.
      ok = __all_sync(0xffffffffu, mbar_wait(&bar[KB_DPFULL], it & 1, abort_flag, err));
      if (!ok) break;
      tc_fence_after();
      if constexpr (ONEPASS) {
        // Row t of the dS tile in shared memory, 128-byte swizzled like a TMA
        // box: 64-query atoms of 128 rows x 128 bytes, 16-byte chunk c of row t
        // at chunk position c ^ (t mod 8) (conflict-free 16-byte stores).
        // Two halves of 64 queries, so only half the packed row is live; the
        // first half's stores wait (d = 128) until dV(it) has read dO_i.
        uint8_t* row = smem + L::ds_tile(st) + t * 128;
#pragma unroll
        for (int h = 0; h < kBlk; h += 64) {
          uint32_t pk[32];
#pragma unroll
          for (int c = h; c < h + 64; c += 32) {
            uint32_t dpv[32];
            tmem_ld32(tP + c, dpv);
            tmem_ld_wait();
            reg_fence<32>(dpv);
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              const float4 d4 = lds128_ordered(dd + c + e);  // -D_q
              float g0, g1, g2, g3;
              f2_unpack(f2_mul(f2_pack(p[c + e], p[c + e + 1]),
                               f2_add(f2_pack(__uint_as_float(dpv[e]), __uint_as_float(dpv[e + 1])),
                                      f2_pack(d4.x, d4.y))),
                        g0, g1);
              f2_unpack(f2_mul(f2_pack(p[c + e + 2], p[c + e + 3]),
                               f2_add(f2_pack(__uint_as_float(dpv[e + 2]), __uint_as_float(dpv[e + 3])),
                                      f2_pack(d4.z, d4.w))),
                        g2, g3);
              pk[(c - h + e) / 2] = pack2<BF16>(g0, g1);
              pk[(c - h + e) / 2 + 1] = pack2<BF16>(g2, g3);
            }
          }
          if constexpr (D == 128) {
            if (h == 0) {
              ok = __all_sync(0xffffffffu, mbar_wait(&bar[KB_DVDONE], it & 1, abort_flag, err));
              if (!ok) break;
              tc_fence_after();
            }
          }
#pragma unroll
          for (int ch = 0; ch < 8; ++ch)  // 16-byte chunk ch of atom h/64: queries h + 8*ch .. +7
            *reinterpret_cast<uint4*>(row + (h / 64) * kAtomBytes + ((ch ^ (t & 7)) * 16)) =
                make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
        }
        if (!ok) break;
        fence_proxy_async_smem();  // generic stores -> tensor-core (async proxy) reads
        tc_fence_before();         // dP^T reads done before dQ overwrites the columns
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[KB_DSREADY]);
      } else {
        // chunk c's 16-bit pairs land on dP^T columns already read.
#pragma unroll
        for (int c = 0; c < kBlk; c += 32) {
          uint32_t dpv[32];
          tmem_ld32(tP + c, dpv);
          tmem_ld_wait();
          reg_fence<32>(dpv);
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const float4 d4 = lds128_ordered(dd + c + e);  // -D_q
            float g0, g1, g2, g3;
            f2_unpack(f2_mul(f2_pack(p[c + e], p[c + e + 1]),
                             f2_add(f2_pack(__uint_as_float(dpv[e]), __uint_as_float(dpv[e + 1])),
                                    f2_pack(d4.x, d4.y))),
                      g0, g1);
            f2_unpack(f2_mul(f2_pack(p[c + e + 2], p[c + e + 3]),
                             f2_add(f2_pack(__uint_as_float(dpv[e + 2]), __uint_as_float(dpv[e + 3])),
                                    f2_pack(d4.z, d4.w))),
                      g2, g3);
            pk[e / 2] = pack2<BF16>(g0, g1);
            pk[e / 2 + 1] = pack2<BF16>(g2, g3);
          }
          tmem_st16(tP + c / 2, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[KB_DSREADY]);
      }
    }
    // Epilogue: dV and dK leave as 16-bit tiles staged in shared memory and
    // written by TMA stores.  dV is final once the last dV MMA has completed.
    // Two-pass: by then every MMA that reads K or V has completed too (they
    // were issued before it), so dV is staged over K while the last dK MMA
    // still runs, and dK over V once every MMA is done.  One-pass: the last dQ
    // MMA, issued after the last dV, still reads K, so dV goes over V (whose
    // last reader, dP^T, came before) and dK over K.
    const bool store_rows = j * kBlk + 32 * warp < N;  // a store box must start inside the tensor
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bar[KB_DVDONE], (n_it - 1) & 1, abort_flag, err));
    if (ok) {
      tc_fence_after();
      uint8_t* st_dv = smem + (ONEPASS ? L::kV : L::kK);
      stage_row_from_tmem<D, BF16>(tmem + lane_off + kColDV, st_dv, t, 1.0f);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && store_rows) {
#pragma unroll
        for (int a = 0; a < kAtoms; ++a)
          tma_store_3d(tm_dv, st_dv + a * kAtomBytes + warp * 4096, a * 64, j * kBlk + 32 * warp, bkv);
        bulk_commit_group();
      }
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bar[KB_FINAL], 0, abort_flag, err));
    if (ok) {
      tc_fence_after();
      uint8_t* st_dk = smem + (ONEPASS ? L::kK : L::kV);
      stage_row_from_tmem<D, BF16>(tmem + lane_off + kColDK, st_dk, t, scale);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && store_rows) {
#pragma unroll
        for (int a = 0; a < kAtoms; ++a)
          tma_store_3d(tm_dk, st_dk + a * kAtomBytes + warp * 4096, a * 64, j * kBlk + 32 * warp, bkv);
        bulk_commit_group();
      }
    }
    // Shared memory stays allocated until every store issued here has read it.
    if (lane == 0) bulk_wait_read_all();
  };
  [[maybe_unused]] auto drain = [&]() {
    // ------------------------------------------------------------ dQ drain (warps 4-7)
    // Loads in the 16 x 256-bit shape: thread l of the warp holds columns
    // 8r + 2(l mod 4), +1 of rows l/4 and l/4 + 8 of a 16-lane slab, so the
    // four threads of a row cover 32 contiguous bytes and one red.v2
    // instruction updates eight whole 32-byte sectors.
    const int quarter = warp & 3;
    const uint32_t tQ = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + kColDQ;
    const int r_lo = quarter * 32 + (lane >> 2);  // row within the tile (+16 slab, +8 high half)
    const int c_lo = 2 * (lane & 3);              // column within an 8-column group
    for (int it = 0; it < n_it; ++it) {
      const int hq = hkv * group + it / n_i;
      const int i = i0 + it % n_i;
      const size_t head_base = static_cast<size_t>(b * Hq + hq) * N;
      if (!__all_sync(0xffffffffu, mbar_wait(&bar[KB_DQFULL], it & 1, abort_flag, err))) break;
      tc_fence_after();
      uint32_t v[2][D / 8][4];  // [slab][8-column group][element]
#pragma unroll
      for (int sl = 0; sl < 2; ++sl)
#pragma unroll
        for (int c = 0; c < D; c += 32)
          tmem_ld16x256_x4(tQ + (static_cast<uint32_t>(sl * 16) << 16) + c, &v[sl][c / 8][0]);
      tmem_ld_wait();
      reg_fence<D>(&v[0][0][0]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[KB_DQFREE]);
#pragma unroll
      for (int sl = 0; sl < 2; ++sl) {
#pragma unroll
        for (int hi = 0; hi < 2; ++hi) {
          const int qrow = i * kBlk + r_lo + 16 * sl + 8 * hi;
          if (qrow < N) {
            float* dst = dq_acc + (head_base + qrow) * D + c_lo;
#pragma unroll
            for (int g = 0; g < D / 8; ++g)
              red_add_f32x2(dst + 8 * g, __uint_as_float(v[sl][g][2 * hi]),
                            __uint_as_float(v[sl][g][2 * hi + 1]));
          }
        }
      }
    }
  };

  if constexpr (ONEPASS) {
    // Register reallocation sits inside each warpgroup's branch, so no compute
    // code is reachable under the control warpgroup's limit.
    if (warp >= 8) {
      setmaxnreg_dec<kOnePassRegsControl>();
      if (warp == kProducer)
        producer();
      else if (warp == kIssuer)
        issuer();
    } else if (warp < 4) {
      setmaxnreg_inc<kOnePassRegsCompute>();
      compute();
    } else {
      setmaxnreg_inc<kOnePassRegsDrain>();
      drain();
    }
  } else {
    if (warp == kProducer)
      producer();
    else if (warp == kIssuer)
      issuer();
    else
      compute();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kIssuer) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace bwd
}  // namespace fa
