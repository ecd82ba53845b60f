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
//     D_i  = sum_c dO_ic O_ic                    (preprocessing kernel)
//     dS   = P o (dP - D)
//     dQ   = scale * dS K,   dK = scale * dS^T Q
//
// Kernels, all on the caller's stream:
//   fa_bwd_pre_kernel   D = rowsum(dO o O) and zero the fp32 dQ accumulator.
//   fa_bwd_kernel       one CTA per (KV head, 128-key tile j); loops over the
//                       KV head's query heads and query tiles i (causal: i >= j).
//                       Transposed formulation, so that the key tile owns the
//                       TMEM lanes and dK, dV accumulate in Tensor Memory over
//                       the whole loop (no atomics for dK / dV, and GQA groups
//                       are summed in-kernel):
//                         S^T  = K_j Q_i^T          tcgen05, SMEM x SMEM
//                         dP^T = V_j dO_i^T         tcgen05, SMEM x SMEM
//                         P^T, dS^T                 compute warps (exp2, fp32)
//                         dV  += P^T dO_i           tcgen05, P^T from TMEM
//                         dK  += dS^T Q_i           tcgen05, dS^T from SMEM
//                         dQ_i = dS K_j             tcgen05, dS^T read MN-major
//                         dQacc_i += dQ_i           fp32 vector atomics
//                       The primer notes that the default backward accumulates
//                       dQ across thread blocks with atomic adds (section
//                       "Backward pass: recomputation instead of storage"); so
//                       does this one.
//   fa_bwd_dq_kernel    dq = scale * dQacc, converted to the 16-bit type.
//
// Warp roles of fa_bwd_kernel (10 warps):
//   warps 0-3  compute: thread t owns key row t of the tile (TMEM lane t).
//   warps 4-7  dQ readout + dK epilogue.
//   warp 8     producer: K_j, V_j once; Q_i, dO_i through a 2-stage ring (TMA);
//              LSE_i and D_i for the tile into shared memory (plain loads).
//   warp 9     MMA issuer (one thread) and TMEM allocator.
// TMEM columns: dV [0,128), dK [128,256), S^T / P^T [256,384), dP^T / dQ [384,512).
#include "fa_internal.h"
#include "ptx.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace fa {
namespace {

constexpr int kBlk = 128;          // rows per tile (keys and queries)
constexpr int kAtomBytes = 16384;  // 128 rows x 128 bytes
constexpr int kThreads = 320;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BwdSmem {
  static constexpr int kTile = kBlk * D * 2;
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTile;
  static constexpr int kQ = kV + kTile;        // 2 stages
  static constexpr int kdO = kQ + 2 * kTile;   // 2 stages
  static constexpr int kdS = kdO + 2 * kTile;  // dS^T, 128 x 128 16-bit = 32 KB
  static constexpr int kLse = kdS + 32768;     // 128 floats: LSE * log2(e)
  static constexpr int kDrow = kLse + 512;     // 128 floats: D
  static constexpr int kBar = kDrow + 512;
  static constexpr int kBytes = kBar + 256;
  static constexpr int kAlloc = kBytes + 1024;
};

enum BwdBars {
  BKV = 0,
  BQFULL = 1,   // +stage
  BQEMPTY = 3,  // +stage
  BLDFULL = 5,
  BLDEMPTY = 6,
  BSDP = 7,     // S^T and dP^T in TMEM
  BPDS = 8,     // P^T in TMEM and dS^T in SMEM
  BDVDONE = 9,  // dV MMA of this iteration done (S/P columns free)
  BDQ = 10,     // dQ tile in TMEM
  BDQFREE = 11, // dQ tile read out (dP/dQ columns free)
  BFINAL = 12,
  NBWDBARS = 13
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

template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
  if constexpr (BF16) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&w);
    return __bfloat1622float2(v);
  } else {
    __half2 v = *reinterpret_cast<__half2*>(&w);
    return __half22float2(v);
  }
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > 200000000ull) break;
  }
}

// ------------------------------------------------------------------ preprocessing
// D_i = sum_c dO_ic O_ic (fp32) and dQacc = 0.  D/8 threads per row, 16 bytes each.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) fa_bwd_pre_kernel(const uint4* __restrict__ O,
                                                         const uint4* __restrict__ dO,
                                                         float* __restrict__ Drow,
                                                         float4* __restrict__ dq_acc, long rows) {
  constexpr int kTpr = D / 8;  // threads per row
  const long total = rows * kTpr;
  const long stride = static_cast<long>(gridDim.x) * blockDim.x;
  const int lane = threadIdx.x & 31;
  const int sub = threadIdx.x % kTpr;
  // Whole warps iterate together so the row reduction's shuffles see all lanes.
  for (long w0 = static_cast<long>(blockIdx.x) * blockDim.x + (threadIdx.x & ~31); w0 < total;
       w0 += stride) {
    const long t = w0 + lane;
    const bool in = t < total;
    const long row = t / kTpr;
    float acc = 0.f;
    if (in) {
      const uint4 a = O[t];
      const uint4 b = dO[t];
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
      const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 x = unpack2<BF16>(aw[e]);
        const float2 y = unpack2<BF16>(bw[e]);
        acc = fmaf(x.x, y.x, acc);
        acc = fmaf(x.y, y.y, acc);
      }
    }
#pragma unroll
    for (int off = kTpr / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (in) {
      if (sub == 0) Drow[row] = acc;
      const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
      dq_acc[row * (D / 4) + 2 * sub] = z;
      dq_acc[row * (D / 4) + 2 * sub + 1] = z;
    }
  }
}

// dq = scale * dQacc in the 16-bit type; 8 elements per thread.
template <bool BF16>
__global__ void __launch_bounds__(256) fa_bwd_dq_kernel(const float4* __restrict__ acc,
                                                        uint4* __restrict__ dq, long n8,
                                                        float scale) {
  const long stride = static_cast<long>(gridDim.x) * blockDim.x;
  for (long t = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; t < n8; t += stride) {
    const float4 a = acc[2 * t];
    const float4 b = acc[2 * t + 1];
    dq[t] = make_uint4(pack2<BF16>(a.x * scale, a.y * scale), pack2<BF16>(a.z * scale, a.w * scale),
                       pack2<BF16>(b.x * scale, b.y * scale), pack2<BF16>(b.z * scale, b.w * scale));
  }
}

// ------------------------------------------------------------------ main kernel
template <int D, bool BF16>
__device__ __forceinline__ void store_rows_from_tmem(uint32_t taddr, uint16_t* row, float mul,
                                                     bool valid) {
#pragma unroll
  for (int c = 0; c < D; c += 32) {
    uint32_t v[32];
    tmem_ld32(taddr + c, v);
    tmem_ld_wait();
    reg_fence<32>(v);
    uint32_t pk[16];
#pragma unroll
    for (int e = 0; e < 16; ++e)
      pk[e] = pack2<BF16>(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
    if (valid) {
      uint4* dst = reinterpret_cast<uint4*>(row + c);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4)
        dst[q4] = make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
    }
  }
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const float* __restrict__ lse, const float* __restrict__ Drow,
                  float* __restrict__ dq_acc, void* __restrict__ dk_out, void* __restrict__ dv_out,
                  int Hq, int Hkv, int N, int causal, float scale, int* err) {
  using L = BwdSmem<D>;
  constexpr int kAtoms = D / 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + NBWDBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* s_lse = reinterpret_cast<float*>(smem + L::kLse);
  float* s_d = reinterpret_cast<float*>(smem + L::kDrow);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bkv = blockIdx.x;  // b * Hkv + hkv
  const int j = blockIdx.y;    // key tile; small j has the most work under causal
  const int b = bkv / Hkv;
  const int hkv = bkv % Hkv;
  const int group = Hq / Hkv;
  const int T = (N + kBlk - 1) / kBlk;
  const int i0 = causal ? j : 0;
  const int n_i = T - i0;
  const int n_it = group * n_i;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NBWDBARS; ++i) {
      uint32_t cnt = 1;
      if (i == BLDFULL) cnt = 32;
      if (i == BLDEMPTY || i == BPDS || i == BDQFREE) cnt = 4;
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
  constexpr uint32_t kColDV = 0, kColDK = 128, kColS = 256, kColDP = 384;

  if (run && warp == 8) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_kv = l2_policy_evict_first();
    const uint64_t pol_q = l2_policy_evict_last();
    int issued = 0;
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      mbar_expect_tx(&bar[BKV], 2 * L::kTile);
      for (int a = 0; a < kAtoms; ++a) {
        tma_load_3d(smem + L::kK + a * kAtomBytes, &tm_k, &bar[BKV], a * 64, j * kBlk, bkv, pol_kv);
        tma_load_3d(smem + L::kV + a * kAtomBytes, &tm_v, &bar[BKV], a * 64, j * kBlk, bkv, pol_kv);
      }
    }
    for (int it = 0; it < n_it; ++it) {
      const int hq = hkv * group + it / n_i;
      const int i = i0 + it % n_i;
      const int bhq = b * Hq + hq;
      const int st = it & 1;
      bool ok = true;
      if (lane == 0) {
        ok = mbar_wait(&bar[BQEMPTY + st], ((it >> 1) & 1) ^ 1, abort_flag, err);
        if (ok) {
          mbar_expect_tx(&bar[BQFULL + st], 2 * L::kTile);
          for (int a = 0; a < kAtoms; ++a) {
            tma_load_3d(smem + L::kQ + st * L::kTile + a * kAtomBytes, &tm_q, &bar[BQFULL + st],
                        a * 64, i * kBlk, bhq, pol_q);
            tma_load_3d(smem + L::kdO + st * L::kTile + a * kAtomBytes, &tm_do, &bar[BQFULL + st],
                        a * 64, i * kBlk, bhq, pol_q);
          }
          issued = it + 1;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (ok && it > 0) ok = __all_sync(0xffffffffu, mbar_wait(&bar[BLDEMPTY], (it - 1) & 1, abort_flag, err));
      if (!ok) break;
      // LSE (as log2) and D of the 128 query rows of this tile; padding rows get
      // LSE = +inf so that their recomputed probabilities are exactly 0.
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = lane * 4 + e;
        const int qrow = i * kBlk + r;
        const size_t g = static_cast<size_t>(bhq) * N + qrow;
        const bool in = qrow < N;
        s_lse[r] = in ? lse[g] * kLog2e : INFINITY;
        s_d[r] = in ? Drow[g] : 0.f;
      }
      mbar_arrive(&bar[BLDFULL]);
    }
    if (lane == 0 && *abort_flag) {
      drain_wait(&bar[BKV], 0);
      for (int it = (issued > 2 ? issued - 2 : 0); it < issued; ++it)
        drain_wait(&bar[BQFULL + (it & 1)], (it >> 1) & 1);
    }
  } else if (run && warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_f16(kBlk, kBlk, BF16, false, false);  // S^T, dP^T
      constexpr uint32_t kIdKV = idesc_f16(kBlk, D, BF16, false, true);     // dV, dK
      constexpr uint32_t kIdQ = idesc_f16(kBlk, D, BF16, true, true);       // dQ
      const uint32_t sk = smem_u32(smem + L::kK);
      const uint32_t sv = smem_u32(smem + L::kV);
      const uint32_t sq = smem_u32(smem + L::kQ);
      const uint32_t sdo = smem_u32(smem + L::kdO);
      const uint32_t sds = smem_u32(smem + L::kdS);
      bool ok = mbar_wait(&bar[BKV], 0, abort_flag, err);
      for (int it = 0; ok && it < n_it; ++it) {
        const int st = it & 1;
        if (!(ok = mbar_wait(&bar[BQFULL + st], (it >> 1) & 1, abort_flag, err))) break;
        if (it > 0 && !(ok = mbar_wait(&bar[BDVDONE], (it - 1) & 1, abort_flag, err))) break;
        tc_fence_after();
        const uint32_t qa = sq + st * L::kTile;
        const uint32_t doa = sdo + st * L::kTile;
        // S^T = K_j Q_i^T
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks >> 2) * kAtomBytes + (ks & 3) * 32;
          mma_ss(tmem + kColS, sdesc_sw128(sk + off, 16, 1024), sdesc_sw128(qa + off, 16, 1024),
                 kIdS, ks > 0);
        }
        if (it > 0 && !(ok = mbar_wait(&bar[BDQFREE], (it - 1) & 1, abort_flag, err))) break;
        tc_fence_after();
        // dP^T = V_j dO_i^T
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks >> 2) * kAtomBytes + (ks & 3) * 32;
          mma_ss(tmem + kColDP, sdesc_sw128(sv + off, 16, 1024), sdesc_sw128(doa + off, 16, 1024),
                 kIdS, ks > 0);
        }
        mma_commit(&bar[BSDP]);
        if (!(ok = mbar_wait(&bar[BPDS], it & 1, abort_flag, err))) break;
        tc_fence_after();
        // dV += P^T dO_i   (P^T: 16-bit pairs in TMEM over the first half of S^T)
#pragma unroll
        for (int ks = 0; ks < kBlk / 16; ++ks)
          mma_ts(tmem + kColDV, tmem + kColS + ks * 8, sdesc_sw128(doa + ks * 2048, kAtomBytes, 1024),
                 kIdKV, (it > 0 || ks > 0) ? 1u : 0u);
        mma_commit(&bar[BDVDONE]);
        // dK += dS^T Q_i   (dS^T in SMEM, K-major over the query index)
#pragma unroll
        for (int ks = 0; ks < kBlk / 16; ++ks) {
          const uint32_t off = (ks >> 2) * kAtomBytes + (ks & 3) * 32;
          mma_ss(tmem + kColDK, sdesc_sw128(sds + off, 16, 1024),
                 sdesc_sw128(qa + ks * 2048, kAtomBytes, 1024), kIdKV, (it > 0 || ks > 0) ? 1u : 0u);
        }
        // dQ_i = dS K_j   (the same dS^T buffer read MN-major; K_j as an MN-major B)
#pragma unroll
        for (int ks = 0; ks < kBlk / 16; ++ks)
          mma_ss(tmem + kColDP, sdesc_sw128(sds + ks * 2048, kAtomBytes, 1024),
                 sdesc_sw128(sk + ks * 2048, kAtomBytes, 1024), kIdQ, ks > 0);
        mma_commit(&bar[BDQ]);
        mma_commit(&bar[BQEMPTY + st]);
      }
      mma_commit(&bar[BFINAL]);
      drain_wait(&bar[BFINAL], 0);
    }
  } else if (run && warp < 4) {
    // ------------------------------------------------------------ compute: P^T, dS^T
    const int t = threadIdx.x;  // key row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tS = tmem + lane_off + kColS;
    const uint32_t tP = tmem + lane_off + kColDP;
    const float sl2 = scale * kLog2e;
    uint8_t* sds = smem + L::kdS;
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int i = i0 + it % n_i;
      ok = __all_sync(0xffffffffu, mbar_wait(&bar[BSDP], it & 1, abort_flag, err) &&
                                       mbar_wait(&bar[BLDFULL], it & 1, abort_flag, err));
      if (!ok) break;
      tc_fence_after();
      const bool diag = causal && (i == j);
#pragma unroll
      for (int c = 0; c < kBlk; c += 32) {
        uint32_t sv[32], dpv[32];
        tmem_ld32(tS + c, sv);
        tmem_ld32(tP + c, dpv);
        tmem_ld_wait();
        reg_fence<32>(sv);
        reg_fence<32>(dpv);
        uint32_t pk[16], dk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 l4 = *reinterpret_cast<const float4*>(s_lse + c + e);
          const float4 d4 = *reinterpret_cast<const float4*>(s_d + c + e);
          const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
          const float dv4[4] = {d4.x, d4.y, d4.z, d4.w};
          float p[4], ds[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            float pv = ex2_approx(fmaf(__uint_as_float(sv[e + u]), sl2, -lv[u]));
            if (diag && (c + e + u) < t) pv = 0.f;  // query i*128+c+e+u before key j*128+t
            p[u] = pv;
            ds[u] = pv * (__uint_as_float(dpv[e + u]) - dv4[u]);
          }
          pk[e / 2] = pack2<BF16>(p[0], p[1]);
          pk[e / 2 + 1] = pack2<BF16>(p[2], p[3]);
          dk[e / 2] = pack2<BF16>(ds[0], ds[1]);
          dk[e / 2 + 1] = pack2<BF16>(ds[2], ds[3]);
        }
        // P^T chunk over S^T columns already read (chunk c/32 -> columns c/2 .. c/2+15)
        tmem_st16(tS + c / 2, pk);
        // dS^T row t, query columns c..c+31: 64 bytes = four 16-byte chunks
        const int atom = c >> 6;
        const int ch0 = (c & 63) >> 3;
#pragma unroll
        for (int u = 0; u < 4; ++u)
          *reinterpret_cast<uint4*>(sds + atom * kAtomBytes + sw128_offset(t, ch0 + u)) =
              make_uint4(dk[4 * u], dk[4 * u + 1], dk[4 * u + 2], dk[4 * u + 3]);
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bar[BLDEMPTY]);
        mbar_arrive(&bar[BPDS]);
      }
    }
    // dV epilogue
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bar[BFINAL], 0, abort_flag, err));
    if (ok) {
      tc_fence_after();
      const int kv = j * kBlk + t;
      uint16_t* row = reinterpret_cast<uint16_t*>(dv_out) + (static_cast<size_t>(bkv) * N + kv) * D;
      store_rows_from_tmem<D, BF16>(tmem + lane_off + kColDV, row, 1.0f, kv < N);
    }
  } else if (run && warp < 8) {
    // ------------------------------------------------------------ dQ readout, dK epilogue
    const int t = threadIdx.x - 128;  // query row within the tile (TMEM lane)
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tQ = tmem + lane_off + kColDP;
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int hq = hkv * group + it / n_i;
      const int i = i0 + it % n_i;
      ok = __all_sync(0xffffffffu, mbar_wait(&bar[BDQ], it & 1, abort_flag, err));
      if (!ok) break;
      tc_fence_after();
      const int qrow = i * kBlk + t;
      float4* dst = reinterpret_cast<float4*>(
          dq_acc + (static_cast<size_t>(b * Hq + hq) * N + qrow) * D);
#pragma unroll
      for (int c = 0; c < D; c += 32) {
        uint32_t v[32];
        tmem_ld32(tQ + c, v);
        tmem_ld_wait();
        reg_fence<32>(v);
        if (qrow < N) {
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4)
            atomicAdd(dst + c / 4 + q4,
                      make_float4(__uint_as_float(v[4 * q4]), __uint_as_float(v[4 * q4 + 1]),
                                  __uint_as_float(v[4 * q4 + 2]), __uint_as_float(v[4 * q4 + 3])));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[BDQFREE]);
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bar[BFINAL], 0, abort_flag, err));
    if (ok) {
      tc_fence_after();
      const int kv = j * kBlk + t;
      uint16_t* row = reinterpret_cast<uint16_t*>(dk_out) + (static_cast<size_t>(bkv) * N + kv) * D;
      store_rows_from_tmem<D, BF16>(tmem + lane_off + kColDK, row, scale, kv < N);
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

int grid_for(long work_items, int per_block) {
  long blocks = (work_items + per_block - 1) / per_block;
  const long cap = 152L * 16;  // 16 resident 256-thread blocks per SM
  if (blocks > cap) blocks = cap;
  return static_cast<int>(blocks < 1 ? 1 : blocks);
}

template <int D, bool BF16>
cudaError_t launch_bwd_t(const AttnShape& s, const BwdArgs& a, cudaStream_t stream) {
  const long rows = static_cast<long>(s.B) * s.Hq * s.N;
  fa_bwd_pre_kernel<D, BF16><<<grid_for(rows * (D / 8), 256), 256, 0, stream>>>(
      static_cast<const uint4*>(a.o), static_cast<const uint4*>(a.dO), a.D,
      reinterpret_cast<float4*>(a.dq_acc), rows);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  auto kern = fa_bwd_kernel<D, BF16>;
  constexpr int smem = BwdSmem<D>::kAlloc;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int T = (s.N + kBlk - 1) / kBlk;
  dim3 grid(static_cast<unsigned>(s.B * s.Hkv), static_cast<unsigned>(T));
  if (a.ev_before_main && (e = cudaEventRecord(a.ev_before_main, stream)) != cudaSuccess) return e;
  kern<<<grid, kThreads, smem, stream>>>(a.tm_q, a.tm_k, a.tm_v, a.tm_do, a.lse, a.D, a.dq_acc,
                                         a.dk, a.dv, s.Hq, s.Hkv, s.N, s.causal, s.scale, a.err);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (a.ev_after_main && (e = cudaEventRecord(a.ev_after_main, stream)) != cudaSuccess) return e;

  const long n8 = rows * D / 8;
  fa_bwd_dq_kernel<BF16><<<grid_for(n8, 256), 256, 0, stream>>>(
      reinterpret_cast<const float4*>(a.dq_acc), static_cast<uint4*>(a.dq), n8, s.scale);
  return cudaGetLastError();
}

}  // namespace

size_t backward_smem_bytes(int d) {
  return d == 64 ? BwdSmem<64>::kAlloc : BwdSmem<128>::kAlloc;
}

cudaError_t launch_backward(const AttnShape& s, const BwdArgs& a, cudaStream_t stream) {
  if (s.d == 64) return s.bf16 ? launch_bwd_t<64, true>(s, a, stream) : launch_bwd_t<64, false>(s, a, stream);
  return s.bf16 ? launch_bwd_t<128, true>(s, a, stream) : launch_bwd_t<128, false>(s, a, stream);
}

}  // namespace fa
