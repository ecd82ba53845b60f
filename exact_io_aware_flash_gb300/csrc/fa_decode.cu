// Split-KV forward for decoding (Flash-Decoding): few query rows, a long key
// sequence.
//
// "Flash Attention" (aiwiki.ai), section "Flash-Decoding": when the query is
// short, batch and heads do not expose enough parallel work, so the key/value
// sequence is split into chunks, each chunk's attention is computed with its
// own log-sum-exp, and a small reduction combines the chunks.
//
// Layout trick for grouped-query attention: q is [B, Hq, Nq, d] =
// [B*Hkv, g*Nq, d] with g = Hq/Hkv, so the query rows of all g heads that share
// a KV head are one contiguous block of Mq = g*Nq rows.  One CTA takes 128 of
// those rows against one chunk of key tiles, so each K/V tile is read from
// HBM once per KV head rather than once per query head.
//
// Kernels:
//   fa_decode_kernel   per (128-row block of a KV head's stacked query rows,
//                      KV head, split): S = Q K^T and O += P V on tcgen05 over
//                      the split's key tiles with online softmax; writes the
//                      normalised partial O (fp32) and its LSE, or, with one
//                      split, the final O and LSE.
//   fa_decode_merge    O = sum_s e^{LSE_s} O_s / sum_s e^{LSE_s},
//                      LSE = ln sum_s e^{LSE_s}.
//
// Warps: 0-3 softmax (thread t <-> row t, TMEM lane t), 4 TMA producer, 5 MMA
// issuer and TMEM allocator.  TMEM: S0 [0,128), S1 [128,256), O [256,256+d);
// P(j) overwrites the first half of S(j & 1).  S(j+1) is issued before PV(j),
// so the tensor core computes the next scores while this tile's softmax runs.
#include "fa_internal.h"
#include "ptx.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace fa {
namespace {

constexpr int kBlk = 128;
constexpr int kAtomBytes = 16384;
constexpr int kThreads = 192;
constexpr int kStages = 3;

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

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > 200000000ull) break;
  }
}

template <int D>
struct DecSmem {
  static constexpr int kTile = kBlk * D * 2;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTile;
  static constexpr int kV = kK + kStages * kTile;
  static constexpr int kBar = kV + kStages * kTile;
  static constexpr int kBytes = kBar + 256;
  static constexpr int kAlloc = kBytes + 1024;
};

enum DecBars {
  DB_Q = 0,
  DB_KFULL = 1,   // +stage
  DB_KEMPTY = 4,  // +stage
  DB_VFULL = 7,   // +stage
  DB_VEMPTY = 10, // +stage
  DB_SFULL = 13,  // +S buffer
  DB_PFULL = 15,  // P(j) in TMEM (4 softmax warps)
  DB_ODONE = 16,  // PV(j) done
  DB_FINAL = 17,
  DB_N = 18
};

template <int D, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    fa_decode_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, void* __restrict__ out,
                     float* __restrict__ lse_out, float* __restrict__ o_part,
                     float* __restrict__ lse_part, int kv_heads, int Mq, int Nk, int chunk_tiles,
                     int splits, float scale_log2, int* err) {
  using L = DecSmem<D>;
  constexpr int kAtoms = D / 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + DB_N);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int QT = (Mq + kBlk - 1) / kBlk;
  const int qt = blockIdx.x % QT;
  const int bkv = (blockIdx.x / QT) % kv_heads;
  const int split = blockIdx.x / (QT * kv_heads);
  const int KT = (Nk + kBlk - 1) / kBlk;
  const int j0 = split * chunk_tiles;
  const int j1 = (j0 + chunk_tiles < KT) ? j0 + chunk_tiles : KT;
  const int n = j1 - j0;  // >= 1 by construction of chunk_tiles

  if (threadIdx.x == 0) {
    for (int i = 0; i < DB_N; ++i) {
      uint32_t cnt = 1;
      if (i == DB_PFULL) cnt = 4;
      mbar_init(&bar[i], cnt);
    }
    *abort_flag = (*reinterpret_cast<volatile int*>(err) != kDevErrNone) ? 1 : 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool run = (*abort_flag == 0);
  constexpr uint32_t kColO = 256;

  if (run && warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      const uint64_t pol_stream = l2_policy_evict_first();
      mbar_expect_tx(&bar[DB_Q], L::kTile);
      for (int a = 0; a < kAtoms; ++a)
        tma_load_3d(smem + L::kQ + a * kAtomBytes, &tm_q, &bar[DB_Q], a * 64, qt * kBlk, bkv,
                    pol_stream);
      int issued = 0;
      for (int jj = 0; jj < n; ++jj) {
        const int st = jj % kStages;
        const uint32_t ph = (jj / kStages) & 1;
        const int kr = (j0 + jj) * kBlk;
        if (!mbar_wait(&bar[DB_KEMPTY + st], ph ^ 1, abort_flag, err)) break;
        mbar_expect_tx(&bar[DB_KFULL + st], L::kTile);
        for (int a = 0; a < kAtoms; ++a)
          tma_load_3d(smem + L::kK + st * L::kTile + a * kAtomBytes, &tm_k, &bar[DB_KFULL + st],
                      a * 64, kr, bkv, pol_stream);
        if (!mbar_wait(&bar[DB_VEMPTY + st], ph ^ 1, abort_flag, err)) {
          issued = 2 * jj + 1;
          break;
        }
        mbar_expect_tx(&bar[DB_VFULL + st], L::kTile);
        for (int a = 0; a < kAtoms; ++a)
          tma_load_3d(smem + L::kV + st * L::kTile + a * kAtomBytes, &tm_v, &bar[DB_VFULL + st],
                      a * 64, kr, bkv, pol_stream);
        issued = 2 * jj + 2;
      }
      if (*abort_flag) {
        drain_wait(&bar[DB_Q], 0);
        for (int x = (issued > 2 * kStages ? issued - 2 * kStages : 0); x < issued; ++x) {
          const int jj = x >> 1;
          drain_wait(&bar[((x & 1) ? DB_VFULL : DB_KFULL) + jj % kStages], (jj / kStages) & 1);
        }
      }
    }
  } else if (run && warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_f16(kBlk, kBlk, BF16, false, false);
      constexpr uint32_t kIdO = idesc_f16(kBlk, D, BF16, false, true);
      const uint32_t sq = smem_u32(smem + L::kQ);
      const uint32_t sk = smem_u32(smem + L::kK);
      const uint32_t sv = smem_u32(smem + L::kV);
      auto issue_s = [&](int jj) {
        const int st = jj % kStages;
        const uint32_t ka = sk + st * L::kTile;
        const uint32_t dt = tmem + (jj & 1) * 128;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks >> 2) * kAtomBytes + (ks & 3) * 32;
          mma_ss(dt, sdesc_sw128(sq + off, 16, 1024), sdesc_sw128(ka + off, 16, 1024), kIdS, ks > 0);
        }
        mma_commit(&bar[DB_SFULL + (jj & 1)]);
        mma_commit(&bar[DB_KEMPTY + st]);
      };
      bool ok = mbar_wait(&bar[DB_Q], 0, abort_flag, err) &&
                mbar_wait(&bar[DB_KFULL], 0, abort_flag, err);
      if (ok) {
        tc_fence_after();
        issue_s(0);
      }
      for (int jj = 0; ok && jj < n; ++jj) {
        if (jj + 1 < n) {
          // S(j+1) goes to buffer (j+1) & 1, whose P(j-1) PV(j-1) reads.
          if (!(ok = mbar_wait(&bar[DB_KFULL + (jj + 1) % kStages], ((jj + 1) / kStages) & 1,
                               abort_flag, err)))
            break;
          if (jj >= 1 && !(ok = mbar_wait(&bar[DB_ODONE], (jj - 1) & 1, abort_flag, err))) break;
          tc_fence_after();
          issue_s(jj + 1);
        }
        const int st = jj % kStages;
        if (!(ok = mbar_wait(&bar[DB_VFULL + st], (jj / kStages) & 1, abort_flag, err))) break;
        if (!(ok = mbar_wait(&bar[DB_PFULL], jj & 1, abort_flag, err))) break;
        tc_fence_after();
        const uint32_t va = sv + st * L::kTile;
        const uint32_t pt = tmem + (jj & 1) * 128;
#pragma unroll
        for (int ks = 0; ks < kBlk / 16; ++ks)
          mma_ts(tmem + kColO, pt + ks * 8, sdesc_sw128(va + ks * 2048, kAtomBytes, 1024), kIdO,
                 (jj > 0 || ks > 0) ? 1u : 0u);
        mma_commit(&bar[DB_ODONE]);
        mma_commit(&bar[DB_VEMPTY + st]);
      }
      mma_commit(&bar[DB_FINAL]);
      drain_wait(&bar[DB_FINAL], 0);
    }
  } else if (run && warp < 4) {
    // ------------------------------------------------------------ softmax + epilogue
    const int r = threadIdx.x;
    const int row = qt * kBlk + r;  // stacked query row of this KV head
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tO = tmem + lane_off + kColO;
    const bool pos_scale = scale_log2 > 0.f;
    const float sfac = pos_scale ? scale_log2 : 1.0f;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int jj = 0; jj < n; ++jj) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bar[DB_SFULL + (jj & 1)], (jj >> 1) & 1, abort_flag, err));
      if (!ok) break;
      tc_fence_after();
      const uint32_t tS = tmem + lane_off + (jj & 1) * 128;
      uint32_t x[kBlk];
#pragma unroll
      for (int c = 0; c < kBlk; c += 32) tmem_ld32(tS + c, x + c);
      tmem_ld_wait();
      reg_fence<kBlk>(x);
      if (!pos_scale) {
#pragma unroll
        for (int c = 0; c < kBlk; ++c) x[c] = __float_as_uint(__uint_as_float(x[c]) * scale_log2);
      }
      const int kbase = (j0 + jj) * kBlk;
      if (kbase + kBlk > Nk) {
        const int lim = Nk - kbase;
#pragma unroll
        for (int c = 0; c < kBlk; ++c)
          if (c >= lim) x[c] = __float_as_uint(-INFINITY);
      }
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
          fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7])) * sfac;
      // Conditional rescale, as in the forward kernel (threshold 8 in the exp2 domain).
      float alpha = 1.0f;
      bool rescale = false;
      if (jj == 0) {
        m_run = mx;
      } else {
        const bool need = mx > m_run + 8.0f;
        rescale = __any_sync(0xffffffffu, need);
        if (need) {
          alpha = ex2_approx(m_run - mx);
          m_run = mx;
        }
      }
      const uint64_t sfac2 = f2_pack(sfac, sfac);
      const uint64_t negm2 = f2_pack(-m_run, -m_run);
      uint64_t rs2[2] = {0ull, 0ull};
#pragma unroll
      for (int c = 0; c < kBlk; c += 32) {
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
          pk[e] = pack2<BF16>(p0, p1);
        }
        tmem_st16(tS + c / 2, pk);
      }
      float r0, r1, r2, r3;
      f2_unpack(rs2[0], r0, r1);
      f2_unpack(rs2[1], r2, r3);
      l_run = l_run * alpha + ((r0 + r1) + (r2 + r3));
      // PV(j-1) must be complete before O is touched (and every phase of the
      // barrier is waited in order, so the parity wait is unambiguous).
      if (jj >= 1) {
        ok = __all_sync(0xffffffffu, mbar_wait(&bar[DB_ODONE], (jj - 1) & 1, abort_flag, err));
        if (!ok) break;
        tc_fence_after();
      }
      if (rescale) {
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
      if (lane == 0) mbar_arrive(&bar[DB_PFULL]);
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bar[DB_ODONE], (n - 1) & 1, abort_flag, err));
    if (ok) {
      tc_fence_after();
      const float inv_l = 1.0f / l_run;
      const bool valid = row < Mq;
      const size_t grow = static_cast<size_t>(bkv) * Mq + row;  // row of [B*Hq*Nq]
      const float lse_row = (m_run + log2f(l_run)) * 0.69314718055994530942f;
      if (splits == 1) {
        uint16_t* orow = reinterpret_cast<uint16_t*>(out) + grow * D;
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          uint32_t o[32];
          tmem_ld32(tO + c, o);
          tmem_ld_wait();
          reg_fence<32>(o);
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack2<BF16>(__uint_as_float(o[2 * e]) * inv_l, __uint_as_float(o[2 * e + 1]) * inv_l);
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4)
              dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
          }
        }
        if (valid) lse_out[grow] = lse_row;
      } else {
        const size_t rows = static_cast<size_t>(kv_heads) * Mq;
        float* prow = o_part + (static_cast<size_t>(split) * rows + grow) * D;
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          uint32_t o[32];
          tmem_ld32(tO + c, o);
          tmem_ld_wait();
          reg_fence<32>(o);
          if (valid) {
            float4* dst = reinterpret_cast<float4*>(prow + c);
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4)
              dst[v4] = make_float4(__uint_as_float(o[4 * v4]) * inv_l, __uint_as_float(o[4 * v4 + 1]) * inv_l,
                                    __uint_as_float(o[4 * v4 + 2]) * inv_l,
                                    __uint_as_float(o[4 * v4 + 3]) * inv_l);
          }
        }
        if (valid) lse_part[static_cast<size_t>(split) * rows + grow] = lse_row;
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

// One warp per row: combine the splits' normalised partials by their LSEs.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) fa_decode_merge(const float* __restrict__ o_part,
                                                       const float* __restrict__ lse_part,
                                                       void* __restrict__ out,
                                                       float* __restrict__ lse_out, long rows,
                                                       int splits) {
  const int lane = threadIdx.x & 31;
  const long warps = static_cast<long>(gridDim.x) * (blockDim.x >> 5);
  for (long row = static_cast<long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); row < rows;
       row += warps) {
    float m = -INFINITY;
    for (int s = 0; s < splits; ++s) m = fmaxf(m, lse_part[s * rows + row]);
    float den = 0.f;
    float acc[D / 32];
#pragma unroll
    for (int e = 0; e < D / 32; ++e) acc[e] = 0.f;
    for (int s = 0; s < splits; ++s) {
      const float w = exp2f((lse_part[s * rows + row] - m) * 1.4426950408889634f);
      den += w;
      const float* p = o_part + (s * rows + row) * D;
#pragma unroll
      for (int e = 0; e < D / 32; ++e) acc[e] = fmaf(w, p[lane + 32 * e], acc[e]);
    }
    const float inv = 1.0f / den;
    uint16_t* orow = reinterpret_cast<uint16_t*>(out) + row * D;
#pragma unroll
    for (int e = 0; e < D / 32; ++e) {
      const float val = acc[e] * inv;
      uint16_t h;
      if constexpr (BF16) {
        __nv_bfloat16 b = __float2bfloat16_rn(val);
        h = *reinterpret_cast<uint16_t*>(&b);
      } else {
        __half b = __float2half_rn(val);
        h = *reinterpret_cast<uint16_t*>(&b);
      }
      orow[lane + 32 * e] = h;
    }
    if (lane == 0) lse_out[row] = m + logf(den);
  }
}

template <int D, bool BF16>
cudaError_t launch_decode_t(const AttnShape& s, const DecodeArgs& a, cudaStream_t stream) {
  auto kern = fa_decode_kernel<D, BF16>;
  constexpr int smem = DecSmem<D>::kAlloc;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), smem,
                                24 + (D == 64 ? 0 : 2) + (BF16 ? 1 : 0));
  if (e != cudaSuccess) return e;
  const int g = s.Hq / s.Hkv;
  const int Mq = g * a.Nq;
  const int QT = (Mq + kBlk - 1) / kBlk;
  const int kv_heads = s.B * s.Hkv;
  const float scale_log2 = s.scale * 1.4426950408889634f;
  dim3 grid(static_cast<unsigned>(QT * kv_heads * a.splits));
  kern<<<grid, kThreads, smem, stream>>>(a.tm_q, a.tm_k, a.tm_v, a.o, a.lse, a.o_part, a.lse_part,
                                         kv_heads, Mq, a.Nk, a.chunk_tiles, a.splits, scale_log2,
                                         a.err);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (a.splits > 1) {
    const long rows = static_cast<long>(kv_heads) * Mq;
    long blocks = (rows + 7) / 8;
    if (blocks > 152L * 16) blocks = 152L * 16;
    fa_decode_merge<D, BF16><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        a.o_part, a.lse_part, a.o, a.lse, rows, a.splits);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace

size_t decode_smem_bytes(int d) { return d == 64 ? DecSmem<64>::kAlloc : DecSmem<128>::kAlloc; }

cudaError_t launch_decode(const AttnShape& s, const DecodeArgs& a, cudaStream_t stream) {
  if (s.d == 64) return s.bf16 ? launch_decode_t<64, true>(s, a, stream) : launch_decode_t<64, false>(s, a, stream);
  return s.bf16 ? launch_decode_t<128, true>(s, a, stream) : launch_decode_t<128, false>(s, a, stream);
}

}  // namespace fa
