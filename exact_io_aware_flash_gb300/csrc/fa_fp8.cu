// FP8 (e4m3) inputs for the low-precision forward: quantization kernels.
//
// "FlashAttention Primer", section "FlashAttention-3: Hopper asynchrony and FP8"
// (block quantization and an incoherent rotation before quantization) and "Flash
// Attention" (aiwiki.ai), section "FlashAttention-3" (the rotation is random signs
// followed by a Hadamard transform, applied to queries and keys alike, which keeps
// their dot products while spreading outlier channels over all channels).
//
//   Q, K: y = (x * s) H_d (Sylvester Hadamard, entries +-1, unnormalised), one scale
//         per 128-row block of a head: amax = max |y|, code = e4m3(y * (448 / amax)),
//         scale = amax * c with c = fl32(1 / (448 sqrt(d))) -- the 1/sqrt(d) makes the
//         dequantized rotation orthogonal -- or fl32(1/448) without rotation.
//   V:    no rotation, one scale per (head, channel) over all N rows (it factors out of
//         P V exactly); codes stored transposed, [d][Np] per head, so that V is a
//         K-major operand of the P V product.
// Every fp32 step that decides a code (sign flip, butterfly sums and differences in a
// fixed order, one division, one product, round-to-nearest-even conversion with
// saturation) is an exactly rounded IEEE operation, so the codes are a definite
// function of the inputs.
#include "fa_internal.h"
#include "ptx.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cmath>

namespace fa {
namespace {

template <bool BF16>
__device__ __forceinline__ float to_f32(uint16_t bits) {
  if constexpr (BF16) {
    return __bfloat162float(__ushort_as_bfloat16(bits));
  } else {
    return __half2float(__ushort_as_half(bits));
  }
}

__device__ __forceinline__ uint32_t e4m3(float x) {
  return static_cast<uint32_t>(__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3));
}

// Two codes, lo in the low byte (round to nearest even, saturated, like e4m3()).
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}

// Q and K, d = 128.  One CTA (8 warps) per (tensor, head, 128-row block).  A
// row belongs to 4 lanes, lane 4r + s holding channels 32s .. 32s + 31 of row r
// of its group of 8; warp w handles rows 16w .. 16w + 15 in two groups of 8.
// Butterfly stages 1 .. 16 run inside a lane, stages 32 and 64 across lanes.
constexpr int kQkThreads = 256;

template <bool BF16>
__global__ void __launch_bounds__(kQkThreads)
    fa_fp8_qk_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
                     const signed char* __restrict__ signs, uint8_t* __restrict__ q8,
                     uint8_t* __restrict__ k8, float* __restrict__ q_scale,
                     float* __restrict__ k_scale, int q_blocks, int N, int T, float cfac) {
  constexpr int D = 128;
  __shared__ float s_max[kQkThreads / 32];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int sub = lane & 3;   // channels 32*sub .. 32*sub + 31
  const int rsub = lane >> 2; // row within a group of 8
  const bool is_q = static_cast<int>(blockIdx.x) < q_blocks;
  const int blk = is_q ? blockIdx.x : blockIdx.x - q_blocks;  // head * T + block
  const int head = blk / T;
  const int t = blk % T;
  const uint16_t* src = (is_q ? q : k) + static_cast<size_t>(head) * N * D;
  uint8_t* dst = (is_q ? q8 : k8) + static_cast<size_t>(head) * N * D;
  // Both groups' loads are issued before any butterfly (the kernel is bound by
  // memory latency, not arithmetic).
  uint4 raw[2][4];
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    const int r = t * 128 + warp * 16 + g * 8 + rsub;
#pragma unroll
    for (int c = 0; c < 4; ++c)
      raw[g][c] = r < N ? *reinterpret_cast<const uint4*>(src + static_cast<size_t>(r) * D + 32 * sub + 8 * c)
                        : make_uint4(0u, 0u, 0u, 0u);
  }
  // A lane's 32 channels as 16 packed pairs (channels 2k, 2k+1).  The packed
  // fp32 operations round each half exactly as the scalar ones would, so the
  // codes are the same as a scalar butterfly's; the kernel is issue-bound and
  // the pairs halve most of its instructions.
  const uint64_t one2 = f2_pack(1.0f, 1.0f);
  const uint64_t neg1x2 = f2_pack(-1.0f, -1.0f);
  uint64_t sgn2[16];  // the random signs of this lane's channels, as packed +-1
  if (signs) {
#pragma unroll
    for (int k = 0; k < 16; ++k)
      sgn2[k] = f2_pack(signs[32 * sub + 2 * k] < 0 ? -1.0f : 1.0f, signs[32 * sub + 2 * k + 1] < 0 ? -1.0f : 1.0f);
  }
  uint64_t y[2][16];
  float amax = 0.f;
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    uint64_t* A = y[g];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t w[4] = {raw[g][c].x, raw[g][c].y, raw[g][c].z, raw[g][c].w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        A[4 * c + e] = f2_pack(to_f32<BF16>(static_cast<uint16_t>(w[e] & 0xFFFFu)),
                               to_f32<BF16>(static_cast<uint16_t>(w[e] >> 16)));
    }
    if (signs) {
#pragma unroll
      for (int k = 0; k < 16; ++k) A[k] = f2_mul(A[k], sgn2[k]);  // exact: x * (+-1)
      // Butterfly stage h pairs channel i (bit h clear) with i + h: (a + b, a - b).
      // h = 1 inside each pair:
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        float lo, hi;
        f2_unpack(A[k], lo, hi);
        A[k] = f2_pack(lo + hi, lo - hi);
      }
      // h = 2 .. 16: pair k with pair k + h/2; a - b as fma(b, -1, a), one rounding.
#pragma unroll
      for (int hp = 1; hp < 16; hp <<= 1) {
#pragma unroll
        for (int k = 0; k < 16; ++k)
          if ((k & hp) == 0) {
            const uint64_t lo = A[k], hi = A[k + hp];
            A[k] = f2_add(lo, hi);
            A[k + hp] = f2_fma(hi, neg1x2, lo);
          }
      }
      // h = 32, 64: channel 32s + e pairs with 32(s ^ m) + e, m = h / 32: the
      // lower lane keeps a + other, the upper one other - a, both as
      // fma(a, +-1, other).
#pragma unroll
      for (int m = 1; m < 4; m <<= 1) {
        const uint64_t sg = (sub & m) == 0 ? one2 : neg1x2;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          float lo, hi;
          f2_unpack(A[k], lo, hi);
          const uint64_t other = f2_pack(__shfl_xor_sync(0xffffffffu, lo, m), __shfl_xor_sync(0xffffffffu, hi, m));
          A[k] = f2_fma(A[k], sg, other);
        }
      }
    }
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      float lo, hi;
      f2_unpack(A[k], lo, hi);
      amax = fmax3(amax, fabsf(lo), fabsf(hi));
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if (lane == 0) s_max[warp] = amax;
  __syncthreads();
  amax = s_max[0];
#pragma unroll
  for (int w = 1; w < kQkThreads / 32; ++w) amax = fmaxf(amax, s_max[w]);
  const float f = amax > 0.f ? 448.0f / amax : 0.f;
  const uint64_t f2 = f2_pack(f, f);
  if (threadIdx.x == 0) (is_q ? q_scale : k_scale)[blk] = amax * cfac;
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    const int r = t * 128 + warp * 16 + g * 8 + rsub;
    if (r < N) {
      uint32_t c[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {  // channels 4e .. 4e+3, the lowest in the lowest byte
        float v0, v1, v2, v3;
        f2_unpack(f2_mul(y[g][2 * e], f2), v0, v1);
        f2_unpack(f2_mul(y[g][2 * e + 1], f2), v2, v3);
        c[e] = e4m3x2(v0, v1) | (e4m3x2(v2, v3) << 16);
      }
      uint4* o = reinterpret_cast<uint4*>(dst + static_cast<size_t>(r) * D + 32 * sub);
      o[0] = make_uint4(c[0], c[1], c[2], c[3]);
      o[1] = make_uint4(c[4], c[5], c[6], c[7]);
    }
  }
}

// V, d = 128, in three steps over (head, 128-row block) CTAs, every access
// coalesced:
//   1. channel maxima of the block, merged into v_scale by atomicMax on the
//      fp32 bit patterns (non-negative floats order like their bits; the max
//      does not depend on the order, so the result is deterministic);
//   2. each block encodes with f_c = 448 / amax_c and writes its 128 keys of
//      every channel into the transposed codes through a shared-memory tile;
//   3. v_scale <- amax * fl32(1/448) in place.
// v_scale must be zero before step 1 (the launcher clears it).
constexpr int kVThreads = 256;

template <bool BF16>
__global__ void __launch_bounds__(kVThreads)
    fa_fp8_v_amax_kernel(const uint16_t* __restrict__ v, unsigned int* __restrict__ v_amax_bits,
                         int N, int T) {
  constexpr int D = 128;
  __shared__ float s_max[kVThreads / 32][D];
  const int head = blockIdx.x / T;
  const int t = blockIdx.x % T;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint16_t* src = v + static_cast<size_t>(head) * N * D;
  uint2 raw[16];
#pragma unroll
  for (int rr = 0; rr < 16; ++rr) {
    const int r = t * 128 + warp * 16 + rr;
    raw[rr] = r < N ? *reinterpret_cast<const uint2*>(src + static_cast<size_t>(r) * D + 4 * lane)
                    : make_uint2(0u, 0u);
  }
  float m[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int rr = 0; rr < 16; ++rr) {
    m[0] = fmaxf(m[0], fabsf(to_f32<BF16>(static_cast<uint16_t>(raw[rr].x & 0xFFFFu))));
    m[1] = fmaxf(m[1], fabsf(to_f32<BF16>(static_cast<uint16_t>(raw[rr].x >> 16))));
    m[2] = fmaxf(m[2], fabsf(to_f32<BF16>(static_cast<uint16_t>(raw[rr].y & 0xFFFFu))));
    m[3] = fmaxf(m[3], fabsf(to_f32<BF16>(static_cast<uint16_t>(raw[rr].y >> 16))));
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) s_max[warp][4 * lane + e] = m[e];
  __syncthreads();
  if (threadIdx.x < D) {
    float a = s_max[0][threadIdx.x];
#pragma unroll
    for (int w = 1; w < kVThreads / 32; ++w) a = fmaxf(a, s_max[w][threadIdx.x]);
    atomicMax(v_amax_bits + static_cast<size_t>(head) * D + threadIdx.x, __float_as_uint(a));
  }
}

template <bool BF16>
__global__ void __launch_bounds__(kVThreads)
    fa_fp8_v_encode_kernel(const uint16_t* __restrict__ v, const float* __restrict__ v_amax,
                           uint8_t* __restrict__ v8t, int N, int Np, int T) {
  constexpr int D = 128;
  // Codes of the block, channel-major: row c holds keys t*128 .. t*128 + 127
  // (+4 bytes of padding per row against bank conflicts on the transposed writes).
  __shared__ uint32_t s_codes[D][128 / 4 + 1];
  const int head = blockIdx.x / T;
  const int t = blockIdx.x % T;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint16_t* src = v + static_cast<size_t>(head) * N * D;
  float f[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float a = v_amax[static_cast<size_t>(head) * D + 4 * lane + e];
    f[e] = a > 0.f ? 448.0f / a : 0.f;
  }
  // warp w encodes rows 16w .. 16w + 15 (channels 4 lane .. 4 lane + 3 per lane);
  // four consecutive rows' codes of one channel form one 32-bit word
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t word[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int rl = warp * 16 + q * 4 + b;  // row within the block
      const int r = t * 128 + rl;
      uint2 w = make_uint2(0u, 0u);
      if (r < N) w = *reinterpret_cast<const uint2*>(src + static_cast<size_t>(r) * D + 4 * lane);
      const float x[4] = {to_f32<BF16>(static_cast<uint16_t>(w.x & 0xFFFFu)),
                          to_f32<BF16>(static_cast<uint16_t>(w.x >> 16)),
                          to_f32<BF16>(static_cast<uint16_t>(w.y & 0xFFFFu)),
                          to_f32<BF16>(static_cast<uint16_t>(w.y >> 16))};
#pragma unroll
      for (int e = 0; e < 4; ++e) word[e] |= (r < N ? e4m3(x[e] * f[e]) : 0u) << (8 * b);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) s_codes[4 * lane + e][warp * 4 + q] = word[e];
  }
  __syncthreads();
  // row c of the output gets keys t*128 .. t*128 + 127 of channel c, as 32 words
  uint8_t* dst = v8t + static_cast<size_t>(head) * D * Np;
  const int nbytes = (t * 128 + 128 <= Np) ? 128 : Np - t * 128;  // the last block may be short
  for (int i = threadIdx.x; i < D * 32; i += kVThreads) {
    const int c = i >> 5;
    const int wi = i & 31;
    if (4 * wi < nbytes)
      *reinterpret_cast<uint32_t*>(dst + static_cast<size_t>(c) * Np + t * 128 + 4 * wi) = s_codes[c][wi];
  }
}

__global__ void fa_fp8_v_scale_kernel(float* __restrict__ v_scale, int n, float cfac) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) v_scale[i] = v_scale[i] * cfac;  // the slot holds amax until now
}

}  // namespace

cudaError_t launch_quantize_fp8(const AttnShape& s, const Fp8QuantArgs& a, cudaStream_t stream) {
  const int T = (s.N + 127) / 128;
  const int qb = s.B * s.Hq * T, kb = s.B * s.Hkv * T;
  const float cfac_qk = a.signs ? static_cast<float>(1.0 / (448.0 * std::sqrt(128.0)))
                                : static_cast<float>(1.0 / 448.0);
  const float cfac_v = static_cast<float>(1.0 / 448.0);
  if (s.bf16)
    fa_fp8_qk_kernel<true><<<qb + kb, kQkThreads, 0, stream>>>(
        static_cast<const uint16_t*>(a.q), static_cast<const uint16_t*>(a.k), a.signs, a.q8, a.k8,
        a.q_scale, a.k_scale, qb, s.N, T, cfac_qk);
  else
    fa_fp8_qk_kernel<false><<<qb + kb, kQkThreads, 0, stream>>>(
        static_cast<const uint16_t*>(a.q), static_cast<const uint16_t*>(a.k), a.signs, a.q8, a.k8,
        a.q_scale, a.k_scale, qb, s.N, T, cfac_qk);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int heads_kv = s.B * s.Hkv;
  const int nsc = heads_kv * 128;
  if ((e = cudaMemsetAsync(a.v_scale, 0, sizeof(float) * nsc, stream)) != cudaSuccess) return e;
  if (s.bf16)
    fa_fp8_v_amax_kernel<true><<<heads_kv * T, kVThreads, 0, stream>>>(
        static_cast<const uint16_t*>(a.v), reinterpret_cast<unsigned int*>(a.v_scale), s.N, T);
  else
    fa_fp8_v_amax_kernel<false><<<heads_kv * T, kVThreads, 0, stream>>>(
        static_cast<const uint16_t*>(a.v), reinterpret_cast<unsigned int*>(a.v_scale), s.N, T);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (s.bf16)
    fa_fp8_v_encode_kernel<true><<<heads_kv * T, kVThreads, 0, stream>>>(
        static_cast<const uint16_t*>(a.v), a.v_scale, a.v8t, s.N, a.Np, T);
  else
    fa_fp8_v_encode_kernel<false><<<heads_kv * T, kVThreads, 0, stream>>>(
        static_cast<const uint16_t*>(a.v), a.v_scale, a.v8t, s.N, a.Np, T);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  fa_fp8_v_scale_kernel<<<(nsc + 255) / 256, 256, 0, stream>>>(a.v_scale, nsc, cfac_v);
  return cudaGetLastError();
}

}  // namespace fa
