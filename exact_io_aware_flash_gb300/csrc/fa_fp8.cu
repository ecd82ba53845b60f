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
  float y[2][32];
  float amax = 0.f;
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    float* a = y[g];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t w[4] = {raw[g][c].x, raw[g][c].y, raw[g][c].z, raw[g][c].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        a[8 * c + 2 * e] = to_f32<BF16>(static_cast<uint16_t>(w[e] & 0xFFFFu));
        a[8 * c + 2 * e + 1] = to_f32<BF16>(static_cast<uint16_t>(w[e] >> 16));
      }
    }
    if (signs) {
#pragma unroll
      for (int e = 0; e < 32; ++e)
        if (signs[32 * sub + e] < 0) a[e] = -a[e];
      // Butterfly stage h pairs channel i (bit h clear) with i + h: (a + b, a - b).
#pragma unroll
      for (int h = 1; h < 32; h <<= 1) {
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if ((e & h) == 0) {
            const float lo = a[e], hi = a[e + h];
            a[e] = lo + hi;
            a[e + h] = lo - hi;
          }
      }
      // h = 32, 64: channel 32s + e pairs with 32(s ^ m) + e, m = h / 32.
#pragma unroll
      for (int m = 1; m < 4; m <<= 1) {
        const bool lower = (sub & m) == 0;
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float other = __shfl_xor_sync(0xffffffffu, a[e], m);
          a[e] = lower ? a[e] + other : other - a[e];
        }
      }
    }
#pragma unroll
    for (int e = 0; e < 32; ++e) amax = fmaxf(amax, fabsf(a[e]));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if (lane == 0) s_max[warp] = amax;
  __syncthreads();
  amax = s_max[0];
#pragma unroll
  for (int w = 1; w < kQkThreads / 32; ++w) amax = fmaxf(amax, s_max[w]);
  const float f = amax > 0.f ? 448.0f / amax : 0.f;
  if (threadIdx.x == 0) (is_q ? q_scale : k_scale)[blk] = amax * cfac;
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    const int r = t * 128 + warp * 16 + g * 8 + rsub;
    if (r < N) {
      uint32_t c[8];
#pragma unroll
      for (int e = 0; e < 8; ++e)
        c[e] = e4m3(y[g][4 * e] * f) | (e4m3(y[g][4 * e + 1] * f) << 8) |
               (e4m3(y[g][4 * e + 2] * f) << 16) | (e4m3(y[g][4 * e + 3] * f) << 24);
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
