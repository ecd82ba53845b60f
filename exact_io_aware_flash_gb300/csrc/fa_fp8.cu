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

// Q and K, d = 128.  One CTA (8 warps) per (tensor, head, 128-row block); warp w
// owns rows 16w .. 16w + 15 of the block, lane l channels 4l .. 4l + 3.
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
  const bool is_q = static_cast<int>(blockIdx.x) < q_blocks;
  const int blk = is_q ? blockIdx.x : blockIdx.x - q_blocks;  // head * T + block
  const int head = blk / T;
  const int t = blk % T;
  const uint16_t* src = (is_q ? q : k) + static_cast<size_t>(head) * N * D;
  uint8_t* dst = (is_q ? q8 : k8) + static_cast<size_t>(head) * N * D;
  bool neg[4] = {false, false, false, false};
  if (signs) {
#pragma unroll
    for (int e = 0; e < 4; ++e) neg[e] = signs[4 * lane + e] < 0;
  }
  float y[16][4];
  float amax = 0.f;
#pragma unroll
  for (int rr = 0; rr < 16; ++rr) {
    const int r = t * 128 + warp * 16 + rr;
    float a[4] = {0.f, 0.f, 0.f, 0.f};
    if (r < N) {
      const uint2 w = *reinterpret_cast<const uint2*>(src + static_cast<size_t>(r) * D + 4 * lane);
      a[0] = to_f32<BF16>(static_cast<uint16_t>(w.x & 0xFFFFu));
      a[1] = to_f32<BF16>(static_cast<uint16_t>(w.x >> 16));
      a[2] = to_f32<BF16>(static_cast<uint16_t>(w.y & 0xFFFFu));
      a[3] = to_f32<BF16>(static_cast<uint16_t>(w.y >> 16));
    }
    if (signs) {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (neg[e]) a[e] = -a[e];
      // Butterfly stage h pairs channel i (bit h clear) with i + h: (a + b, a - b).
      // h = 1, 2: inside the lane's four channels.
      float b0 = a[0] + a[1], b1 = a[0] - a[1], b2 = a[2] + a[3], b3 = a[2] - a[3];
      a[0] = b0 + b2;
      a[2] = b0 - b2;
      a[1] = b1 + b3;
      a[3] = b1 - b3;
      // h = 4 .. 64: channel 4l + e pairs with 4(l ^ m) + e, m = h / 4.
#pragma unroll
      for (int m = 1; m < 32; m <<= 1) {
        const bool lower = (lane & m) == 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float other = __shfl_xor_sync(0xffffffffu, a[e], m);
          a[e] = lower ? a[e] + other : other - a[e];
        }
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      y[rr][e] = a[e];
      amax = fmaxf(amax, fabsf(a[e]));
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
  if (threadIdx.x == 0) (is_q ? q_scale : k_scale)[blk] = amax * cfac;
#pragma unroll
  for (int rr = 0; rr < 16; ++rr) {
    const int r = t * 128 + warp * 16 + rr;
    if (r < N) {
      const uint32_t c = e4m3(y[rr][0] * f) | (e4m3(y[rr][1] * f) << 8) | (e4m3(y[rr][2] * f) << 16) |
                         (e4m3(y[rr][3] * f) << 24);
      *reinterpret_cast<uint32_t*>(dst + static_cast<size_t>(r) * D + 4 * lane) = c;
    }
  }
}

// V, d = 128.  One CTA per (head, 16-channel slab): pass 1 takes the slab's channel
// maxima over all N rows, pass 2 encodes and writes the codes transposed, row c of
// the [d][Np] output holding channel c of every key (keys N .. Np-1 are zero).
constexpr int kVThreads = 256;
constexpr int kVSlab = 16;

template <bool BF16>
__global__ void __launch_bounds__(kVThreads)
    fa_fp8_v_kernel(const uint16_t* __restrict__ v, uint8_t* __restrict__ v8t,
                    float* __restrict__ v_scale, int N, int Np, float cfac) {
  constexpr int D = 128;
  __shared__ float s_max[kVThreads / 32][kVSlab];
  __shared__ float s_f[kVSlab];
  const int head = blockIdx.x / (D / kVSlab);
  const int c0 = (blockIdx.x % (D / kVSlab)) * kVSlab;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint16_t* src = v + static_cast<size_t>(head) * N * D + c0;
  float m[kVSlab];
#pragma unroll
  for (int c = 0; c < kVSlab; ++c) m[c] = 0.f;
  for (int r = threadIdx.x; r < N; r += kVThreads) {
    const uint4* p = reinterpret_cast<const uint4*>(src + static_cast<size_t>(r) * D);
    const uint4 w0 = p[0], w1 = p[1];
    const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
    for (int c = 0; c < kVSlab; ++c)
      m[c] = fmaxf(m[c], fabsf(to_f32<BF16>(static_cast<uint16_t>(w[c / 2] >> (16 * (c & 1))))));
  }
#pragma unroll
  for (int c = 0; c < kVSlab; ++c) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m[c] = fmaxf(m[c], __shfl_xor_sync(0xffffffffu, m[c], off));
    if (lane == 0) s_max[warp][c] = m[c];
  }
  __syncthreads();
  if (threadIdx.x < kVSlab) {
    float a = s_max[0][threadIdx.x];
#pragma unroll
    for (int w = 1; w < kVThreads / 32; ++w) a = fmaxf(a, s_max[w][threadIdx.x]);
    s_f[threadIdx.x] = a > 0.f ? 448.0f / a : 0.f;
    v_scale[static_cast<size_t>(head) * D + c0 + threadIdx.x] = a * cfac;
  }
  __syncthreads();
  float f[kVSlab];
#pragma unroll
  for (int c = 0; c < kVSlab; ++c) f[c] = s_f[c];
  uint8_t* dst = v8t + (static_cast<size_t>(head) * D + c0) * Np;
  for (int r = threadIdx.x; r < Np; r += kVThreads) {
    uint32_t w[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (r < N) {
      const uint4* p = reinterpret_cast<const uint4*>(src + static_cast<size_t>(r) * D);
      const uint4 w0 = p[0], w1 = p[1];
      w[0] = w0.x; w[1] = w0.y; w[2] = w0.z; w[3] = w0.w;
      w[4] = w1.x; w[5] = w1.y; w[6] = w1.z; w[7] = w1.w;
    }
#pragma unroll
    for (int c = 0; c < kVSlab; ++c) {
      const float x = to_f32<BF16>(static_cast<uint16_t>(w[c / 2] >> (16 * (c & 1))));
      dst[static_cast<size_t>(c) * Np + r] = static_cast<uint8_t>(r < N ? e4m3(x * f[c]) : 0u);
    }
  }
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
  const int vb = s.B * s.Hkv * (128 / kVSlab);
  if (s.bf16)
    fa_fp8_v_kernel<true><<<vb, kVThreads, 0, stream>>>(static_cast<const uint16_t*>(a.v), a.v8t,
                                                        a.v_scale, s.N, a.Np, cfac_v);
  else
    fa_fp8_v_kernel<false><<<vb, kVThreads, 0, stream>>>(static_cast<const uint16_t*>(a.v), a.v8t,
                                                         a.v_scale, s.N, a.Np, cfac_v);
  return cudaGetLastError();
}

}  // namespace fa
