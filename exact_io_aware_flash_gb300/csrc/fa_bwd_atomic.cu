// One-pass backward: dQ accumulated across key tiles with atomic adds.
//
// The primer ("FlashAttention Primer: IO-Aware Attention, from FA1 to FA4",
// section "Backward pass: recomputation instead of storage") describes the
// default backward as accumulating dQ across thread blocks with atomic adds,
// which makes it bitwise nondeterministic, and a deterministic option as
// slower.  This file is that default form; fa_bwd.cu is the deterministic one.
//
// Kernels, in launch order on the caller's stream:
//   fa_bwd_pre_kernel      D_r = sum_c dO_rc O_rc for every query row, and the
//                          row's fp32 dQ accumulator set to zero   (HBM-bound)
//   fa_bwd_onepass_kernel  one CTA per (KV head, 128-key tile j): the key-tile
//                          pass of dkdv_body.cuh with its dQ share, 5 products
//                          per (query tile, key tile) pair:
//                            S^T, dP^T, dV += P^T dO, dK += dS^T Q, dQ_i += dS K_j
//                          dQ_i's partial sums go into the accumulator with
//                          red.global.add (fp32, in L2)
//   fa_bwd_post_kernel     dQ = scale * accumulator -> 16-bit        (HBM-bound)
#include "dkdv_body.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

using namespace bwd;

constexpr int kEwThreads = 256;  // the two row-wise kernels

// Thread group of D/8 threads per row, each with one 16-byte chunk (8 elements).
template <int D, bool BF16>
__global__ void __launch_bounds__(kEwThreads)
    fa_bwd_pre_kernel(const uint4* __restrict__ o, const uint4* __restrict__ dO, float* __restrict__ Drow,
                      float4* __restrict__ dq_acc, long long rows) {
  constexpr int kTpr = D / 8;
  constexpr int kRowsPerBlock = kEwThreads / kTpr;
  const int sub = threadIdx.x % kTpr;
  for (long long base = static_cast<long long>(blockIdx.x) * kRowsPerBlock; base < rows;
       base += static_cast<long long>(gridDim.x) * kRowsPerBlock) {
    const long long r = base + threadIdx.x / kTpr;
    const bool valid = r < rows;
    float acc = 0.f;
    if (valid) {
      const long long c = r * kTpr + sub;
      const uint4 a = o[c];
      const uint4 g = dO[c];
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
      const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 af = unpack2<BF16>(aw[e]);
        const float2 gf = unpack2<BF16>(gw[e]);
        acc = fmaf(af.x, gf.x, acc);
        acc = fmaf(af.y, gf.y, acc);
      }
      const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
      dq_acc[2 * c] = z;
      dq_acc[2 * c + 1] = z;
    }
    // groups of kTpr lanes are aligned within the warp, so xor offsets below
    // kTpr stay inside the row's group
#pragma unroll
    for (int off = kTpr / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (valid && sub == 0) Drow[r] = acc;
  }
}

template <int D, bool BF16, bool WIN>
__global__ void __launch_bounds__(kOnePassThreads, 1)
    fa_bwd_onepass_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                          const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                          const float* __restrict__ lse, const float* __restrict__ Drow,
                          float* __restrict__ dq_acc, int heads, int head_group, int Hq, int Hkv, int N,
                          int causal, int window, float scale, int* err) {
  dkdv_body<D, BF16, WIN, true>(&tm_q, &tm_k, &tm_v, &tm_do, &tm_dk, &tm_dv, lse, Drow, dq_acc, heads,
                                head_group, Hq, Hkv, N, causal, window, scale, err);
}

// Eight accumulator floats -> eight 16-bit dQ elements per thread and step.
template <bool BF16>
__global__ void __launch_bounds__(kEwThreads)
    fa_bwd_post_kernel(const float4* __restrict__ dq_acc, uint4* __restrict__ dq, long long n8,
                       float scale) {
  for (long long x = static_cast<long long>(blockIdx.x) * kEwThreads + threadIdx.x; x < n8;
       x += static_cast<long long>(gridDim.x) * kEwThreads) {
    const float4 a = dq_acc[2 * x];
    const float4 b = dq_acc[2 * x + 1];
    dq[x] = make_uint4(pack2<BF16>(a.x * scale, a.y * scale), pack2<BF16>(a.z * scale, a.w * scale),
                       pack2<BF16>(b.x * scale, b.y * scale), pack2<BF16>(b.z * scale, b.w * scale));
  }
}

// Grid of a grid-stride element-wise kernel: enough blocks for `work` items of
// `per_block` each, at most 16 resident blocks per SM.
unsigned ew_grid(long long work, int per_block) {
  const long long need = (work + per_block - 1) / per_block;
  const long long cap = 16LL * sm_count();
  return static_cast<unsigned>(need < cap ? (need > 0 ? need : 1) : cap);
}

template <int D, bool BF16, bool WIN>
cudaError_t launch_atomic_t(const AttnShape& s, const BwdArgs& a, float* dq_acc, cudaStream_t stream) {
  const int T = (s.N + kBlk - 1) / kBlk;
  auto k1 = fa_bwd_onepass_kernel<D, BF16, WIN>;
  constexpr int smem1 = DkdvSmem<D, true>::kAlloc;
  const int slot = 32 + (WIN ? 4 : 0) + (D == 64 ? 0 : 2) + (BF16 ? 1 : 0);
  cudaError_t e;
  if ((e = set_smem_once(reinterpret_cast<const void*>(k1), smem1, slot)) != cudaSuccess) return e;
  // The register reallocation inside the kernel draws on threads x launch
  // registers; it is sized for 168 per thread, so refuse any other build.
  static const int launch_regs = [&] {
    cudaFuncAttributes fa{};
    return cudaFuncGetAttributes(&fa, reinterpret_cast<const void*>(k1)) == cudaSuccess ? fa.numRegs : -1;
  }();
  if (launch_regs != 168) return cudaErrorInvalidKernelImage;
  const long long rows = static_cast<long long>(s.B) * s.Hq * s.N;

  if (a.ev_before_dq && (e = cudaEventRecord(a.ev_before_dq, stream)) != cudaSuccess) return e;
  fa_bwd_pre_kernel<D, BF16><<<ew_grid(rows, kEwThreads / (D / 8)), kEwThreads, 0, stream>>>(
      static_cast<const uint4*>(a.o), static_cast<const uint4*>(a.dO), a.D,
      reinterpret_cast<float4*>(dq_acc), rows);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (a.ev_before_dkdv && (e = cudaEventRecord(a.ev_before_dkdv, stream)) != cudaSuccess) return e;
  k1<<<dim3(static_cast<unsigned>(T * s.B * s.Hkv)), kOnePassThreads, smem1, stream>>>(
      a.tm_q, a.tm_k, a.tm_v, a.tm_do, a.tm_dk, a.tm_dv, a.lse, a.D, dq_acc, s.B * s.Hkv,
      l2_head_group(4L * s.N * D * (s.Hq / s.Hkv)), s.Hq, s.Hkv, s.N, s.causal, s.window, s.scale,
      a.err);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (a.ev_after_dkdv && (e = cudaEventRecord(a.ev_after_dkdv, stream)) != cudaSuccess) return e;
  const long long n8 = rows * (D / 8);
  fa_bwd_post_kernel<BF16><<<ew_grid(n8, kEwThreads), kEwThreads, 0, stream>>>(
      reinterpret_cast<const float4*>(dq_acc), static_cast<uint4*>(a.dq), n8, s.scale);
  return cudaGetLastError();
}

}  // namespace

size_t backward_atomic_smem_bytes(int d) {
  return d == 64 ? DkdvSmem<64, true>::kAlloc : DkdvSmem<128, true>::kAlloc;
}

cudaError_t launch_backward_atomic(const AttnShape& s, const BwdArgs& a, float* dq_acc,
                                   cudaStream_t stream) {
  if (s.window > 0) {  // causal sliding window
    if (s.d == 64)
      return s.bf16 ? launch_atomic_t<64, true, true>(s, a, dq_acc, stream)
                    : launch_atomic_t<64, false, true>(s, a, dq_acc, stream);
    return s.bf16 ? launch_atomic_t<128, true, true>(s, a, dq_acc, stream)
                  : launch_atomic_t<128, false, true>(s, a, dq_acc, stream);
  }
  if (s.d == 64)
    return s.bf16 ? launch_atomic_t<64, true, false>(s, a, dq_acc, stream)
                  : launch_atomic_t<64, false, false>(s, a, dq_acc, stream);
  return s.bf16 ? launch_atomic_t<128, true, false>(s, a, dq_acc, stream)
                : launch_atomic_t<128, false, false>(s, a, dq_acc, stream);
}

}  // namespace fa
