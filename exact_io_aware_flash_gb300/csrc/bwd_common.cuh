// Pieces shared by the backward kernels: tile constants, 16-bit packing,
// shared-memory matrix descriptors over 128-byte-swizzled tiles, the staging of
// TMEM rows for TMA stores, and the launch-order head grouping.
#pragma once

#include "ptx.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace fa {
namespace bwd {

constexpr int kBlk = 128;          // rows per tile (keys and queries)
constexpr int kAtomBytes = 16384;  // 128 rows x 128 bytes
constexpr float kLog2e = 1.4426950408889634f;

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

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) &
                                    ~static_cast<uintptr_t>(1023));
}

// K-major operand (rows of 128 bytes, 8-row groups 1024 bytes apart), k-step ks of 16 elements.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile, int ks) {
  return sdesc_sw128(tile + (ks >> 2) * kAtomBytes + (ks & 3) * 32, 16, 1024);
}
// MN-major operand over a [128 K-rows][D] tile, k-step ks of 16 K-rows.
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t tile, int ks) {
  return sdesc_sw128(tile + ks * 2048, kAtomBytes, 1024);
}
// The same descriptors from the k-step-0 descriptor d0 of the tile: only the
// start-address field (bits 0-13, address >> 4) moves, and shared-memory
// addresses stay below 2^18, so one add of a compile-time constant per
// operand replaces the full encoding in the MMA-issuing thread, whose
// instruction count is on every iteration's critical path.
__device__ __forceinline__ uint64_t kmajor_step(uint64_t d0, int ks) {
  return d0 + static_cast<uint64_t>(((ks >> 2) * kAtomBytes + (ks & 3) * 32) >> 4);
}
__device__ __forceinline__ uint64_t mnmajor_step(uint64_t d0, int ks) {
  return d0 + static_cast<uint64_t>((ks * 2048) >> 4);
}

// TMEM row (D fp32 columns at taddr) * mul -> 16-bit row `row` of a 128-row
// tile in shared memory, in the layout a 128-byte-swizzled TMA box expects:
// 64-column atoms of 128 x 128 bytes, 16-byte chunk c of row r at chunk
// position c ^ (r mod 8).  Eight consecutive rows cover all 32 banks, so a
// warp's 16-byte stores are conflict-free.
template <int D, bool BF16>
__device__ __forceinline__ void stage_row_from_tmem(uint32_t taddr, uint8_t* tile, int row,
                                                    float mul) {
#pragma unroll
  for (int c = 0; c < D; c += 64) {  // one 64-column atom per TMEM round trip
    uint32_t v[64];
    tmem_ld32(taddr + c, v);
    tmem_ld32(taddr + c + 32, v + 32);
    tmem_ld_wait();
    reg_fence<64>(v);
    uint8_t* rowp = tile + (c / 64) * kAtomBytes + row * 128;
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {  // 16-byte chunk ch: columns c + 8*ch .. +7
      uint32_t pk[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        pk[e] = pack2<BF16>(__uint_as_float(v[8 * ch + 2 * e]) * mul,
                            __uint_as_float(v[8 * ch + 2 * e + 1]) * mul);
      *reinterpret_cast<uint4*>(rowp + ((ch ^ (row & 7)) * 16)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
  }
}

// First key tile a causal sliding window of `window` keys exposes to query
// tile t: its first row, t*128, sees keys t*128 - window + 1 .. t*128.
__device__ __forceinline__ int window_first_tile(int t, int window) {
  const int first_key = t * kBlk - window + 1;
  return first_key > 0 ? first_key / kBlk : 0;
}

// Heads scheduled side by side so that the operands they stream (per_head_bytes
// each) stay within about a quarter of the 129 MB L2: 16 heads at N = 4096,
// d = 128 (2 MB each), 4 at N = 16384.
inline int l2_head_group(long per_head_bytes) {
  long g = (32L << 20) / (per_head_bytes > 0 ? per_head_bytes : 1);
  return static_cast<int>(g < 1 ? 1 : (g > 64 ? 64 : g));
}

}  // namespace bwd
}  // namespace fa
