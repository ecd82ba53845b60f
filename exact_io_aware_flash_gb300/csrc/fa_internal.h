// Host-side interface between the C-ABI front end (fa_api.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace fa {

struct AttnShape {
  int B, Hq, Hkv, N, d;
  int causal;
  float scale;
  int bf16;  // 1 = bfloat16, 0 = float16
  // > 0: causal sliding window, key k visible to query i iff i - window < k <= i
  // (requires causal = 1 and window < N); 0: none
  int window;
};

// Tensor maps over [B*H, N, d] 16-bit tensors, box {64, 128, 1}, 128-byte swizzle.
struct FwdArgs {
  CUtensorMap tm_q, tm_k, tm_v;
  void* o;
  float* lse;
  int* err;
  // e4m3 inputs only (launch_forward_fp8): dequantization scales per 128-row
  // block of Q [B*Hq][T] and K [B*Hkv][T], and per channel of V [B*Hkv][d]
  const float* q_scale;
  const float* k_scale;
  const float* v_scale;
};

struct BwdArgs {
  CUtensorMap tm_q, tm_k, tm_v, tm_do, tm_o;
  // Store maps over dq [B*Hq, N, d] and dk, dv [B*Hkv, N, d]: box {64, 32, 1},
  // 128-byte swizzle (one warp's 32 rows of a 128-row tile per store).
  CUtensorMap tm_dq, tm_dk, tm_dv;
  const void* o;
  const void* dO;
  const float* lse;
  float* D;  // [B*Hq*N], written by the dQ kernel, read by the dK/dV kernel
  void* dq;
  void* dk;
  void* dv;
  int* err;
  // may be null: recorded before the dQ kernel, between it and the dK/dV
  // kernel, and after the dK/dV kernel
  cudaEvent_t ev_before_dq;
  cudaEvent_t ev_before_dkdv;
  cudaEvent_t ev_after_dkdv;
};

// Split-KV forward (decoding): q [B, Hq, Nq, d] seen as [B*Hkv, (Hq/Hkv)*Nq, d].
struct DecodeArgs {
  CUtensorMap tm_q, tm_k, tm_v;
  void* o;
  float* lse;
  float* o_part;    // [splits][B*Hq*Nq][d] fp32 (splits > 1)
  float* lse_part;  // [splits][B*Hq*Nq]
  int Nq, Nk, splits, chunk_tiles;
  int* err;
};

// FP8 (e4m3) quantization of 16-bit Q, K, V (d = 128): codes q8 [B*Hq][N][d],
// k8 [B*Hkv][N][d], v8t [B*Hkv][d][Np]; scales per 128-row block (Q, K) and per
// channel (V).  signs: d bytes of +1/-1 on the device, or null for no rotation.
struct Fp8QuantArgs {
  const void* q;
  const void* k;
  const void* v;
  const signed char* signs;
  uint8_t* q8;
  uint8_t* k8;
  uint8_t* v8t;
  float* q_scale;  // [B*Hq][ceil(N/128)]
  float* k_scale;  // [B*Hkv][ceil(N/128)]
  float* v_scale;  // [B*Hkv][d]
  int Np;          // row stride of v8t in bytes: N rounded up to a multiple of 16
};

// Each returns cudaSuccess or the launch error.  `stream` is the caller's.
cudaError_t launch_forward(const AttnShape& s, const FwdArgs& a, cudaStream_t stream);
// e4m3 codes (tm_q, tm_k over [B*H][N][d] bytes; tm_v over the transposed V
// codes [B*Hkv][d][Np]), d = 128, bfloat16 O.
cudaError_t launch_forward_fp8(const AttnShape& s, const FwdArgs& a, cudaStream_t stream);
cudaError_t launch_backward(const AttnShape& s, const BwdArgs& a, cudaStream_t stream);
// One-pass backward (fa_bwd_atomic.cu): a.D and dq_acc ([B*Hq][N][d] fp32) are
// workspace, overwritten; tm_dq and ev_* as for launch_backward (the events
// bracket the preprocessing kernel and the main kernel).
cudaError_t launch_backward_atomic(const AttnShape& s, const BwdArgs& a, float* dq_acc,
                                   cudaStream_t stream);
cudaError_t launch_decode(const AttnShape& s, const DecodeArgs& a, cudaStream_t stream);
cudaError_t launch_quantize_fp8(const AttnShape& s, const Fp8QuantArgs& a, cudaStream_t stream);

// Raises a kernel's dynamic shared-memory limit to `bytes` once per device
// (cudaFuncSetAttribute is a host round trip; calls after the first are free).
cudaError_t set_smem_once(const void* kernel, int bytes, int slot);

// Streaming multiprocessors of the current device (cached per device).
int sm_count();

// Records `fmt` as the calling thread's fa_last_error() message; returns `code`.
int set_last_error(int code, const char* fmt, ...);

// Shared-memory bytes the forward kernel needs for head dimension d (for checks).
size_t forward_smem_bytes(int d);
size_t backward_smem_bytes(int d);
size_t backward_atomic_smem_bytes(int d);
size_t decode_smem_bytes(int d);

}  // namespace fa
