// fa_backward_noalloc: the backward pass for callers that cannot allocate
// device memory.  Its scratch (the D vector that fa_backward otherwise takes
// as a caller-provided workspace) lives in one
// fixed-size array that is part of the library's device image.  It exists
// only on the library side: the attention method itself has no counterpart.
#include "../../include/fa.h"
#include "fa_internal.h"

#include <cuda_runtime.h>

#include <mutex>

namespace {

// FA_NOALLOC_SCRATCH_BYTES (40 MiB), 256-byte aligned.  Loaded with the
// library's module, so every GPU that uses the library holds it until the
// process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

struct ScratchState {
  std::once_flag once;
  cudaError_t status = cudaSuccess;
  void* ptr = nullptr;
};

ScratchState g_scratch[kMaxDevices];

}  // namespace

extern "C" {

int fa_backward_noalloc(const void* q, const void* k, const void* v, const void* o,
                        const float* lse, const void* dO, void* dq, void* dk, void* dv, int B,
                        int Hq, int Hkv, int N, int d, int causal, float scale, int dtype,
                        void* stream) {
  const size_t need = fa_backward_workspace_size(B, Hq, N, d);
  if (need == 0) return fa::set_last_error(FA_ERR_INVALID, "sizes must be positive");
  if (need > static_cast<size_t>(FA_NOALLOC_SCRATCH_BYTES))
    return fa::set_last_error(
        FA_ERR_UNSUPPORTED,
        "fa_backward_noalloc: these sizes need %zu bytes of scratch, more than the %d-byte built-in "
        "scratch array (use fa_backward with a caller-provided workspace)",
        need, FA_NOALLOC_SCRATCH_BYTES);
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fa::set_last_error(FA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fa::set_last_error(FA_ERR_UNSUPPORTED, "device index %d", dev);
  ScratchState& st = g_scratch[dev];
  // Once per device, with that device current: the device address of the
  // array (in host code its name is only a host-side stand-in, never a
  // device address).
  std::call_once(st.once, [&st]() {
    void* p = nullptr;
    st.status = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (st.status == cudaSuccess) st.ptr = p;
  });
  if (st.status != cudaSuccess || st.ptr == nullptr)
    return fa::set_last_error(FA_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s",
                              cudaGetErrorString(st.status));
  return fa_backward(q, k, v, o, lse, dO, dq, dk, dv, st.ptr,
                     static_cast<size_t>(FA_NOALLOC_SCRATCH_BYTES), B, Hq, Hkv, N, d, causal,
                     scale, dtype, stream);
}

}  // extern "C"
