// fa_backward_noalloc: the backward pass for callers that cannot allocate
// device memory.  Its scratch (the D vector that fa_backward otherwise takes
// as a caller-provided workspace) lives in one fixed-size array in the
// library's device code.  It exists only on the library side: the attention
// method itself has no counterpart.
//
// The library is built without relocatable device code and the CUDA runtime
// loads modules lazily, so the array is placed in device memory when this
// file's module is first loaded on a device -- in practice on the first
// fa_backward_noalloc call on that device, by the address lookup below --
// not when the library is loaded.
#include "../../include/fa.h"
#include "fa_internal.h"

#include <cuda_runtime.h>

#include <mutex>

namespace {

// FA_NOALLOC_SCRATCH_BYTES (40 MiB), 256-byte aligned.  Once placed on a
// device it stays there until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// Device address of the array per device; null until a lookup succeeds.  A
// failed lookup (e.g. the device had no memory left to place the module) is
// not remembered: the next call tries again.
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

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
  // With the device current, the device address of the array (in host code
  // its name is only a host-side stand-in, never a device address).  Looked
  // up once per device; the lookup is what places the array on the device.
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess || p == nullptr) {
        (void)cudaGetLastError();  // do not leave the failure for the caller's next check
        return fa::set_last_error(FA_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s",
                                  cudaGetErrorString(e));
      }
      g_scratch_ptr[dev] = p;
    }
    scratch = g_scratch_ptr[dev];
  }
  return fa_backward(q, k, v, o, lse, dO, dq, dk, dv, scratch,
                     static_cast<size_t>(FA_NOALLOC_SCRATCH_BYTES), B, Hq, Hkv, N, d, causal,
                     scale, dtype, stream);
}

}  // extern "C"
