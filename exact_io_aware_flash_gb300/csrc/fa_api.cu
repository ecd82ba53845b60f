// C ABI of libfa.so (declared in include/fa.h): argument checks, Tensor Memory
// Accelerator descriptor encoding, the device error word, and kernel launches.
// Host code only; the kernels live in fa_fwd.cu and fa_bwd.cu.
#include "../../include/fa.h"
#include "fa_internal.h"
#include "ptx.cuh"

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>
#include <string>

namespace {

// Device error word: set by a kernel whose bounded wait expired.  One per
// device (a __device__ variable is instantiated in every context).
__device__ int g_fa_error_word;

thread_local std::string t_last_error;

// Self-test of the bounded waits: one thread waits on an mbarrier that nothing
// ever completes; the wait gives up after limit_ns and raises the error word,
// exactly as a stalled pipeline stage in the attention kernels would.
__global__ void fa_selftest_wait_kernel(int* err, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    fa::mbar_init(&bar, 1);
    abort_flag = 0;
    fa::fence_mbar_init();
    (void)fa::mbar_wait_for(&bar, 0, &abort_flag, err, limit_ns);
  }
}
thread_local cudaEvent_t t_ev_hooks[3] = {nullptr, nullptr, nullptr};

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return code;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

constexpr int kMaxDevices = 64;

struct DeviceState {
  std::once_flag once;
  int status = FA_OK;
  std::string msg;
  int* err_word = nullptr;
};

DeviceState g_dev[kMaxDevices];
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;
std::string g_encode_msg;

int get_device_state(DeviceState** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(FA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(FA_ERR_UNSUPPORTED, "device index %d", dev);
  DeviceState& st = g_dev[dev];
  std::call_once(st.once, [&st, dev]() {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3) {
      st.status = FA_ERR_UNSUPPORTED;
      st.msg = "device " + std::to_string(dev) + " is sm_" + std::to_string(major) +
               std::to_string(minor) + "; this library is built for sm_103a only";
      return;
    }
    void* p = nullptr;
    cudaError_t ee = cudaGetSymbolAddress(&p, g_fa_error_word);
    if (ee != cudaSuccess) {
      st.status = FA_ERR_CUDA;
      st.msg = std::string("cudaGetSymbolAddress(error word): ") + cudaGetErrorString(ee);
      return;
    }
    st.err_word = static_cast<int*>(p);
  });
  if (st.status != FA_OK) return fail(st.status, "%s", st.msg.c_str());
  std::call_once(g_encode_once, []() {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t ee =
        cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (ee != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr) {
      g_encode_msg = "cuTensorMapEncodeTiled entry point not available";
      return;
    }
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  if (!g_encode) return fail(FA_ERR_CUDA, "%s", g_encode_msg.c_str());
  *out = &st;
  return FA_OK;
}

// [heads, N, d] 16-bit tensor, box {64, box_rows, 1}, 128-byte swizzle, zero fill out of
// bounds.  Loads use 128-row boxes; the backward's stores use 32-row boxes (one warp each).
int encode_tile_map(CUtensorMap* map, const void* base, int heads, int N, int d, int bf16,
                    const char* name, int box_rows = 128) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(heads)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                           static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(d) * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                        3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed: %d", name, (int)r);
  return FA_OK;
}

// Byte tensor [heads][rows][cols] (e4m3 codes), box {128, 128, 1}, 128-byte swizzle:
// one box is a 128 x 128-byte tile, a single swizzle atom wide.
int encode_u8_map(CUtensorMap* map, const void* base, int heads, int rows, int cols,
                  const char* name) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(heads)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols),
                           static_cast<cuuint64_t>(rows) * static_cast<cuuint64_t>(cols)};
  cuuint32_t box[3] = {128, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides,
                        box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed: %d", name, (int)r);
  return FA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_common(int B, int Hq, int Hkv, int N, int d, float scale, int dtype) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || N <= 0)
    return fail(FA_ERR_INVALID, "sizes must be positive (B=%d Hq=%d Hkv=%d N=%d)", B, Hq, Hkv, N);
  if (Hq % Hkv != 0) return fail(FA_ERR_INVALID, "Hq (%d) must be a multiple of Hkv (%d)", Hq, Hkv);
  if (!std::isfinite(scale)) return fail(FA_ERR_INVALID, "scale must be finite");
  if (d != 64 && d != 128) return fail(FA_ERR_UNSUPPORTED, "head dimension d=%d (supported: 64, 128)", d);
  if (dtype != FA_DTYPE_FP16 && dtype != FA_DTYPE_BF16)
    return fail(FA_ERR_UNSUPPORTED, "dtype %d (supported: FA_DTYPE_FP16, FA_DTYPE_BF16)", dtype);
  // One-dimensional grids enumerate (head, 128-row tile) work items; the TMA
  // head coordinate and row indices are 32-bit.
  if ((long long)B * Hq * N > 0x7fffffffLL) return fail(FA_ERR_UNSUPPORTED, "B*Hq*N exceeds 2^31-1");
  return FA_OK;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

namespace fa {

int sm_count() {
  static std::atomic<int> cached[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

cudaError_t set_smem_once(const void* kernel, int bytes, int slot) {
  // slot: a small per-kernel index; one flag per (device, slot)
  static std::atomic<int> done[kMaxDevices][64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices || slot < 0 || slot >= 64)
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (done[dev][slot].load(std::memory_order_acquire)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done[dev][slot].store(1, std::memory_order_release);
  return e;
}

int set_last_error(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return code;
}

}  // namespace fa

extern "C" {

const char* fa_version(void) { return "fa-gb300 0.1.0 (sm_103a, tcgen05/TMEM/TMA)"; }

const char* fa_last_error(void) { return t_last_error.c_str(); }

}  // extern "C"

namespace {

// Shared body of fa_forward and fa_forward_window (window > 0: causal sliding
// window narrower than N; 0: none).
int forward_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                 int Hkv, int N, int d, int causal, int window, float scale, int dtype,
                 void* stream) {
  if (!q || !k || !v || !o || !lse) return fail(FA_ERR_INVALID, "null tensor pointer");
  int rc = check_common(B, Hq, Hkv, N, d, scale, dtype);
  if (rc) return rc;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return fail(FA_ERR_UNSUPPORTED, "all tensor pointers must be 16-byte aligned");
  DeviceState* st = nullptr;
  if ((rc = get_device_state(&st))) return rc;
  fa::AttnShape s{B, Hq, Hkv, N, d, causal ? 1 : 0, scale, dtype == FA_DTYPE_BF16, window};
  fa::FwdArgs a{};
  if ((rc = encode_tile_map(&a.tm_q, q, B * Hq, N, d, s.bf16, "q"))) return rc;
  if ((rc = encode_tile_map(&a.tm_k, k, B * Hkv, N, d, s.bf16, "k"))) return rc;
  if ((rc = encode_tile_map(&a.tm_v, v, B * Hkv, N, d, s.bf16, "v"))) return rc;
  a.o = o;
  a.lse = lse;
  a.err = st->err_word;
  cudaError_t e = fa::launch_forward(s, a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(FA_ERR_CUDA, "forward launch: %s", cudaGetErrorString(e));
  return FA_OK;
}

}  // namespace

extern "C" {

int fa_forward(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
               int Hkv, int N, int d, int causal, float scale, int dtype, void* stream) {
  t_last_error.clear();
  return forward_impl(q, k, v, o, lse, B, Hq, Hkv, N, d, causal, 0, scale, dtype, stream);
}

int fa_forward_window(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                      int Hq, int Hkv, int N, int d, int window, float scale, int dtype,
                      void* stream) {
  t_last_error.clear();
  if (window < 1) return fail(FA_ERR_INVALID, "window must be at least 1 (got %d)", window);
  // A window of N or more keys hides nothing that causal masking does not.
  return forward_impl(q, k, v, o, lse, B, Hq, Hkv, N, d, 1, window < N ? window : 0, scale, dtype,
                      stream);
}

namespace {

struct SplitPlan {
  int splits, chunk_tiles;
};

// Key chunks for the split-KV forward: at least one 128-key tile per chunk,
// no empty chunk.  Chosen automatically, the split count s minimises the
// modelled time waves(s) x (chunk(s) + 2): the CTAs (one per SM at a time)
// run in ceil(base*s / SMs) waves, each as long as a chunk of ceil(KT / s)
// key tiles plus a CTA's fixed cost (prologue and epilogue, about two tiles'
// worth of loads).  A count that leaves a nearly empty last wave loses most
// of a wave's time; this picks one that fills the waves (ties: fewer splits,
// less merge work).  Chunks stay at least 4 tiles long.
SplitPlan plan_splits(int B, int Hq, int Hkv, int Nq, int Nk, int requested) {
  const long Mq = static_cast<long>(Hq / Hkv) * Nq;
  const long base = ((Mq + 127) / 128) * B * Hkv;
  const int KT = (Nk + 127) / 128;
  long want = requested;
  if (want <= 0) {
    int sms = 148;
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) sms = fa::sm_count();
    const long s_max = KT >= 8 ? KT / 4 : 1;
    long best_cost = -1;
    want = 1;
    for (long sp = 1; sp <= s_max; ++sp) {
      const long chunk = (KT + sp - 1) / sp;
      const long waves = (base * sp + sms - 1) / sms;
      const long cost = waves * (chunk + 2);
      if (best_cost < 0 || cost < best_cost) {
        best_cost = cost;
        want = sp;
      }
    }
  }
  if (want < 1) want = 1;
  if (want > KT) want = KT;
  const int chunk = static_cast<int>((KT + want - 1) / want);
  return SplitPlan{(KT + chunk - 1) / chunk, chunk};
}

size_t splitkv_ws_bytes(int B, int Hq, int Nq, int d, int splits) {
  if (splits <= 1) return 0;
  const size_t rows = static_cast<size_t>(B) * Hq * Nq;
  return round_up(static_cast<size_t>(splits) * rows * d * 4, 256) +
         round_up(static_cast<size_t>(splits) * rows * 4, 256);
}

}  // namespace

size_t fa_forward_splitkv_workspace_size(int B, int Hq, int Hkv, int Nq, int Nk, int d,
                                         int num_splits) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Nq <= 0 || Nk <= 0 || d <= 0 || Hq % Hkv) return 0;
  return splitkv_ws_bytes(B, Hq, Nq, d, plan_splits(B, Hq, Hkv, Nq, Nk, num_splits).splits);
}

int fa_forward_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int Hq, int Hkv, int Nq, int Nk, int d, float scale, int dtype,
                       int num_splits, void* workspace, size_t ws_bytes, void* stream) {
  t_last_error.clear();
  if (!q || !k || !v || !o || !lse) return fail(FA_ERR_INVALID, "null tensor pointer");
  if (Nk <= 0) return fail(FA_ERR_INVALID, "Nk must be positive");
  int rc = check_common(B, Hq, Hkv, Nq, d, scale, dtype);
  if (rc) return rc;
  if ((long long)B * Hkv * Nk > 0x7fffffffLL) return fail(FA_ERR_UNSUPPORTED, "B*Hkv*Nk exceeds 2^31-1");
  const void* ptrs[] = {q, k, v, o, lse};
  for (const void* p : ptrs)
    if (!aligned16(p)) return fail(FA_ERR_UNSUPPORTED, "all tensor pointers must be 16-byte aligned");
  DeviceState* st = nullptr;
  if ((rc = get_device_state(&st))) return rc;
  const SplitPlan plan = plan_splits(B, Hq, Hkv, Nq, Nk, num_splits);
  const size_t need = splitkv_ws_bytes(B, Hq, Nq, d, plan.splits);
  if (need > 0) {
    if (!workspace || ws_bytes < need)
      return fail(FA_ERR_INVALID, "split-KV workspace of %zu bytes is smaller than the %zu required",
                  workspace ? ws_bytes : (size_t)0, need);
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
      return fail(FA_ERR_UNSUPPORTED, "workspace must be 256-byte aligned");
  }
  const long grid = ((static_cast<long>(Hq / Hkv) * Nq + 127) / 128) * B * Hkv * plan.splits;
  if (grid > 0x7fffffffL) return fail(FA_ERR_UNSUPPORTED, "problem too large for one launch");
  fa::AttnShape s{B, Hq, Hkv, Nq, d, 0, scale, dtype == FA_DTYPE_BF16};
  fa::DecodeArgs a{};
  const int Mq = (Hq / Hkv) * Nq;
  if ((rc = encode_tile_map(&a.tm_q, q, B * Hkv, Mq, d, s.bf16, "q"))) return rc;
  if ((rc = encode_tile_map(&a.tm_k, k, B * Hkv, Nk, d, s.bf16, "k"))) return rc;
  if ((rc = encode_tile_map(&a.tm_v, v, B * Hkv, Nk, d, s.bf16, "v"))) return rc;
  a.o = o;
  a.lse = lse;
  const size_t rows = static_cast<size_t>(B) * Hq * Nq;
  a.o_part = static_cast<float*>(workspace);
  a.lse_part = need ? reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                               round_up(static_cast<size_t>(plan.splits) * rows * d * 4, 256))
                    : nullptr;
  a.Nq = Nq;
  a.Nk = Nk;
  a.splits = plan.splits;
  a.chunk_tiles = plan.chunk_tiles;
  a.err = st->err_word;
  cudaError_t e = fa::launch_decode(s, a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(FA_ERR_CUDA, "split-KV forward launch: %s", cudaGetErrorString(e));
  return FA_OK;
}

int fa_fp8_vt_stride(int N) {
  if (N <= 0 || N > 0x7fffffff - 15) return 0;
  return (N + 15) / 16 * 16;
}

int fa_forward_fp8(const void* q8, const void* k8, const void* v8t, const float* q_scale,
                   const float* k_scale, const float* v_scale, void* o, float* lse, int B, int Hq,
                   int Hkv, int N, int d, int causal, float scale, void* stream) {
  t_last_error.clear();
  if (!q8 || !k8 || !v8t || !q_scale || !k_scale || !v_scale || !o || !lse)
    return fail(FA_ERR_INVALID, "null tensor pointer");
  int rc = check_common(B, Hq, Hkv, N, d, scale, FA_DTYPE_BF16);
  if (rc) return rc;
  if (d != 128) return fail(FA_ERR_UNSUPPORTED, "FP8 path: head dimension d=%d (supported: 128)", d);
  const void* ptrs[] = {q8, k8, v8t, q_scale, k_scale, v_scale, o, lse};
  for (const void* p : ptrs)
    if (!aligned16(p)) return fail(FA_ERR_UNSUPPORTED, "all tensor pointers must be 16-byte aligned");
  DeviceState* st = nullptr;
  if ((rc = get_device_state(&st))) return rc;
  fa::AttnShape s{B, Hq, Hkv, N, d, causal ? 1 : 0, scale, 1, 0};
  fa::FwdArgs a{};
  if ((rc = encode_u8_map(&a.tm_q, q8, B * Hq, N, d, "q8"))) return rc;
  if ((rc = encode_u8_map(&a.tm_k, k8, B * Hkv, N, d, "k8"))) return rc;
  if ((rc = encode_u8_map(&a.tm_v, v8t, B * Hkv, d, fa_fp8_vt_stride(N), "v8t"))) return rc;
  a.o = o;
  a.lse = lse;
  a.err = st->err_word;
  a.q_scale = q_scale;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  cudaError_t e = fa::launch_forward_fp8(s, a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(FA_ERR_CUDA, "FP8 forward launch: %s", cudaGetErrorString(e));
  return FA_OK;
}

int fa_quantize_fp8(const void* q, const void* k, const void* v, const signed char* signs, void* q8,
                    void* k8, void* v8t, float* q_scale, float* k_scale, float* v_scale, int B,
                    int Hq, int Hkv, int N, int d, int dtype, void* stream) {
  t_last_error.clear();
  if (!q || !k || !v || !q8 || !k8 || !v8t || !q_scale || !k_scale || !v_scale)
    return fail(FA_ERR_INVALID, "null tensor pointer");
  int rc = check_common(B, Hq, Hkv, N, d, 1.0f, dtype);
  if (rc) return rc;
  if (d != 128) return fail(FA_ERR_UNSUPPORTED, "FP8 path: head dimension d=%d (supported: 128)", d);
  if (fa_fp8_vt_stride(N) == 0) return fail(FA_ERR_UNSUPPORTED, "N=%d too large for the V code layout", N);
  const void* ptrs[] = {q, k, v, q8, k8, v8t, q_scale, k_scale, v_scale};
  for (const void* p : ptrs)
    if (!aligned16(p)) return fail(FA_ERR_UNSUPPORTED, "all tensor pointers must be 16-byte aligned");
  DeviceState* st = nullptr;
  if ((rc = get_device_state(&st))) return rc;
  fa::AttnShape s{B, Hq, Hkv, N, d, 0, 1.0f, dtype == FA_DTYPE_BF16, 0};
  fa::Fp8QuantArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.signs = signs;
  a.q8 = static_cast<uint8_t*>(q8);
  a.k8 = static_cast<uint8_t*>(k8);
  a.v8t = static_cast<uint8_t*>(v8t);
  a.q_scale = q_scale;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.Np = fa_fp8_vt_stride(N);
  cudaError_t e = fa::launch_quantize_fp8(s, a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(FA_ERR_CUDA, "FP8 quantization launch: %s", cudaGetErrorString(e));
  return FA_OK;
}

size_t fa_backward_workspace_size(int B, int Hq, int N, int d) {
  if (B <= 0 || Hq <= 0 || N <= 0 || d <= 0) return 0;
  const size_t rows = static_cast<size_t>(B) * Hq * N;
  return round_up(rows * 4, 256);
}

size_t fa_backward_atomic_workspace_size(int B, int Hq, int N, int d) {
  if (B <= 0 || Hq <= 0 || N <= 0 || d <= 0) return 0;
  const size_t rows = static_cast<size_t>(B) * Hq * N;
  return round_up(rows * 4, 256) + round_up(rows * static_cast<size_t>(d) * 4, 256);
}

}  // extern "C"

namespace {

// Shared body of fa_backward, fa_backward_window (window as in forward_impl)
// and, with atomic = true, fa_backward_atomic.
int backward_impl(const void* q, const void* k, const void* v, const void* o, const float* lse,
                  const void* dO, void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes,
                  int B, int Hq, int Hkv, int N, int d, int causal, int window, float scale,
                  int dtype, void* stream, bool atomic = false) {
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv || !workspace)
    return fail(FA_ERR_INVALID, "null tensor pointer");
  int rc = check_common(B, Hq, Hkv, N, d, scale, dtype);
  if (rc) return rc;
  const size_t need = atomic ? fa_backward_atomic_workspace_size(B, Hq, N, d)
                             : fa_backward_workspace_size(B, Hq, N, d);
  if (ws_bytes < need)
    return fail(FA_ERR_INVALID, "workspace of %zu bytes is smaller than the %zu required", ws_bytes, need);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(FA_ERR_UNSUPPORTED, "workspace must be 256-byte aligned");
  const void* ptrs[] = {q, k, v, o, lse, dO, dq, dk, dv};
  for (const void* p : ptrs)
    if (!aligned16(p)) return fail(FA_ERR_UNSUPPORTED, "all tensor pointers must be 16-byte aligned");
  DeviceState* st = nullptr;
  if ((rc = get_device_state(&st))) return rc;
  fa::AttnShape s{B, Hq, Hkv, N, d, causal ? 1 : 0, scale, dtype == FA_DTYPE_BF16, window};
  fa::BwdArgs a{};
  if ((rc = encode_tile_map(&a.tm_q, q, B * Hq, N, d, s.bf16, "q"))) return rc;
  if ((rc = encode_tile_map(&a.tm_k, k, B * Hkv, N, d, s.bf16, "k"))) return rc;
  if ((rc = encode_tile_map(&a.tm_v, v, B * Hkv, N, d, s.bf16, "v"))) return rc;
  if ((rc = encode_tile_map(&a.tm_do, dO, B * Hq, N, d, s.bf16, "dO"))) return rc;
  if (!atomic) {  // the one-pass kernels read O and write dq with plain vector accesses
    if ((rc = encode_tile_map(&a.tm_o, o, B * Hq, N, d, s.bf16, "o"))) return rc;
    if ((rc = encode_tile_map(&a.tm_dq, dq, B * Hq, N, d, s.bf16, "dq", 32))) return rc;
  }
  if ((rc = encode_tile_map(&a.tm_dk, dk, B * Hkv, N, d, s.bf16, "dk", 32))) return rc;
  if ((rc = encode_tile_map(&a.tm_dv, dv, B * Hkv, N, d, s.bf16, "dv", 32))) return rc;
  a.o = o;
  a.dO = dO;
  a.lse = lse;
  a.D = static_cast<float*>(workspace);
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.err = st->err_word;
  a.ev_before_dq = t_ev_hooks[0];
  a.ev_before_dkdv = t_ev_hooks[1];
  a.ev_after_dkdv = t_ev_hooks[2];
  cudaError_t e;
  if (atomic) {
    float* dq_acc = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                             fa_backward_workspace_size(B, Hq, N, d));
    e = fa::launch_backward_atomic(s, a, dq_acc, static_cast<cudaStream_t>(stream));
  } else {
    e = fa::launch_backward(s, a, static_cast<cudaStream_t>(stream));
  }
  if (e != cudaSuccess) return fail(FA_ERR_CUDA, "backward launch: %s", cudaGetErrorString(e));
  return FA_OK;
}

}  // namespace

extern "C" {

int fa_backward(const void* q, const void* k, const void* v, const void* o, const float* lse,
                const void* dO, void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes,
                int B, int Hq, int Hkv, int N, int d, int causal, float scale, int dtype,
                void* stream) {
  t_last_error.clear();
  return backward_impl(q, k, v, o, lse, dO, dq, dk, dv, workspace, ws_bytes, B, Hq, Hkv, N, d,
                       causal, 0, scale, dtype, stream);
}

int fa_backward_window(const void* q, const void* k, const void* v, const void* o,
                       const float* lse, const void* dO, void* dq, void* dk, void* dv,
                       void* workspace, size_t ws_bytes, int B, int Hq, int Hkv, int N, int d,
                       int window, float scale, int dtype, void* stream) {
  t_last_error.clear();
  if (window < 1) return fail(FA_ERR_INVALID, "window must be at least 1 (got %d)", window);
  return backward_impl(q, k, v, o, lse, dO, dq, dk, dv, workspace, ws_bytes, B, Hq, Hkv, N, d, 1,
                       window < N ? window : 0, scale, dtype, stream);
}

int fa_backward_atomic(const void* q, const void* k, const void* v, const void* o,
                       const float* lse, const void* dO, void* dq, void* dk, void* dv,
                       void* workspace, size_t ws_bytes, int B, int Hq, int Hkv, int N, int d,
                       int causal, int window, float scale, int dtype, void* stream) {
  t_last_error.clear();
  if (window < 0) return fail(FA_ERR_INVALID, "window must be 0 (none) or at least 1 (got %d)", window);
  if (window > 0 && !causal) return fail(FA_ERR_INVALID, "a sliding window needs causal = 1");
  return backward_impl(q, k, v, o, lse, dO, dq, dk, dv, workspace, ws_bytes, B, Hq, Hkv, N, d,
                       causal, window < N ? window : 0, scale, dtype, stream, true);
}

int fa_set_backward_event_hooks(void* before_dq, void* before_dkdv, void* after_dkdv) {
  t_last_error.clear();
  const int n = (before_dq != nullptr) + (before_dkdv != nullptr) + (after_dkdv != nullptr);
  if (n != 0 && n != 3) return fail(FA_ERR_INVALID, "pass all three events or none");
  t_ev_hooks[0] = static_cast<cudaEvent_t>(before_dq);
  t_ev_hooks[1] = static_cast<cudaEvent_t>(before_dkdv);
  t_ev_hooks[2] = static_cast<cudaEvent_t>(after_dkdv);
  return FA_OK;
}

int fa_selftest_bounded_wait(int limit_ms, void* stream) {
  t_last_error.clear();
  if (limit_ms < 1 || limit_ms > 2000) return fail(FA_ERR_INVALID, "limit_ms must be in [1, 2000]");
  DeviceState* st = nullptr;
  int rc = get_device_state(&st);
  if (rc) return rc;
  fa_selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      st->err_word, static_cast<unsigned long long>(limit_ms) * 1000000ull);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(FA_ERR_CUDA, "self-test launch: %s", cudaGetErrorString(e));
  return FA_OK;
}

int fa_check_errors(void* stream) {
  t_last_error.clear();
  DeviceState* st = nullptr;
  int rc = get_device_state(&st);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail(FA_ERR_CUDA, "stream synchronize: %s", cudaGetErrorString(e));
  int word = 0;
  e = cudaMemcpyFromSymbolAsync(&word, g_fa_error_word, sizeof(int), 0, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail(FA_ERR_CUDA, "reading the error word: %s", cudaGetErrorString(e));
  if (word != 0) {
    const int zero = 0;
    cudaMemcpyToSymbolAsync(g_fa_error_word, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
    cudaStreamSynchronize(s);
    return fail(FA_ERR_TIMEOUT, "a kernel's bounded wait expired (device error word %d)", word);
  }
  return FA_OK;
}

}  // extern "C"
