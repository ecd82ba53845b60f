/*
 * fa.h -- C ABI of libfa.so: exact IO-aware scaled-dot-product attention on
 * NVIDIA GB300 (sm_103a).
 *
 * The operation ("FlashAttention Primer: IO-Aware Attention, from FA1 to FA4",
 * section "Why attention is quadratic", the SDPA equation; "Flash Attention"
 * (aiwiki.ai), section "Definition and scope"):
 *
 *     S = scale * Q K^T,   P = rowsoftmax(S),   O = P V
 *
 * computed exactly (up to floating-point rounding order) by a tiled schedule
 * that never writes S or P to device memory: the forward keeps a running row
 * maximum and sum (online softmax, "FlashAttention Primer", section
 * "FlashAttention-1"; "Flash Attention", section "Online softmax") and saves
 * only O and the per-row log-sum-exp; the backward recomputes P block by block
 * from that log-sum-exp ("FlashAttention Primer", section "Backward pass:
 * recomputation instead of storage").
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *   never frees or keeps them beyond the call's stream work.
 * - Layouts are dense row-major:
 *     q, o, dO, dq : [B, Hq,  N, d]   (element type `dtype`)
 *     k, v, dk, dv : [B, Hkv, N, d]   (element type `dtype`)
 *     lse          : [B, Hq,  N]      (float32)
 *   Every base pointer must be 16-byte aligned (the tiles are moved by the
 *   Tensor Memory Accelerator, whose global addresses must be 16-byte aligned).
 * - d must be 64 or 128.  N >= 1 (any value; ragged tails are masked).
 *   Hq % Hkv == 0; query head h reads key/value head floor(h * Hkv / Hq)
 *   (contiguous groups of Hq/Hkv query heads share one KV head).
 * - causal != 0 masks key k for query i when k > i (square attention only).
 * - scale multiplies Q K^T; pass 1/sqrt(d) for standard attention.  Any finite
 *   value is accepted.
 * - dtype: FA_DTYPE_FP16 or FA_DTYPE_BF16 (both operands and outputs).
 * - stream: a cudaStream_t passed as void* (NULL = legacy default stream).
 *   Every call only enqueues work on that stream and returns; it never
 *   synchronises.  Calls on different streams may run concurrently.
 * - Return value: FA_OK, or one of the FA_ERR_* codes below.  On any error
 *   nothing has been enqueued and a message is available from fa_last_error()
 *   on the same host thread.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Exported symbols keep default visibility even when the library is built with
   -fvisibility=hidden. */
#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

#define FA_OK 0
#define FA_ERR_INVALID 1     /* null pointer, non-positive size, Hq % Hkv != 0, non-finite scale,
                                workspace too small */
#define FA_ERR_UNSUPPORTED 2 /* d not in {64,128}, unknown dtype, misaligned pointer, size over
                                the limits, device is not sm_103 */
#define FA_ERR_CUDA 3        /* a CUDA runtime/driver call or a launch failed */
#define FA_ERR_TIMEOUT 4     /* a kernel's bounded wait expired (reported by fa_check_errors) */

#define FA_DTYPE_FP16 0
#define FA_DTYPE_BF16 1

/*
 * Forward pass: O = softmax(scale * Q K^T) V and LSE.
 *
 * lse[b,h,i] = ln( sum_k exp(scale * q_i . k_k) ) over the visible keys k,
 * the natural-log log-sum-exp of the scaled scores of row i ("FlashAttention
 * Primer", section "Backward pass: recomputation instead of storage": the
 * forward stores O and the per-row log-sum-exp, not the N x N matrix).
 *
 * Reads q, k, v; writes o and lse (every element with i < N).  Allocates
 * nothing on the device.  Deterministic: the same inputs give bitwise the
 * same outputs.
 */
FA_API int fa_forward(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
               int Hkv, int N, int d, int causal, float scale, int dtype, void* stream);

/*
 * Sliding-window (local) causal forward: like fa_forward with causal = 1, but
 * query i attends only to the `window` most recent keys, i - window < k <= i
 * ("Flash Attention" (aiwiki.ai), section "Features": local sliding windows;
 * section "Block-sparse FlashAttention": blocks the mask leaves empty are
 * skipped, so the work grows with the retained blocks, about N * window,
 * instead of N^2 / 2).
 *
 * window >= 1 (FA_ERR_INVALID otherwise); window >= N gives exactly the causal
 * result.  Key tiles outside every row's window are neither loaded nor
 * computed; tiles the window's edge crosses are masked element-wise.  Outputs,
 * layouts, errors, determinism and asynchrony as fa_forward.
 */
FA_API int fa_forward_window(const void* q, const void* k, const void* v, void* o, float* lse,
                             int B, int Hq, int Hkv, int N, int d, int window, float scale,
                             int dtype, void* stream);

/*
 * FP8 (e4m3) forward ("FlashAttention Primer", section "FlashAttention-3: Hopper
 * asynchrony and FP8": block quantization, and an incoherent rotation applied
 * before quantization that lowers the FP8 error; "Flash Attention" (aiwiki.ai),
 * section "FlashAttention-3": the rotation is random signs and a Hadamard
 * transform, applied to queries and keys alike so that their dot products are
 * kept).  d = 128 only.
 *
 * fa_quantize_fp8: q, k, v (16-bit, [B,H,N,d] as fa_forward, element type
 * dtype) -> e4m3 codes and fp32 dequantization scales:
 *   q8 [B,Hq,N,d], k8 [B,Hkv,N,d]: row y = (x * s) H_d (s = signs, +1/-1 per
 *     channel, d bytes in device memory; H_d the Sylvester Hadamard matrix, entries
 *     +-1), then per 128-row block of a head: amax = max |y|, code =
 *     e4m3(y * 448/amax) (round to nearest even, saturating);
 *   q_scale [B,Hq,ceil(N/128)], k_scale [B,Hkv,ceil(N/128)]: amax / (448 sqrt(d)),
 *     so that code * scale is the orthogonally rotated input (x * s) H_d / sqrt(d);
 *   v8t [B,Hkv,d,Np], Np = fa_fp8_vt_stride(N): V transposed (channel-major),
 *     code = e4m3(v * 448/amax_c) with one amax per (head, channel) over all N
 *     rows, keys N..Np-1 zero; v_scale [B,Hkv,d] = amax_c / 448.
 * signs may be NULL: no rotation, and q_scale, k_scale = amax / 448.  Every fp32
 * step that decides a code is exactly rounded in a fixed order, so the codes are
 * reproducible bit for bit.
 *
 * fa_forward_fp8: attention over the dequantized inputs -- O = softmax(scale *
 * Qh Kh^T) Vh with Qh = code * q_scale per block etc. -- on e4m3 tensor cores,
 * the probabilities rounded to e4m3 for the P V product; O is written in
 * bfloat16 [B,Hq,N,d], lse (fp32 [B,Hq,N]) as in fa_forward.  The rotation
 * leaves Q K^T unchanged, so `scale` is the usual one (1/sqrt(d)).
 *
 * Both allocate nothing, run asynchronously on `stream`, and return the
 * fa_forward error codes (FA_ERR_UNSUPPORTED for d != 128).
 */
FA_API int fa_fp8_vt_stride(int N);  /* Np for N >= 1 (0 if N < 1 or Np would overflow an int) */
FA_API int fa_quantize_fp8(const void* q, const void* k, const void* v, const signed char* signs,
                           void* q8, void* k8, void* v8t, float* q_scale, float* k_scale,
                           float* v_scale, int B, int Hq, int Hkv, int N, int d, int dtype,
                           void* stream);
FA_API int fa_forward_fp8(const void* q8, const void* k8, const void* v8t, const float* q_scale,
                          const float* k_scale, const float* v_scale, void* o, float* lse, int B,
                          int Hq, int Hkv, int N, int d, int causal, float scale, void* stream);

/*
 * Split-KV forward for decoding: a few query rows against a long key sequence
 * ("Flash Attention" (aiwiki.ai), section "Flash-Decoding": split the keys
 * into chunks, attend to each chunk with its own log-sum-exp, combine).
 *
 *   q, o : [B, Hq, Nq, d]    k, v : [B, Hkv, Nk, d]    lse : [B, Hq, Nq] fp32
 *
 * Non-causal: every query row attends to all Nk keys (a decoding step's new
 * tokens against the full cache).  O and LSE have the same meaning as in
 * fa_forward.  The query rows of the Hq/Hkv heads that share a KV head are
 * processed together, so each key/value tile is read once per KV head.
 *
 * num_splits: number of key chunks; <= 0 chooses one from the problem size and
 * the device's SM count; it is clamped to the number of 128-key tiles.  With
 * more than one split the partial results go through `workspace` (device
 * memory, 256-byte aligned, at least fa_forward_splitkv_workspace_size() bytes
 * for the same arguments; may be NULL when that size is 0).  Nq, Nk >= 1.
 * Same conventions, errors and asynchrony as fa_forward otherwise.
 */
FA_API size_t fa_forward_splitkv_workspace_size(int B, int Hq, int Hkv, int Nq, int Nk, int d,
                                                int num_splits);
FA_API int fa_forward_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                              int B, int Hq, int Hkv, int Nq, int Nk, int d, float scale, int dtype,
                              int num_splits, void* workspace, size_t ws_bytes, void* stream);

/*
 * Bytes of device workspace fa_backward needs for these sizes: round_up(4 *
 * B*Hq*N, 256).  Returns 0 if the sizes are invalid.  Layout: D float32
 * [B, Hq, N] at offset 0, D_i = sum_c dO_ic * O_ic.
 */
FA_API size_t fa_backward_workspace_size(int B, int Hq, int N, int d);

/*
 * Backward pass from the saved statistics: given q, k, v, the forward's o and
 * lse, and dO = dL/dO, writes dq, dk, dv (element type dtype).
 *
 * Steps, all on `stream`:
 *   1. per query tile, D_i = rowsum(dO_i * O_i) (written to the workspace),
 *      then recompute S and P = exp(scale * Q K^T - LSE) block by block and
 *      accumulate dQ += scale * dS K over all key tiles inside one CTA, with
 *      dS = P * (dO V^T - D);
 *   2. per key/value tile, recompute S^T and P^T the same way and accumulate
 *      dV += P^T dO and dK += scale * dS^T Q over all query tiles (and, for
 *      grouped query attention, over the KV head's query heads) inside one
 *      CTA, reading D from the workspace.
 * The gradient is that of the definition: the primer's printed dS omits the
 * -D term and the scale factor, which this library applies (the oracle's
 * finite-difference checks fix the formula).  No atomic adds are used: every
 * sum runs in a fixed order, so dq, dk and dv are bitwise reproducible.
 *
 * workspace: device memory of at least fa_backward_workspace_size() bytes,
 * 256-byte aligned, owned by the caller, not used concurrently by another
 * call.
 */
FA_API int fa_backward(const void* q, const void* k, const void* v, const void* o, const float* lse,
                const void* dO, void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes,
                int B, int Hq, int Hkv, int N, int d, int causal, float scale, int dtype,
                void* stream);

/*
 * Backward pass of fa_forward_window: the gradients of the sliding-window
 * causal attention (i - window < k <= i) from the saved O and LSE.  Same
 * arguments, workspace, outputs, errors and asynchrony as fa_backward, with
 * `window` (>= 1) in place of `causal`; window >= N equals the causal
 * backward.  Only the key/query tile pairs some window reaches are computed.
 */
FA_API int fa_backward_window(const void* q, const void* k, const void* v, const void* o,
                              const float* lse, const void* dO, void* dq, void* dk, void* dv,
                              void* workspace, size_t ws_bytes, int B, int Hq, int Hkv, int N,
                              int d, int window, float scale, int dtype, void* stream);

/*
 * Bytes of device workspace fa_backward_atomic needs: round_up(4 * B*Hq*N, 256)
 * + round_up(4 * B*Hq*N*d, 256).  Returns 0 if the sizes are invalid.  Layout:
 * D float32 [B, Hq, N] at offset 0, then the float32 dQ accumulator
 * [B, Hq, N, d].
 */
FA_API size_t fa_backward_atomic_workspace_size(int B, int Hq, int N, int d);

/*
 * Backward pass in one sweep over the key tiles, with dQ accumulated across
 * thread blocks by atomic adds: the primer's default backward ("FlashAttention
 * Primer: IO-Aware Attention, from FA1 to FA4", section "Backward pass:
 * recomputation instead of storage", which notes that it is bitwise
 * nondeterministic and that the deterministic form is slower).
 *
 * Same inputs and outputs as fa_backward; `causal` as there and `window` as in
 * fa_backward_window (0: none; >= 1 needs causal = 1; window >= N is causal).
 * Steps, all on `stream`:
 *   1. D_i = rowsum(dO_i * O_i) into the workspace, and the workspace's dQ
 *      accumulator set to zero;
 *   2. per key/value tile j: recompute S^T, P^T and dS^T against every query
 *      tile i that sees it (and every query head of the KV head), accumulate
 *      dV += P^T dO and dK += scale * dS^T Q in one CTA, and add the partial
 *      dQ_i += dS K_j into the accumulator with float32 atomic adds;
 *   3. dq = scale * accumulator, rounded to dtype.
 * Five N x N x d products per tile pair instead of fa_backward's seven.  dk
 * and dv are summed in a fixed order (bitwise reproducible); dq is the same
 * sum in an order that varies between runs, so its last bits may differ from
 * run to run and from fa_backward's.
 *
 * workspace: at least fa_backward_atomic_workspace_size() bytes of device
 * memory, 256-byte aligned, owned by the caller, not used concurrently by
 * another call.  Errors as fa_backward, plus FA_ERR_INVALID for window < 0 or
 * window > 0 with causal = 0.  The event hooks of
 * fa_set_backward_event_hooks bracket step 1 (before_dq .. before_dkdv) and
 * step 2 (before_dkdv .. after_dkdv).
 */
FA_API int fa_backward_atomic(const void* q, const void* k, const void* v, const void* o,
                              const float* lse, const void* dO, void* dq, void* dk, void* dv,
                              void* workspace, size_t ws_bytes, int B, int Hq, int Hkv, int N,
                              int d, int causal, int window, float scale, int dtype, void* stream);

/*
 * Backward pass that allocates nothing.  (Library-side addition: the attention
 * method has no counterpart of it.)
 *
 * Same arguments, outputs, errors and asynchrony as fa_backward, minus the
 * workspace: the scratch fa_backward needs (the D vector,
 * fa_backward_workspace_size() bytes) is taken from one
 * FA_NOALLOC_SCRATCH_BYTES-byte array compiled into the library's device code.
 * The array is placed in device memory on the first call on each device (the
 * runtime loads the library's device code lazily) and stays there until the
 * process exits.  It is
 * for callers that may not call cudaMalloc or any other allocator: a host
 * program that reserves all device memory up front and forbids allocation
 * afterwards, a plugin running inside a framework that gives it no allocator,
 * or a latency-critical loop that cannot afford an allocation's implicit
 * device synchronisation.  The caller still provides every input and output.
 *
 * - Sizes whose fa_backward_workspace_size() exceeds FA_NOALLOC_SCRATCH_BYTES
 *   are rejected with FA_ERR_UNSUPPORTED (nothing is enqueued); use
 *   fa_backward with a workspace for those.
 * - The first call on each device places the array and looks up its device
 *   address, with that device current.  Make that first call before the
 *   caller reserves the rest of the device's memory and before any stream
 *   capture.  If it fails (FA_ERR_CUDA, e.g. no memory left to place the
 *   array) nothing is enqueued and a later call tries again.
 * - Every call on a device shares the one array and leaves its contents
 *   behind; each call overwrites every element it later reads, so nothing
 *   has to start at zero.  Calls whose GPU work overlaps (different streams, or
 *   different host threads, without ordering between them) race on the array
 *   and give wrong gradients: serialise them.
 * - Calls no cudaMalloc, cudaFree or other allocating routine.
 */
#define FA_NOALLOC_SCRATCH_BYTES (40 * 1024 * 1024)
FA_API int fa_backward_noalloc(const void* q, const void* k, const void* v, const void* o,
                               const float* lse, const void* dO, void* dq, void* dk, void* dv,
                               int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                               int dtype, void* stream);

/*
 * Profiling hook for the backward's two kernels.  After this call, every
 * fa_backward issued from the calling host thread records, on its stream,
 * `before_dq` immediately before launching the dQ kernel (which runs first),
 * `before_dkdv` between it and the dK/dV kernel, and `after_dkdv` immediately
 * after the dK/dV kernel; cudaEventElapsedTime between consecutive events is
 * each kernel's device time.  All are cudaEvent_t handles passed as void*, created and
 * owned by the caller; pass three NULLs to stop.  Thread-local; never
 * synchronises.  Returns FA_OK, or FA_ERR_INVALID if only some are NULL.
 */
FA_API int fa_set_backward_event_hooks(void* before_dq, void* before_dkdv, void* after_dkdv);

/*
 * Synchronises `stream`, then reads and clears the device error word that the
 * kernels set when a bounded wait expires.  Returns FA_OK, FA_ERR_TIMEOUT, or
 * FA_ERR_CUDA if the synchronisation itself failed.
 */
FA_API int fa_check_errors(void* stream);

/*
 * Self-test of the failure detection.  Enqueues on `stream` a one-thread
 * kernel that waits on an mbarrier nothing ever completes, using the same
 * bounded wait as the attention kernels but with a limit of `limit_ms`
 * milliseconds (1..2000).  When the limit expires the kernel raises the device
 * error word and returns normally, so a following fa_check_errors(stream)
 * reports FA_ERR_TIMEOUT (and clears the word) while the CUDA context stays
 * usable.  Returns FA_OK once enqueued, FA_ERR_INVALID for a bad limit.
 */
FA_API int fa_selftest_bounded_wait(int limit_ms, void* stream);

/* Message for the last error returned on the calling host thread ("" if none). */
FA_API const char* fa_last_error(void);

/* Library version string. */
FA_API const char* fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
