"""ctypes binding of libfa.so: argument marshalling only.

Every step of the attention path runs in the library's CUDA kernels; this
module checks tensors, allocates outputs with torch, and passes raw device
pointers and the current CUDA stream through the C ABI declared in
``include/fa.h``.  If the library is missing it raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libfa.so")

FA_OK, FA_ERR_INVALID, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT = 0, 1, 2, 3, 4
FA_DTYPE_FP16, FA_DTYPE_BF16 = 0, 1
_CODES = {FA_ERR_INVALID: "FA_ERR_INVALID", FA_ERR_UNSUPPORTED: "FA_ERR_UNSUPPORTED",
          FA_ERR_CUDA: "FA_ERR_CUDA", FA_ERR_TIMEOUT: "FA_ERR_TIMEOUT"}

_lock = threading.Lock()
_lib = None


class FAError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{_CODES.get(code, code)}: {msg}")
        self.code = code


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libfa.so (built by ``exact_io_aware_flash_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} not found: the CUDA library is required (build it with "
                "`python -m exact_io_aware_flash_gb300.build`); there is no CPU fallback")
        lib = ctypes.CDLL(path)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.fa_forward.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp]
        lib.fa_forward.restype = i
        lib.fa_forward_window.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp]
        lib.fa_forward_window.restype = i
        lib.fa_backward_workspace_size.argtypes = [i, i, i, i]
        lib.fa_backward_workspace_size.restype = sz
        lib.fa_backward.argtypes = [vp] * 10 + [sz] + [i] * 6 + [f, i, vp]
        lib.fa_backward.restype = i
        lib.fa_backward_window.argtypes = [vp] * 10 + [sz] + [i] * 6 + [f, i, vp]
        lib.fa_backward_window.restype = i
        lib.fa_backward_atomic_workspace_size.argtypes = [i, i, i, i]
        lib.fa_backward_atomic_workspace_size.restype = sz
        lib.fa_backward_atomic.argtypes = [vp] * 10 + [sz] + [i] * 7 + [f, i, vp]
        lib.fa_backward_atomic.restype = i
        lib.fa_fp8_vt_stride.argtypes = [i]
        lib.fa_fp8_vt_stride.restype = i
        lib.fa_quantize_fp8.argtypes = [vp] * 10 + [i] * 6 + [vp]
        lib.fa_quantize_fp8.restype = i
        lib.fa_forward_fp8.argtypes = [vp] * 8 + [i] * 6 + [f, vp]
        lib.fa_forward_fp8.restype = i
        lib.fa_forward_splitkv_workspace_size.argtypes = [i] * 7
        lib.fa_forward_splitkv_workspace_size.restype = sz
        lib.fa_forward_splitkv.argtypes = [vp] * 5 + [i] * 6 + [f, i, i, vp, sz, vp]
        lib.fa_forward_splitkv.restype = i
        lib.fa_backward_noalloc.argtypes = [vp] * 9 + [i] * 6 + [f, i, vp]
        lib.fa_backward_noalloc.restype = i
        lib.fa_set_backward_event_hooks.argtypes = [vp, vp, vp]
        lib.fa_set_backward_event_hooks.restype = i
        lib.fa_selftest_bounded_wait.argtypes = [i, vp]
        lib.fa_selftest_bounded_wait.restype = i
        lib.fa_check_errors.argtypes = [vp]
        lib.fa_check_errors.restype = i
        lib.fa_last_error.argtypes = []
        lib.fa_last_error.restype = ctypes.c_char_p
        lib.fa_version.argtypes = []
        lib.fa_version.restype = ctypes.c_char_p
        _lib = lib
        return lib


def _raise(code: int):
    if code != FA_OK:
        raise FAError(code, load().fa_last_error().decode())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return FA_DTYPE_FP16
    if t.dtype == torch.bfloat16:
        return FA_DTYPE_BF16
    raise TypeError(f"unsupported dtype {t.dtype}: use float16 or bfloat16")


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _check(t: torch.Tensor, name: str, shape, dtype):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous [B, H, N, d]")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")


def version() -> str:
    return load().fa_version().decode()


def workspace_size(B: int, Hq: int, N: int, d: int, deterministic: bool = True) -> int:
    """Bytes of backward workspace (fa_backward, or fa_backward_atomic when not deterministic)."""
    lib = load()
    if deterministic:
        return int(lib.fa_backward_workspace_size(B, Hq, N, d))
    return int(lib.fa_backward_atomic_workspace_size(B, Hq, N, d))


def _window_arg(window, causal) -> int:
    window = int(window)
    if not causal:
        raise ValueError("a sliding window is causal: pass causal=True with window")
    if window < 1:
        raise ValueError(f"window must be at least 1, got {window}")
    return window


def forward(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
            stream=None, window: int | None = None):
    """O = softmax(scale q k^T) v and the natural-log LSE per row, on the GPU.

    q: [B, Hq, N, d]; k, v: [B, Hkv, N, d]; fp16 or bf16, contiguous, CUDA.
    window: with causal=True, a sliding window of that many keys (query i sees
    keys i - window < k <= i), through fa_forward_window.
    Returns (o [B,Hq,N,d] in q's dtype, lse [B,Hq,N] float32).
    """
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    _check(q, "q", (B, Hq, N, d), q.dtype)
    _check(k, "k", (B, Hkv, N, d), q.dtype)
    _check(v, "v", (B, Hkv, N, d), q.dtype)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device)
    _check(out, "out", (B, Hq, N, d), q.dtype)
    _check(lse, "lse", (B, Hq, N), torch.float32)
    if window is not None:
        rc = load().fa_forward_window(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                      lse.data_ptr(), B, Hq, Hkv, N, d, _window_arg(window, causal),
                                      float(scale), _dtype_code(q), _stream_handle(stream))
    else:
        rc = load().fa_forward(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                               lse.data_ptr(), B, Hq, Hkv, N, d, int(bool(causal)), float(scale),
                               _dtype_code(q), _stream_handle(stream))
    _raise(rc)
    return out, lse


def quantize_fp8(q, k, v, signs=None, stream=None) -> dict:
    """e4m3 codes and scales of q, k, v (16-bit, d = 128) for forward_fp8 (see fa.h).

    signs: int8 CUDA tensor of d values +1/-1 (the random signs of the Hadamard
    rotation of q and k), or None for no rotation.  Returns a dict with q8, k8
    (uint8 [B,H,N,d]), v8t (uint8 [B,Hkv,d,Np], V transposed), q_scale, k_scale
    (float32 [B,H,ceil(N/128)]) and v_scale (float32 [B,Hkv,d]).
    """
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    _check(q, "q", (B, Hq, N, d), q.dtype)
    _check(k, "k", (B, Hkv, N, d), q.dtype)
    _check(v, "v", (B, Hkv, N, d), q.dtype)
    if signs is not None:
        _check(signs, "signs", (d,), torch.int8)
    lib = load()
    Np = int(lib.fa_fp8_vt_stride(N))
    T = (N + 127) // 128
    dev = q.device
    out = dict(q8=torch.empty((B, Hq, N, d), dtype=torch.uint8, device=dev),
               k8=torch.empty((B, Hkv, N, d), dtype=torch.uint8, device=dev),
               v8t=torch.empty((B, Hkv, d, Np), dtype=torch.uint8, device=dev),
               q_scale=torch.empty((B, Hq, T), dtype=torch.float32, device=dev),
               k_scale=torch.empty((B, Hkv, T), dtype=torch.float32, device=dev),
               v_scale=torch.empty((B, Hkv, d), dtype=torch.float32, device=dev))
    rc = lib.fa_quantize_fp8(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                             None if signs is None else signs.data_ptr(),
                             *(out[n].data_ptr() for n in ("q8", "k8", "v8t", "q_scale", "k_scale",
                                                           "v_scale")),
                             B, Hq, Hkv, N, d, _dtype_code(q), _stream_handle(stream))
    _raise(rc)
    return out


def forward_fp8(fp8: dict, causal: bool = False, scale: float | None = None, out=None, lse=None,
                stream=None):
    """Attention over e4m3 inputs from quantize_fp8 (see fa.h); O in bfloat16.

    Returns (o [B,Hq,N,d] bfloat16, lse [B,Hq,N] float32).
    """
    q8, k8, v8t = fp8["q8"], fp8["k8"], fp8["v8t"]
    B, Hq, N, d = q8.shape
    Hkv = k8.shape[1]
    Np = int(load().fa_fp8_vt_stride(N))
    T = (N + 127) // 128
    _check(q8, "q8", (B, Hq, N, d), torch.uint8)
    _check(k8, "k8", (B, Hkv, N, d), torch.uint8)
    _check(v8t, "v8t", (B, Hkv, d, Np), torch.uint8)
    _check(fp8["q_scale"], "q_scale", (B, Hq, T), torch.float32)
    _check(fp8["k_scale"], "k_scale", (B, Hkv, T), torch.float32)
    _check(fp8["v_scale"], "v_scale", (B, Hkv, d), torch.float32)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = torch.empty((B, Hq, N, d), dtype=torch.bfloat16, device=q8.device) if out is None else out
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q8.device) if lse is None else lse
    _check(out, "out", (B, Hq, N, d), torch.bfloat16)
    _check(lse, "lse", (B, Hq, N), torch.float32)
    rc = load().fa_forward_fp8(q8.data_ptr(), k8.data_ptr(), v8t.data_ptr(),
                               fp8["q_scale"].data_ptr(), fp8["k_scale"].data_ptr(),
                               fp8["v_scale"].data_ptr(), out.data_ptr(), lse.data_ptr(), B, Hq, Hkv,
                               N, d, int(bool(causal)), float(scale), _stream_handle(stream))
    _raise(rc)
    return out, lse


def forward_splitkv(q, k, v, scale: float | None = None, num_splits: int = 0, out=None, lse=None,
                    workspace=None, stream=None):
    """Split-KV (decoding) forward: q [B, Hq, Nq, d] against k, v [B, Hkv, Nk, d], non-causal.

    Returns (o [B,Hq,Nq,d], lse [B,Hq,Nq] float32).  num_splits <= 0 lets the
    library choose the number of key chunks.
    """
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    _check(q, "q", (B, Hq, Nq, d), q.dtype)
    _check(k, "k", (B, Hkv, Nk, d), q.dtype)
    _check(v, "v", (B, Hkv, Nk, d), q.dtype)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device) if lse is None else lse
    _check(out, "out", (B, Hq, Nq, d), q.dtype)
    _check(lse, "lse", (B, Hq, Nq), torch.float32)
    lib = load()
    ws_bytes = int(lib.fa_forward_splitkv_workspace_size(B, Hq, Hkv, Nq, Nk, d, int(num_splits)))
    if workspace is None and ws_bytes:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_len = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = lib.fa_forward_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                lse.data_ptr(), B, Hq, Hkv, Nq, Nk, d, float(scale), _dtype_code(q),
                                int(num_splits), ws_ptr, ws_len, _stream_handle(stream))
    _raise(rc)
    return out, lse


def backward(q, k, v, o, lse, dO, causal: bool = False, scale: float | None = None, dq=None,
             dk=None, dv=None, workspace=None, stream=None, window: int | None = None,
             deterministic: bool = True):
    """dq, dk, dv of O = softmax(scale q k^T) v given the forward's o, lse and dO = dL/dO.

    window: the forward's sliding window (with causal=True).
    deterministic: True runs fa_backward / fa_backward_window (two passes, every
    sum in a fixed order); False runs fa_backward_atomic (one pass, dq summed
    with atomic adds, so its last bits vary between runs).
    """
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    for t, name, H in ((q, "q", Hq), (k, "k", Hkv), (v, "v", Hkv), (o, "o", Hq), (dO, "dO", Hq)):
        _check(t, name, (B, H, N, d), q.dtype)
    _check(lse, "lse", (B, Hq, N), torch.float32)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check(dq, "dq", (B, Hq, N, d), q.dtype)
    _check(dk, "dk", (B, Hkv, N, d), q.dtype)
    _check(dv, "dv", (B, Hkv, N, d), q.dtype)
    ws_bytes = workspace_size(B, Hq, N, d, deterministic)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    if workspace.numel() * workspace.element_size() < ws_bytes:
        raise ValueError(f"workspace must hold at least {ws_bytes} bytes")
    lib = load()
    ptrs = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dO.data_ptr(),
            dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), workspace.data_ptr(),
            workspace.numel() * workspace.element_size())
    if not deterministic:
        w = 0 if window is None else _window_arg(window, causal)
        rc = lib.fa_backward_atomic(*ptrs, B, Hq, Hkv, N, d, int(bool(causal)), w, float(scale),
                                    _dtype_code(q), _stream_handle(stream))
    elif window is not None:
        rc = lib.fa_backward_window(*ptrs, B, Hq, Hkv, N, d, _window_arg(window, causal),
                                    float(scale), _dtype_code(q), _stream_handle(stream))
    else:
        rc = lib.fa_backward(*ptrs, B, Hq, Hkv, N, d, int(bool(causal)), float(scale),
                             _dtype_code(q), _stream_handle(stream))
    _raise(rc)
    return dq, dk, dv


def set_backward_event_hooks(before_dq=None, before_dkdv=None, after_dkdv=None) -> None:
    """Record CUDA events around the backward's dQ and dK/dV kernels (see fa.h).

    The arguments are torch.cuda.Event objects that have been recorded at
    least once (so their CUDA handles exist); three Nones stop the hook.
    """
    evs = (before_dq, before_dkdv, after_dkdv)
    _raise(load().fa_set_backward_event_hooks(*(None if e is None else e.cuda_event for e in evs)))


def selftest_bounded_wait(limit_ms: int = 50, stream=None) -> None:
    """Enqueue a kernel whose bounded wait runs out (see fa.h); check_errors() then raises."""
    _raise(load().fa_selftest_bounded_wait(int(limit_ms), _stream_handle(stream)))


def check_errors(stream=None) -> None:
    """Synchronise the stream and raise FAError if a kernel's bounded wait expired."""
    _raise(load().fa_check_errors(_stream_handle(stream)))
