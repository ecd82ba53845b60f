"""fp64 CPU oracle for exact attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package.  The CUDA library never loads, links or calls it, and
it shares no code with the CUDA path.

Contents
  * ``forward`` / ``backward``: ctypes front end of ``oracle.c`` -- the plain
    definition of scaled-dot-product attention and of its gradient, in fp64,
    parallel over rows / KV heads with OpenMP.
  * ``naive``: a numpy materialising implementation (S and P as full N x N
    matrices) used as an independent brute-force check on tiny inputs.
  * ``online``: the pages' tiled online-softmax recurrences (the FA1 form with
    separate alpha/beta factors and the FA2 form that divides once at the end),
    written in numpy fp64, used to check that the recurrence reproduces the
    definition.

  * FP8 (e4m3) inputs (``e4m3_encode`` / ``e4m3_decode``, ``fp8_quantize_qk``,
    ``fp8_quantize_v``, ``fp8_dequantize``, ``forward_fp8``): the definition of the
    FlashAttention-3 low-precision forward's quantized inputs -- random-sign
    Hadamard rotation of Q and K, one scale per 128-row block (Q, K) or per
    channel (V), e4m3 codes -- and the plain attention over their values.
  * ``fp8_baseline``: per-tensor FP8 attention, the baseline of the pages' FP8
    error comparison.

Citations are to the web pages the method is described on:
  "FlashAttention Primer: IO-Aware Attention, from FA1 to FA4" (oripoin.me),
  "Flash Attention" (aiwiki.ai), "FlashAttention" concept page (praveentn.live).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` with gcc + OpenMP (fp64, no fast-math)."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp", "-shared",
           "-fPIC", "-std=c11", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _as_f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor: exact widening of the rounded values
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _as_f32(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor: exact widening of the 16-bit values
        x = x.detach().to("cpu").float().numpy()
    return np.asarray(x, dtype=np.float32)


def _fptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def _u8ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


class Oracle:
    """ctypes front end of one build of ``oracle.c``."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        dp = ctypes.POINTER(ctypes.c_double)
        i = ctypes.c_int
        lib.oracle_forward.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, i, i, ctypes.c_double]
        lib.oracle_forward.restype = i
        lib.oracle_backward.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp,
                                        i, i, i, i, i, i, ctypes.c_double]
        lib.oracle_backward.restype = i
        lib.oracle_forward_rect.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, i, i, ctypes.c_double]
        lib.oracle_forward_rect.restype = i
        lib.oracle_forward_window.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, i, i, ctypes.c_double]
        lib.oracle_forward_window.restype = i
        lib.oracle_backward_window.argtypes = [dp] * 7 + [i] * 6 + [ctypes.c_double]
        lib.oracle_backward_window.restype = i
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = i
        self.lib = lib

        u8p = ctypes.POINTER(ctypes.c_uint8)
        fp = ctypes.POINTER(ctypes.c_float)
        i8p = ctypes.POINTER(ctypes.c_int8)
        lib.oracle_e4m3_encode_array.argtypes = [fp, u8p, ctypes.c_long]
        lib.oracle_e4m3_encode_array.restype = i
        lib.oracle_e4m3_decode_array.argtypes = [u8p, dp, ctypes.c_long]
        lib.oracle_e4m3_decode_array.restype = i
        lib.oracle_fp8_quantize_qk.argtypes = [fp, i8p, i, i, i, u8p, fp]
        lib.oracle_fp8_quantize_qk.restype = i
        lib.oracle_fp8_quantize_v.argtypes = [fp, i, i, i, u8p, fp]
        lib.oracle_fp8_quantize_v.restype = i

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def forward(self, q, k, v, causal: bool, scale: float):
        """O and LSE of softmax(scale q k^T) v, fp64.

        q: [B, Hq, N, d]; k, v: [B, Hkv, N, d].  Returns (o [B,Hq,N,d], lse [B,Hq,N]).
        LSE is the natural-log log-sum-exp of the scaled scores of each row.
        """
        q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
        B, Hq, N, d = q.shape
        Hkv = k.shape[1]
        assert k.shape == (B, Hkv, N, d) and v.shape == k.shape
        o = np.empty_like(q)
        lse = np.empty((B, Hq, N), dtype=np.float64)
        rc = self.lib.oracle_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                     B, Hq, Hkv, N, d, int(bool(causal)), float(scale))
        if rc != 0:
            raise ValueError(f"oracle_forward failed with code {rc}")
        return o, lse

    def forward_rect(self, q, k, v, scale: float):
        """Non-causal forward with Nq query rows and Nk keys: q [B,Hq,Nq,d], k, v [B,Hkv,Nk,d]."""
        q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
        B, Hq, Nq, d = q.shape
        Hkv, Nk = k.shape[1], k.shape[2]
        assert k.shape == (B, Hkv, Nk, d) and v.shape == k.shape
        o = np.empty_like(q)
        lse = np.empty((B, Hq, Nq), dtype=np.float64)
        rc = self.lib.oracle_forward_rect(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                          B, Hq, Hkv, Nq, Nk, d, float(scale))
        if rc != 0:
            raise ValueError(f"oracle_forward_rect failed with code {rc}")
        return o, lse

    def forward_window(self, q, k, v, window: int, scale: float):
        """Sliding-window causal forward: key k visible to query i iff i - window < k <= i."""
        q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
        B, Hq, N, d = q.shape
        Hkv = k.shape[1]
        assert k.shape == (B, Hkv, N, d) and v.shape == k.shape
        o = np.empty_like(q)
        lse = np.empty((B, Hq, N), dtype=np.float64)
        rc = self.lib.oracle_forward_window(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                            B, Hq, Hkv, N, d, int(window), float(scale))
        if rc != 0:
            raise ValueError(f"oracle_forward_window failed with code {rc}")
        return o, lse

    def backward_window(self, q, k, v, dO, window: int, scale: float):
        """Gradients of the sliding-window causal forward.  Returns (dq, dk, dv)."""
        q, k, v, dO = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dO)
        B, Hq, N, d = q.shape
        Hkv = k.shape[1]
        dq, dk, dv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
        rc = self.lib.oracle_backward_window(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(dq),
                                             _ptr(dk), _ptr(dv), B, Hq, Hkv, N, d, int(window),
                                             float(scale))
        if rc != 0:
            raise ValueError(f"oracle_backward_window failed with code {rc}")
        return dq, dk, dv

    # ------------------------------------------------------------ FP8 (e4m3) inputs
    def e4m3_encode(self, x) -> np.ndarray:
        """Nearest e4m3 code of each fp32 value (ties to even, saturating at 448)."""
        x = np.ascontiguousarray(_as_f32(x))
        out = np.empty(x.shape, dtype=np.uint8)
        rc = self.lib.oracle_e4m3_encode_array(_fptr(x), _u8ptr(out), x.size)
        if rc:
            raise ValueError(f"oracle_e4m3_encode_array failed with code {rc}")
        return out

    def e4m3_decode(self, codes) -> np.ndarray:
        codes = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
        out = np.empty(codes.shape, dtype=np.float64)
        rc = self.lib.oracle_e4m3_decode_array(_u8ptr(codes), _ptr(out), codes.size)
        if rc:
            raise ValueError(f"oracle_e4m3_decode_array failed with code {rc}")
        return out

    def fp8_quantize_qk(self, x, signs):
        """Q or K [B, H, N, d] -> (codes uint8 [B, H, N, d], scales float32 [B, H, ceil(N/128)]).
        signs: d values of +1/-1 (the random signs of the rotation), or None for no rotation."""
        x = np.ascontiguousarray(_as_f32(x))
        B, H, N, d = x.shape
        codes = np.empty(x.shape, dtype=np.uint8)
        scales = np.empty((B, H, (N + 127) // 128), dtype=np.float32)
        sg = None if signs is None else np.ascontiguousarray(np.asarray(signs, dtype=np.int8))
        rc = self.lib.oracle_fp8_quantize_qk(_fptr(x), None if sg is None else sg.ctypes.data_as(
            ctypes.POINTER(ctypes.c_int8)), B * H, N, d, _u8ptr(codes), _fptr(scales))
        if rc:
            raise ValueError(f"oracle_fp8_quantize_qk failed with code {rc}")
        return codes, scales

    def fp8_quantize_v(self, v):
        """V [B, H, N, d] -> (codes uint8 [B, H, N, d], scales float32 [B, H, d])."""
        v = np.ascontiguousarray(_as_f32(v))
        B, H, N, d = v.shape
        codes = np.empty(v.shape, dtype=np.uint8)
        scales = np.empty((B, H, d), dtype=np.float32)
        rc = self.lib.oracle_fp8_quantize_v(_fptr(v), B * H, N, d, _u8ptr(codes), _fptr(scales))
        if rc:
            raise ValueError(f"oracle_fp8_quantize_v failed with code {rc}")
        return codes, scales

    def fp8_dequantize(self, q_codes, q_scales, k_codes, k_scales, v_codes, v_scales):
        """fp64 values the codes stand for: code x scale of its block (Q, K) or channel (V)."""
        def rows(codes, scales):
            N = codes.shape[2]
            per_row = np.repeat(np.asarray(scales, dtype=np.float64), 128, axis=2)[:, :, :N]
            return self.e4m3_decode(codes) * per_row[..., None]
        vh = self.e4m3_decode(v_codes) * np.asarray(v_scales, dtype=np.float64)[:, :, None, :]
        return rows(q_codes, q_scales), rows(k_codes, k_scales), vh

    def forward_fp8(self, q_codes, q_scales, k_codes, k_scales, v_codes, v_scales, causal: bool,
                    scale: float):
        """Attention (the plain definition, fp64) over the dequantized FP8 inputs."""
        qh, kh, vh = self.fp8_dequantize(q_codes, q_scales, k_codes, k_scales, v_codes, v_scales)
        return self.forward(qh, kh, vh, causal, scale)

    def backward(self, q, k, v, dO, causal: bool, scale: float):
        """dQ, dK, dV (and D = rowsum(dO * O)) of the definition, fp64.

        Recomputes P and O from (q, k, v) itself.  Returns (dq, dk, dv, D).
        """
        q, k, v, dO = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dO)
        B, Hq, N, d = q.shape
        Hkv = k.shape[1]
        assert dO.shape == q.shape and k.shape == (B, Hkv, N, d) and v.shape == k.shape
        dq = np.empty_like(q)
        dk = np.empty_like(k)
        dv = np.empty_like(v)
        D = np.empty((B, Hq, N), dtype=np.float64)
        rc = self.lib.oracle_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(dq), _ptr(dk),
                                      _ptr(dv), _ptr(D), B, Hq, Hkv, N, d,
                                      int(bool(causal)), float(scale))
        if rc != 0:
            raise ValueError(f"oracle_backward failed with code {rc}")
        return dq, dk, dv, D


def _default() -> Oracle:
    global _lib
    with _lock:
        if _lib is None:
            _lib = Oracle(build())
    return _lib


def num_threads() -> int:
    return _default().num_threads()


def forward(q, k, v, causal: bool, scale: float):
    """See ``Oracle.forward``."""
    return _default().forward(q, k, v, causal, scale)


def backward(q, k, v, dO, causal: bool, scale: float):
    """See ``Oracle.backward``."""
    return _default().backward(q, k, v, dO, causal, scale)


def forward_rect(q, k, v, scale: float):
    """See ``Oracle.forward_rect``."""
    return _default().forward_rect(q, k, v, scale)


def forward_window(q, k, v, window: int, scale: float):
    """See ``Oracle.forward_window``."""
    return _default().forward_window(q, k, v, window, scale)


def backward_window(q, k, v, dO, window: int, scale: float):
    """See ``Oracle.backward_window``."""
    return _default().backward_window(q, k, v, dO, window, scale)


def e4m3_encode(x):
    """See ``Oracle.e4m3_encode``."""
    return _default().e4m3_encode(x)


def e4m3_decode(codes):
    """See ``Oracle.e4m3_decode``."""
    return _default().e4m3_decode(codes)


def fp8_quantize_qk(x, signs):
    """See ``Oracle.fp8_quantize_qk``."""
    return _default().fp8_quantize_qk(x, signs)


def fp8_quantize_v(v):
    """See ``Oracle.fp8_quantize_v``."""
    return _default().fp8_quantize_v(v)


def fp8_dequantize(q_codes, q_scales, k_codes, k_scales, v_codes, v_scales):
    """See ``Oracle.fp8_dequantize``."""
    return _default().fp8_dequantize(q_codes, q_scales, k_codes, k_scales, v_codes, v_scales)


def forward_fp8(q_codes, q_scales, k_codes, k_scales, v_codes, v_scales, causal: bool, scale: float):
    """See ``Oracle.forward_fp8``."""
    return _default().forward_fp8(q_codes, q_scales, k_codes, k_scales, v_codes, v_scales, causal,
                                  scale)
