"""MXFP4 oracle -- TEST INFRASTRUCTURE ONLY.

A plain, slow fp64 CPU statement of the MXFP4 linear layer (``mxfp4_oracle.c``),
loaded through ctypes.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import it; the product library
(``block_scaled_mxfp4_activation_gb300``) never does, and the two share no code.

What each function computes, and which page it follows, is stated in the C file.
Every array crosses the boundary as a contiguous numpy array: bf16 values as
their uint16 bit patterns, codes and scales as uint8.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mxfp4_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
# Tests that plant a mistake in a copy of the oracle point this variable at
# the copy's compiled library; nothing else sets it.
_VARIANT = os.environ.get("MXFP4_ORACLE_VARIANT_LIB")
_lock = threading.Lock()
_lib = None

# Plain ISO C, no fast-math and no FMA contraction: the oracle's arithmetic is
# exactly what the source says.
_CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def compile_source(src: str, out: str) -> str:
    """Compile an oracle source file into a shared library with the oracle's flags."""
    subprocess.run(["gcc", *_CFLAGS, src, "-o", out, "-lm"], check=True)
    return out


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/_build/liboracle.so`` (gcc)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *_CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(_VARIANT if _VARIANT else build())
            P = ctypes.c_void_p
            I = ctypes.c_int64
            lib.oracle_e2m1_decode.argtypes = [ctypes.c_uint8]
            lib.oracle_e2m1_decode.restype = ctypes.c_double
            lib.oracle_e8m0_decode.argtypes = [ctypes.c_uint8]
            lib.oracle_e8m0_decode.restype = ctypes.c_double
            lib.oracle_e2m1_encode.argtypes = [ctypes.c_double]
            lib.oracle_e2m1_encode.restype = ctypes.c_uint8
            lib.oracle_scale_byte.argtypes = [ctypes.c_float]
            lib.oracle_scale_byte.restype = ctypes.c_uint8
            lib.oracle_bf16_from_f64.argtypes = [ctypes.c_double]
            lib.oracle_bf16_from_f64.restype = ctypes.c_uint16
            lib.oracle_quantize.argtypes = [P, I, I, I, P, P]
            lib.oracle_dequantize.argtypes = [P, P, I, I, P]
            lib.oracle_gemm.argtypes = [P, P, P, P, I, I, I, P, P]
            lib.oracle_gemm_sampled.argtypes = [P, P, P, P, I, P, P, I, P, P]
            lib.oracle_quant_gemm.argtypes = [P, I, P, P, I, I, I, P, P, P, P]
            lib.oracle_e2m1_encode_array.argtypes = [P, I, P]
            lib.oracle_scale_byte_array.argtypes = [P, I, P]
            lib.oracle_bf16_from_f64_array.argtypes = [P, I, P]
            for fn in ("oracle_quantize", "oracle_dequantize", "oracle_gemm", "oracle_gemm_sampled",
                       "oracle_quant_gemm", "oracle_e2m1_encode_array", "oracle_scale_byte_array",
                       "oracle_bf16_from_f64_array"):
                getattr(lib, fn).restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(x) -> np.ndarray:
    """bf16 bit patterns as a contiguous uint16 array (accepts a torch bf16 tensor)."""
    if hasattr(x, "view") and hasattr(x, "dtype") and str(getattr(x, "dtype", "")) == "torch.bfloat16":
        import torch

        x = x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    return np.ascontiguousarray(x, dtype=np.uint16)


# ----------------------------------------------------------------------------- scalar rules
def e2m1_decode(code: int) -> float:
    return _load().oracle_e2m1_decode(code)


def e8m0_decode(byte: int) -> float:
    return _load().oracle_e8m0_decode(byte)


def e2m1_encode(q: float) -> int:
    return int(_load().oracle_e2m1_encode(q))


def scale_byte(amax: float) -> int:
    return int(_load().oracle_scale_byte(amax))


def bf16_from_f64(d: float) -> int:
    return int(_load().oracle_bf16_from_f64(d))


def e2m1_encode_array(q: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.float64)
    out = np.empty(q.shape, np.uint8)
    _load().oracle_e2m1_encode_array(_ptr(q), q.size, _ptr(out))
    return out


def scale_byte_array(amax: np.ndarray) -> np.ndarray:
    amax = np.ascontiguousarray(amax, dtype=np.float32)
    out = np.empty(amax.shape, np.uint8)
    _load().oracle_scale_byte_array(_ptr(amax), amax.size, _ptr(out))
    return out


def bf16_from_f64_array(d: np.ndarray) -> np.ndarray:
    d = np.ascontiguousarray(d, dtype=np.float64)
    out = np.empty(d.shape, np.uint16)
    _load().oracle_bf16_from_f64_array(_ptr(d), d.size, _ptr(out))
    return out


# ----------------------------------------------------------------------------- matrix functions
def quantize(x) -> tuple[np.ndarray, np.ndarray]:
    """bf16 [rows, cols] -> (codes uint8 [rows, cols/2], scales uint8 [rows, cols/32])."""
    x = _u16(x)
    rows, cols = x.shape
    assert cols % 32 == 0, "cols must be a multiple of 32"
    q = np.empty((rows, cols // 2), np.uint8)
    s = np.empty((rows, cols // 32), np.uint8)
    _load().oracle_quantize(_ptr(x), rows, cols, cols, _ptr(q), _ptr(s))
    return q, s


def dequantize(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = np.ascontiguousarray(s, dtype=np.uint8)
    rows, cols = q.shape[0], q.shape[1] * 2
    x = np.empty((rows, cols), np.float64)
    _load().oracle_dequantize(_ptr(q), _ptr(s), rows, cols, _ptr(x))
    return x


def gemm(aq, as_, bq, bs) -> tuple[np.ndarray, np.ndarray]:
    """C = deq(A) @ deq(B)^T: returns (fp64 sums [M, N], bf16 bits uint16 [M, N])."""
    aq, as_, bq, bs = (np.ascontiguousarray(t, dtype=np.uint8) for t in (aq, as_, bq, bs))
    M, K = aq.shape[0], aq.shape[1] * 2
    N = bq.shape[0]
    assert bq.shape[1] * 2 == K and as_.shape == (M, K // 32) and bs.shape == (N, K // 32)
    c64 = np.empty((M, N), np.float64)
    c16 = np.empty((M, N), np.uint16)
    _load().oracle_gemm(_ptr(aq), _ptr(as_), _ptr(bq), _ptr(bs), M, N, K, _ptr(c64), _ptr(c16))
    return c64, c16


def gemm_sampled(aq, as_, bq, bs, ms, ns) -> tuple[np.ndarray, np.ndarray]:
    """The GEMM at the listed output positions only: C[ms[i], ns[i]]."""
    aq, as_, bq, bs = (np.ascontiguousarray(t, dtype=np.uint8) for t in (aq, as_, bq, bs))
    K = aq.shape[1] * 2
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    assert ms.shape == ns.shape
    c64 = np.empty(ms.shape, np.float64)
    c16 = np.empty(ms.shape, np.uint16)
    _load().oracle_gemm_sampled(_ptr(aq), _ptr(as_), _ptr(bq), _ptr(bs), K, _ptr(ms), _ptr(ns),
                                ms.size, _ptr(c64), _ptr(c16))
    return c64, c16


def quant_gemm(a, bq, bs):
    """The whole layer: quantize bf16 A, multiply by pre-quantized B.

    Returns (aq, as, c64, c16)."""
    a = _u16(a)
    M, K = a.shape
    bq = np.ascontiguousarray(bq, dtype=np.uint8)
    bs = np.ascontiguousarray(bs, dtype=np.uint8)
    N = bq.shape[0]
    aq = np.empty((M, K // 2), np.uint8)
    as_ = np.empty((M, K // 32), np.uint8)
    c64 = np.empty((M, N), np.float64)
    c16 = np.empty((M, N), np.uint16)
    _load().oracle_quant_gemm(_ptr(a), K, _ptr(bq), _ptr(bs), M, N, K, _ptr(aq), _ptr(as_),
                              _ptr(c64), _ptr(c16))
    return aq, as_, c64, c16
