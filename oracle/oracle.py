"""CPU oracle for the weight-only quantized linear layer -- TEST INFRASTRUCTURE.

Only the test-suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline leg may import this module.  It wraps ``w4q_oracle.c`` (plain C,
fp64) with numpy arrays; it shares no code with the CUDA library and never
imports it.

Every function cites the page and section it follows (see the C file's
header for the readings taken where the pages are silent):

* quantize_w4 / dequant_w4 -- "test_int4_quantized_gemm.py", _packed_with_dense
  (INT4, group 32 along K, asymmetric min-max).
* w4a16 -- "test_int4_quantized_gemm.py", the dequant + F.linear reference.
* act_quant / w4a8_group_dots / w4a8 -- "test_int4_quantized_gemm.py",
  W4A8 bucket kernels and Int4QuantizedGemmPrecisionTest (one activation
  scale per (row, group of 32)).
* act_quant_row / w4a8_row -- the same W4A8 with one activation scale per
  whole row (scale = absmax / 127), the scheme of the 39936 x 6656 W4A8
  workload.
* w8 -- "gpt-fast issue #114", WeightOnlyInt8Linear.forward.
* pack_w4 / unpack_w4 -- this library's packed layout (no page counterpart).
* quantize_w4c / dequant_w4c / pack_w4c / unpack_w4c / w4a16c -- the compact
  metadata of "test_int4_quantized_gemm.py"'s CudaCoalescedInt4Tensor (uint8
  scale and zero_point codes per group, float16 scale_step and
  zero_point_step per row), read as code x step for both (the page prints
  no dequant formula); the packed form is this library's own.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w4q_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

GROUP = 32


def build(force: bool = False) -> str:
    """Compile w4q_oracle.c into liboracle.so (OpenMP when gcc has it)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", "-fexcess-precision=standard", "-Wall"]
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    try:
        subprocess.run(base + ["-fopenmp", _SRC, "-o", tmp, "-lm"], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + [_SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            I = ctypes.c_int64
            sig = {
                "oracle_quantize_w4": [P, I, I, P, P, P],
                "oracle_dequant_w4": [P, P, P, I, I, P],
                "oracle_packed_bytes": [I, I],
                "oracle_pack_w4": [P, P, P, I, I, P],
                "oracle_unpack_w4": [P, I, I, P, P, P],
                "oracle_w4a16": [P, P, P, P, I, I, I, I, I, P],
                "oracle_act_quant": [P, I, I, P, P],
                "oracle_w4a8_group_dots": [P, P, P, I, I, I, P],
                "oracle_w4a8": [P, P, P, P, P, I, I, I, I, I, P],
                "oracle_act_quant_row": [P, I, I, P, P],
                "oracle_w4a8_row": [P, P, P, P, P, I, I, I, I, I, P],
                "oracle_w8": [P, P, P, I, I, I, I, I, P],
                "oracle_quantize_w4c": [P, I, I, P, P, P, P],
                "oracle_dequant_w4c": [P, P, P, P, I, I, P],
                "oracle_packed_bytes_c": [I, I],
                "oracle_pack_w4c": [P, P, P, P, I, I, P],
                "oracle_unpack_w4c": [P, I, I, P, P, P, P],
                "oracle_w4a16c": [P, P, P, P, P, I, I, I, I, I, P],
                "oracle_set_threads": [ctypes.c_int],
            }
            for name, args in sig.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = None
            lib.oracle_packed_bytes.restype = I
            lib.oracle_packed_bytes_c.restype = I
            lib.oracle_set_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _u16(a) -> np.ndarray:
    """bf16 data as raw uint16 bit patterns (accepts a torch tensor)."""
    if hasattr(a, "view") and hasattr(a, "dtype") and "torch" in str(type(a)):
        import torch
        a = a.detach().cpu().contiguous().view(torch.int16).numpy()
    return np.ascontiguousarray(a).view(np.uint16)


def set_threads(n: int = 0) -> int:
    """Set the OpenMP thread count (0 = leave as is); returns the count."""
    return int(_load().oracle_set_threads(int(n)))


def quantize_w4(W_bf16, N: int, K: int):
    """bf16 [N,K] -> (q u8 [N,K], s bf16-bits u16 [N,K/32], z u8 [N,K/32])."""
    W = _u16(W_bf16).reshape(N, K)
    q = np.empty((N, K), np.uint8)
    s = np.empty((N, K // GROUP), np.uint16)
    z = np.empty((N, K // GROUP), np.uint8)
    _load().oracle_quantize_w4(_ptr(W), N, K, _ptr(q), _ptr(s), _ptr(z))
    return q, s, z


def dequant_w4(q, s, z) -> np.ndarray:
    N, K = q.shape
    out = np.empty((N, K), np.float64)
    _load().oracle_dequant_w4(_ptr(q), _ptr(s), _ptr(z), N, K, _ptr(out))
    return out


def packed_bytes(N: int, K: int) -> int:
    return int(_load().oracle_packed_bytes(N, K))


def pack_w4(q, s, z) -> np.ndarray:
    N, K = q.shape
    out = np.empty(packed_bytes(N, K), np.uint8)
    _load().oracle_pack_w4(_ptr(q), _ptr(s), _ptr(z), N, K, _ptr(out))
    return out


def unpack_w4(packed, N: int, K: int):
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    q = np.empty((N, K), np.uint8)
    s = np.empty((N, K // GROUP), np.uint16)
    z = np.empty((N, K // GROUP), np.uint8)
    _load().oracle_unpack_w4(_ptr(packed), N, K, _ptr(q), _ptr(s), _ptr(z))
    return q, s, z


def w4a16(x_bf16, q, s, z, n0: int = 0, n1: int | None = None) -> np.ndarray:
    """fp64 out[M, n1-n0] of x . dequant(W)[n0:n1]^T."""
    N, K = q.shape
    x = _u16(x_bf16).reshape(-1, K)
    M = x.shape[0]
    n1 = N if n1 is None else n1
    out = np.empty((M, n1 - n0), np.float64)
    _load().oracle_w4a16(_ptr(x), _ptr(q), _ptr(s), _ptr(z), M, N, K, n0, n1,
                         _ptr(out))
    return out


def act_quant(x_bf16, K: int):
    """Symmetric int8 activations, one scale per (row, group of 32):
    (xq i8 [M,K], sx f32 [M, K/32])."""
    x = _u16(x_bf16).reshape(-1, K)
    M = x.shape[0]
    xq = np.empty((M, K), np.int8)
    sx = np.empty((M, K // GROUP), np.float32)
    _load().oracle_act_quant(_ptr(x), M, K, _ptr(xq), _ptr(sx))
    return xq, sx


def act_quant_row(x_bf16, K: int):
    """Symmetric int8 activations, one scale per whole row:
    (xq i8 [M,K], sx f32 [M])."""
    x = _u16(x_bf16).reshape(-1, K)
    M = x.shape[0]
    xq = np.empty((M, K), np.int8)
    sx = np.empty((M,), np.float32)
    _load().oracle_act_quant_row(_ptr(x), M, K, _ptr(xq), _ptr(sx))
    return xq, sx


def w4a8_group_dots(xq, q, z) -> np.ndarray:
    N, K = q.shape
    M = xq.shape[0]
    D = np.empty((M, N, K // GROUP), np.int32)
    _load().oracle_w4a8_group_dots(_ptr(np.ascontiguousarray(xq)), _ptr(q),
                                   _ptr(z), M, N, K, _ptr(D))
    return D


def w4a8(xq, sx, q, s, z, n0: int = 0, n1: int | None = None) -> np.ndarray:
    N, K = q.shape
    M = xq.shape[0]
    n1 = N if n1 is None else n1
    out = np.empty((M, n1 - n0), np.float64)
    _load().oracle_w4a8(_ptr(np.ascontiguousarray(xq)),
                        _ptr(np.ascontiguousarray(sx, dtype=np.float32)),
                        _ptr(q), _ptr(s), _ptr(z), M, N, K, n0, n1, _ptr(out))
    return out


def w4a8_row(xq, sx, q, s, z, n0: int = 0, n1: int | None = None) -> np.ndarray:
    """fp64 out[M, n1-n0] = sx[m] * sum_g s * D for per-row int8 activations."""
    N, K = q.shape
    M = xq.shape[0]
    n1 = N if n1 is None else n1
    out = np.empty((M, n1 - n0), np.float64)
    _load().oracle_w4a8_row(_ptr(np.ascontiguousarray(xq)),
                            _ptr(np.ascontiguousarray(sx, dtype=np.float32).reshape(M)),
                            _ptr(q), _ptr(s), _ptr(z), M, N, K, n0, n1, _ptr(out))
    return out


def w8(x_bf16, W_i8, scales_bf16, n0: int = 0, n1: int | None = None) -> np.ndarray:
    W = np.ascontiguousarray(W_i8, dtype=np.int8)
    N, K = W.shape
    x = _u16(x_bf16).reshape(-1, K)
    sc = _u16(scales_bf16).reshape(N)
    M = x.shape[0]
    n1 = N if n1 is None else n1
    out = np.empty((M, n1 - n0), np.float64)
    _load().oracle_w8(_ptr(x), _ptr(W), _ptr(sc), M, N, K, n0, n1, _ptr(out))
    return out


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- compact

def quantize_w4c(W_bf16, N: int, K: int):
    """bf16 [N,K] -> (q u8 [N,K], sc u8 [N,K/32], zc u8 [N,K/32], steps fp16-bits u16 [N,2])."""
    W = _u16(W_bf16).reshape(N, K)
    q = np.empty((N, K), np.uint8)
    sc = np.empty((N, K // GROUP), np.uint8)
    zc = np.empty((N, K // GROUP), np.uint8)
    steps = np.empty((N, 2), np.uint16)
    _load().oracle_quantize_w4c(_ptr(W), N, K, _ptr(q), _ptr(sc), _ptr(zc), _ptr(steps))
    return q, sc, zc, steps


def dequant_w4c(q, sc, zc, steps) -> np.ndarray:
    N, K = q.shape
    out = np.empty((N, K), np.float64)
    _load().oracle_dequant_w4c(_ptr(q), _ptr(sc), _ptr(zc), _ptr(np.ascontiguousarray(steps)),
                               N, K, _ptr(out))
    return out


def packed_bytes_c(N: int, K: int) -> int:
    return int(_load().oracle_packed_bytes_c(N, K))


def pack_w4c(q, sc, zc, steps) -> np.ndarray:
    N, K = q.shape
    out = np.empty(packed_bytes_c(N, K), np.uint8)
    _load().oracle_pack_w4c(_ptr(q), _ptr(sc), _ptr(zc), _ptr(np.ascontiguousarray(steps)),
                            N, K, _ptr(out))
    return out


def unpack_w4c(packed, N: int, K: int):
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    q = np.empty((N, K), np.uint8)
    sc = np.empty((N, K // GROUP), np.uint8)
    zc = np.empty((N, K // GROUP), np.uint8)
    steps = np.empty((N, 2), np.uint16)
    _load().oracle_unpack_w4c(_ptr(packed), N, K, _ptr(q), _ptr(sc), _ptr(zc), _ptr(steps))
    return q, sc, zc, steps


def w4a16c(x_bf16, q, sc, zc, steps, n0: int = 0, n1: int | None = None) -> np.ndarray:
    """fp64 out[M, n1-n0] of x . dequant_c(W)[n0:n1]^T."""
    N, K = q.shape
    x = _u16(x_bf16).reshape(-1, K)
    M = x.shape[0]
    n1 = N if n1 is None else n1
    out = np.empty((M, n1 - n0), np.float64)
    _load().oracle_w4a16c(_ptr(x), _ptr(q), _ptr(sc), _ptr(zc), _ptr(np.ascontiguousarray(steps)),
                          M, N, K, n0, n1, _ptr(out))
    return out
