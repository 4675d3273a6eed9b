"""Python binding of libw4q.so (include/w4q.h): argument marshalling only.

Every function takes torch CUDA tensors, checks dtype / shape / contiguity,
allocates outputs and workspace with torch when the caller passes none, and
calls the C entry point of the same name on the current CUDA stream.  All
arithmetic happens in the library's CUDA kernels; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libw4q.so")
GROUP = 32

_lib = None
_lock = threading.Lock()

W4Q_OK = 0
STATUS = {
    0: "W4Q_OK", 1: "W4Q_ERR_INVALID_ARG", 2: "W4Q_ERR_UNSUPPORTED", 3: "W4Q_ERR_MISALIGNED",
    4: "W4Q_ERR_WORKSPACE", 5: "W4Q_ERR_CUDA", 6: "W4Q_ERR_DEVICE",
}

# name -> (restype, argtypes) for every symbol of include/w4q.h
_P, _I64, _INT, _SZ, _U32P = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t,
                              ctypes.POINTER(ctypes.c_uint32))
SIGNATURES = {
    "w4q_status_string": (ctypes.c_char_p, [_INT]),
    "w4_packed_bytes": (_SZ, [_I64, _I64, _INT]),
    "w4_pack_weights": (_INT, [_P, _I64, _I64, _INT, _P, _P]),
    "w4_unpack_weights": (_INT, [_P, _I64, _I64, _INT, _P, _P, _P, _P]),
    "w4_workspace_bytes": (_SZ, [_I64, _I64, _I64, _INT]),
    "w4_workspace_bytes_split": (_SZ, [_I64, _I64, _I64, _INT, _INT]),
    "w4_split_choice": (_INT, [_I64, _I64, _I64, _INT]),
    "w4_kernel_launches": (_INT, [_I64, _I64, _I64, _INT, _INT]),
    "w4a16_gemm": (_INT, [_P, _P, _P, _I64, _I64, _I64, _INT, _P, _SZ, _P]),
    "w4a16_gemm_split": (_INT, [_P, _P, _P, _I64, _I64, _I64, _INT, _INT, _P, _SZ, _P]),
    "w4a16_gemm_noalloc": (_INT, [_P, _P, _P, _I64, _I64, _I64, _INT, _P]),
    "w4a8_gemm": (_INT, [_P, _P, _P, _I64, _I64, _I64, _INT, _P, _SZ, _P]),
    "w4a8_gemm_split": (_INT, [_P, _P, _P, _I64, _I64, _I64, _INT, _INT, _P, _SZ, _P]),
    "w4a8_quantize_act": (_INT, [_P, _I64, _I64, _P, _P, _P]),
    "w4a8_group_dots": (_INT, [_P, _P, _I64, _I64, _I64, _INT, _P, _P, _SZ, _P]),
    "w4a8_gemm_rowscale": (_INT, [_P, _P, _P, _I64, _I64, _I64, _INT, _P, _SZ, _P]),
    "w4a8_gemm_rowscale_split": (_INT, [_P, _P, _P, _I64, _I64, _I64, _INT, _INT, _P, _SZ, _P]),
    "w4a8_quantize_act_rowscale": (_INT, [_P, _I64, _I64, _P, _P, _P]),
    "w4a8_group_dots_rowscale": (_INT, [_P, _P, _I64, _I64, _I64, _INT, _P, _P, _SZ, _P]),
    "w8_gemv": (_INT, [_P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "w8_gemm": (_INT, [_P, _P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P]),
    "w8_workspace_bytes": (_SZ, [_I64, _I64, _I64]),
    "w8_kernel_launches": (_INT, [_I64, _I64, _I64]),
    "w4_packed_bytes_compact": (_SZ, [_I64, _I64, _INT]),
    "w4_pack_weights_compact": (_INT, [_P, _I64, _I64, _INT, _P, _P]),
    "w4_unpack_weights_compact": (_INT, [_P, _I64, _I64, _INT, _P, _P, _P, _P, _P]),
    "w4a16_gemm_compact": (_INT, [_P, _P, _P, _I64, _I64, _I64, _INT, _P]),
    "w4q_device_error": (_INT, [_U32P]),
    "w4q_selftest_wait_expiry": (_INT, [ctypes.c_uint, _P]),
}


class W4QError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__("%s failed: %s" % (fn, STATUS.get(status, status)))


def lib():
    """The loaded libw4q.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError("libw4q.so is not built (run __graft_entry__.build() or "
                                   "python gemv_w4a16_gemm_gb300/build.py)")
            l = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(l, name)
                fn.restype = res
                fn.argtypes = args
            _lib = l
    return _lib


def _check(fn: str, status: int):
    if status != W4Q_OK:
        raise W4QError(fn, status)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _cuda(t: torch.Tensor, dtype, name: str):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t.data_ptr()


def status_string(status: int) -> str:
    return lib().w4q_status_string(status).decode()


def packed_bytes(N: int, K: int, group: int = GROUP) -> int:
    return int(lib().w4_packed_bytes(N, K, group))


def workspace_bytes(M: int, N: int, K: int, group: int = GROUP, split_k: int | None = None) -> int:
    if split_k is None:
        return int(lib().w4_workspace_bytes(M, N, K, group))
    return int(lib().w4_workspace_bytes_split(M, N, K, group, split_k))


def split_choice(M: int, N: int, K: int, group: int = GROUP) -> int:
    return int(lib().w4_split_choice(M, N, K, group))


def kernel_launches(M: int, N: int, K: int, w4a8=False, group: int = GROUP) -> int:
    """Kernels one call launches: w4a8 False = W4A16, True or "group" = W4A8
    with a scale per group of 32, "row" = W4A8 with a scale per row."""
    mode = 2 if w4a8 == "row" else (1 if w4a8 else 0)
    return int(lib().w4_kernel_launches(M, N, K, group, mode))


def _workspace(M, N, K, group, split_k, workspace, device):
    # a given workspace is passed as is (the library checks its size)
    if workspace is None:
        need = workspace_bytes(M, N, K, group, split_k)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=device)
    return workspace, workspace.numel() * workspace.element_size()


def w4_pack_weights(W: torch.Tensor, group: int = GROUP, out: torch.Tensor | None = None,
                    stream=None) -> torch.Tensor:
    """bf16 [N,K] CUDA weight -> packed uint8 buffer (layout of include/w4q.h)."""
    N, K = W.shape
    pw = _cuda(W, torch.bfloat16, "W")
    nbytes = packed_bytes(N, K, group)
    if nbytes == 0:
        raise W4QError("w4_pack_weights", 2)
    if out is None:
        out = torch.empty(nbytes, dtype=torch.uint8, device=W.device)
    po = _cuda(out, torch.uint8, "out")
    _check("w4_pack_weights", lib().w4_pack_weights(pw, N, K, group, po, _stream(stream)))
    return out


def w4_unpack_weights(packed: torch.Tensor, N: int, K: int, group: int = GROUP, stream=None):
    """packed -> (q u8 [N,K], scale bf16 [N,K/32], zero u8 [N,K/32])."""
    dev = packed.device
    q = torch.empty(N, K, dtype=torch.uint8, device=dev)
    s = torch.empty(N, K // group, dtype=torch.bfloat16, device=dev)
    z = torch.empty(N, K // group, dtype=torch.uint8, device=dev)
    _check("w4_unpack_weights", lib().w4_unpack_weights(
        _cuda(packed, torch.uint8, "packed"), N, K, group, q.data_ptr(), s.data_ptr(),
        z.data_ptr(), _stream(stream)))
    return q, s, z


def _gemm(name, x, packed, N, K, group, split_k, out, workspace, stream):
    M = x.shape[0]
    if x.dim() != 2 or x.shape[1] != K:
        raise ValueError("x must be [M, %d]" % K)
    px = _cuda(x, torch.bfloat16, "x")
    pp = _cuda(packed, torch.uint8, "packed")
    if out is None:
        out = torch.empty(M, N, dtype=torch.bfloat16, device=x.device)
    po = _cuda(out, torch.bfloat16, "out")
    ws, wsb = _workspace(M, N, K, group, split_k, workspace, x.device)
    pws = _cuda(ws, ws.dtype, "workspace")
    l = lib()
    if split_k is None:
        st = getattr(l, name)(px, pp, po, M, N, K, group, pws, wsb, _stream(stream))
    else:
        st = getattr(l, name + "_split")(px, pp, po, M, N, K, group, split_k, pws, wsb,
                                         _stream(stream))
    _check(name, st)
    return out


def w4a16_gemm(x, packed, N, K, group=GROUP, split_k=None, out=None, workspace=None, stream=None):
    """out[M,N] = x . dequant(packed)^T (W4A16); split_k None = library choice."""
    return _gemm("w4a16_gemm", x, packed, N, K, group, split_k, out, workspace, stream)


def w4a16_gemm_noalloc(x, packed, N, K, group=GROUP, out=None, stream=None):
    """W4A16 without any workspace: the library's own static scratch array is
    used (for callers that cannot allocate; see include/w4q.h)."""
    M = x.shape[0]
    if x.dim() != 2 or x.shape[1] != K:
        raise ValueError("x must be [M, %d]" % K)
    if out is None:
        out = torch.empty(M, N, dtype=torch.bfloat16, device=x.device)
    _check("w4a16_gemm_noalloc", lib().w4a16_gemm_noalloc(
        _cuda(x, torch.bfloat16, "x"), _cuda(packed, torch.uint8, "packed"),
        _cuda(out, torch.bfloat16, "out"), M, N, K, group, _stream(stream)))
    return out


def w4a8_gemm(x, packed, N, K, group=GROUP, split_k=None, out=None, workspace=None, stream=None):
    """out[M,N] = x . dequant(packed)^T, W4A8 with one int8 activation scale
    per (row, group of 32)."""
    return _gemm("w4a8_gemm", x, packed, N, K, group, split_k, out, workspace, stream)


def w4a8_gemm_rowscale(x, packed, N, K, group=GROUP, split_k=None, out=None, workspace=None,
                       stream=None):
    """out[M,N] = x . dequant(packed)^T, W4A8 with one int8 activation scale
    per row (absmax / 127)."""
    return _gemm("w4a8_gemm_rowscale", x, packed, N, K, group, split_k, out, workspace, stream)


def _quantize_act(name, x, row, stream):
    M, K = x.shape
    xq = torch.empty(M, K, dtype=torch.int8, device=x.device)
    sx = torch.empty((M,) if row else (M, K // GROUP), dtype=torch.float32, device=x.device)
    _check(name, getattr(lib(), name)(
        _cuda(x, torch.bfloat16, "x"), M, K, xq.data_ptr(), sx.data_ptr(), _stream(stream)))
    return xq, sx


def w4a8_quantize_act(x: torch.Tensor, stream=None):
    """(xq int8 [M,K], sx fp32 [M, K/32]): the per-group W4A8 quantizer."""
    return _quantize_act("w4a8_quantize_act", x, False, stream)


def w4a8_quantize_act_rowscale(x: torch.Tensor, stream=None):
    """(xq int8 [M,K], sx fp32 [M]): the per-row W4A8 quantizer."""
    return _quantize_act("w4a8_quantize_act_rowscale", x, True, stream)


def _group_dots(name, x, packed, N, K, group, workspace, stream):
    M = x.shape[0]
    D = torch.empty(M, N, K // group, dtype=torch.int32, device=x.device)
    ws, wsb = _workspace(M, N, K, group, None, workspace, x.device)
    _check(name, getattr(lib(), name)(
        _cuda(x, torch.bfloat16, "x"), _cuda(packed, torch.uint8, "packed"), M, N, K, group,
        D.data_ptr(), ws.data_ptr(), wsb, _stream(stream)))
    return D


def w4a8_group_dots(x, packed, N, K, group=GROUP, workspace=None, stream=None):
    """Exact int32 W4A8 group dots [M, N, K/32] (per-group activation scales)."""
    return _group_dots("w4a8_group_dots", x, packed, N, K, group, workspace, stream)


def w4a8_group_dots_rowscale(x, packed, N, K, group=GROUP, workspace=None, stream=None):
    """Exact int32 W4A8 group dots [M, N, K/32] (per-row activation scales)."""
    return _group_dots("w4a8_group_dots_rowscale", x, packed, N, K, group, workspace, stream)


def packed_bytes_compact(N: int, K: int, group: int = GROUP) -> int:
    return int(lib().w4_packed_bytes_compact(N, K, group))


def w4_pack_weights_compact(W: torch.Tensor, group: int = GROUP, out: torch.Tensor | None = None,
                            stream=None) -> torch.Tensor:
    """bf16 [N,K] CUDA weight -> packed uint8 buffer with the compact metadata
    (uint8 scale / zero codes, fp16 row steps; layout of include/w4q.h)."""
    N, K = W.shape
    pw = _cuda(W, torch.bfloat16, "W")
    nbytes = packed_bytes_compact(N, K, group)
    if nbytes == 0:
        raise W4QError("w4_pack_weights_compact", 2)
    if out is None:
        out = torch.empty(nbytes, dtype=torch.uint8, device=W.device)
    po = _cuda(out, torch.uint8, "out")
    _check("w4_pack_weights_compact",
           lib().w4_pack_weights_compact(pw, N, K, group, po, _stream(stream)))
    return out


def w4_unpack_weights_compact(packed: torch.Tensor, N: int, K: int, group: int = GROUP,
                              stream=None):
    """packed -> (q u8 [N,K], scale codes u8 [N,K/32], zero codes u8 [N,K/32],
    steps fp16 [N,2])."""
    dev = packed.device
    q = torch.empty(N, K, dtype=torch.uint8, device=dev)
    sc = torch.empty(N, K // group, dtype=torch.uint8, device=dev)
    zc = torch.empty(N, K // group, dtype=torch.uint8, device=dev)
    st = torch.empty(N, 2, dtype=torch.float16, device=dev)
    _check("w4_unpack_weights_compact", lib().w4_unpack_weights_compact(
        _cuda(packed, torch.uint8, "packed"), N, K, group, q.data_ptr(), sc.data_ptr(),
        zc.data_ptr(), st.data_ptr(), _stream(stream)))
    return q, sc, zc, st


def w4a16_gemm_compact(x, packed, N, K, group=GROUP, out=None, stream=None):
    """out[M,N] = x . dequant(packed)^T with the compact metadata (M <= 8)."""
    M = x.shape[0]
    if x.dim() != 2 or x.shape[1] != K:
        raise ValueError("x must be [M, %d]" % K)
    if out is None:
        out = torch.empty(M, N, dtype=torch.bfloat16, device=x.device)
    _check("w4a16_gemm_compact", lib().w4a16_gemm_compact(
        _cuda(x, torch.bfloat16, "x"), _cuda(packed, torch.uint8, "packed"),
        _cuda(out, torch.bfloat16, "out"), M, N, K, group, _stream(stream)))
    return out


def w8_gemv(x, W, scales, out=None, stream=None):
    """out[M,N] = bf16((x . W^T) * scales), int8 W [N,K], bf16 scales [N]."""
    M, K = x.shape
    N = W.shape[0]
    px = _cuda(x, torch.bfloat16, "x")
    pw = _cuda(W, torch.int8, "W")
    ps = _cuda(scales, torch.bfloat16, "scales")
    if out is None:
        out = torch.empty(M, N, dtype=torch.bfloat16, device=x.device)
    po = _cuda(out, torch.bfloat16, "out")
    _check("w8_gemv", lib().w8_gemv(px, pw, ps, po, M, N, K, _stream(stream)))
    return out


def w8_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(lib().w8_workspace_bytes(M, N, K))


def w8_kernel_launches(M: int, N: int, K: int) -> int:
    return int(lib().w8_kernel_launches(M, N, K))


def w8_gemm(x, W, scales, out=None, workspace=None, stream=None):
    """w8_gemv for 1 <= M <= 64 (the tensor-core path needs a workspace;
    one is allocated when none is given)."""
    M, K = x.shape
    N = W.shape[0]
    px = _cuda(x, torch.bfloat16, "x")
    pw = _cuda(W, torch.int8, "W")
    ps = _cuda(scales, torch.bfloat16, "scales")
    if out is None:
        out = torch.empty(M, N, dtype=torch.bfloat16, device=x.device)
    po = _cuda(out, torch.bfloat16, "out")
    need = w8_workspace_bytes(M, N, K)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    pws = _cuda(workspace, torch.uint8, "workspace") if workspace is not None else None
    nbytes = workspace.numel() if workspace is not None else 0
    _check("w8_gemm", lib().w8_gemm(px, pw, ps, po, M, N, K, pws, nbytes, _stream(stream)))
    return out


def device_error() -> int:
    """Read and clear the device-side error word (synchronizes)."""
    v = ctypes.c_uint32(0)
    st = lib().w4q_device_error(ctypes.byref(v))
    if st not in (W4Q_OK, 6):
        raise W4QError("w4q_device_error", st)
    return int(v.value)
