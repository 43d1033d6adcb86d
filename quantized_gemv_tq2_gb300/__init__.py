"""Python binding of the GB300-native ternary (TQ2_0-style) matvec library.

Argument marshalling only: every step of the computation runs in the CUDA
library ``_lib/libtq2_gb300.so`` through its C ABI (``include/tq2.h``).
PyTorch supplies device memory and streams; there is no CPU fallback, and
the functions raise if the library is missing or a call fails.

Functions take CUDA tensors and the current torch stream (or an explicit
``stream``); outputs may be passed in or are allocated with torch.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

from . import build as _build

__all__ = [
    "TQ2Error", "lib", "load", "declared_symbols",
    "pack", "unpack", "from_dense", "matvec", "matvec_grouped", "gemm", "gemm_static_ws", "affine4_matvec",
    "matvec_workspace_size", "gemm_workspace_size",
    "status_string", "version",
    "F32", "F16", "FLAG_BAD_CODE", "FLAG_NONFINITE", "FLAG_INEXACT", "FLAG_TIMEOUT", "FLAG_BOUNDS",
    "bounds_checked", "traced", "trace_read",
    "IMPL_AUTO", "IMPL_MMA", "IMPL_SIMT", "IMPL_PS", "IMPL_GEMM", "IMPL_SMALLN",
]

F32, F16 = 0, 1
FLAG_BAD_CODE, FLAG_NONFINITE, FLAG_INEXACT, FLAG_TIMEOUT, FLAG_BOUNDS = 1, 2, 4, 8, 16
# (3 and 5 are retired kernel numbers: TQ2_ERR_ARG)
IMPL_AUTO, IMPL_MMA, IMPL_SIMT, IMPL_PS, IMPL_GEMM, IMPL_SMALLN = 0, 1, 2, 4, 6, 7
HEADER = os.path.join(os.path.dirname(_build.PKG), "include", "tq2.h")

_lock = threading.Lock()
_lib = None


class TQ2Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {status_string(status)} (status {status})"
        if status == 6:
            msg += f" [{load().tq2_last_cuda_error().decode()}]"
        super().__init__(msg)


def bounds_checked() -> bool:
    """True when this process uses the bounds-checked debug library
    (environment TQ2_BOUNDS_CHECK=1, read at the first load)."""
    return os.environ.get("TQ2_BOUNDS_CHECK", "0") not in ("", "0")


def traced() -> bool:
    """True when this process uses the trace library (environment
    TQ2_TRACE=1, read at the first load; the bounds-checked one wins)."""
    return not bounds_checked() and os.environ.get("TQ2_TRACE", "0") not in ("", "0")


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load the CUDA library (building it in-tree first if it is missing):
    the release build, or the bounds-checked one when TQ2_BOUNDS_CHECK=1."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        variant = "check" if bounds_checked() else ("trace" if traced() else "release")
        path = _build.lib_path(variant=variant)
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError(f"CUDA library not built: {path}")
            _build.build(variant=variant)
        L = ctypes.CDLL(path)
        P, I64, I32, F, SZ = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float,
                              ctypes.c_size_t)
        L.tq2_pack.argtypes = [P, I64, I64, P, P, P]
        L.tq2_unpack.argtypes = [P, I64, I64, P, P]
        L.tq2_from_dense.argtypes = [P, I32, I64, I64, P, P, P, P]
        L.tq2_matvec.argtypes = [P, I64, P, P, I64, I64, P, I32, F, P, SZ, P, P]
        L.tq2_matvec_impl.argtypes = [P, I64, P, P, I64, I64, P, I32, F, P, SZ, P, P, I32]
        L.tq2_matvec_requant.argtypes = [P, I64, P, P, I64, I64, P, I32, F, F, P, SZ, P, P, I32]
        L.tq2_matvec_grouped.argtypes = [P, I64, I64, I32, P, P, P, P, I32, F, P, SZ, P, P]
        L.tq2_matvec_grouped_requant.argtypes = [P, I64, I64, I32, P, P, P, P, I32, F, P, P, SZ, P, P]
        L.tq2_matvec_grouped_workspace_size.argtypes = [I64, I64, I32, P]
        L.tq2_matvec_grouped_workspace_size.restype = SZ
        L.tq2_gemm.argtypes = [P, I64, P, P, I64, I64, P, I32, F, F, P, SZ, P, P, I32]
        L.tq2_affine4_matvec.argtypes = [P, I64, P, P, P, I64, I64, I64, P, I32, P, P]
        L.tq2_test_matvec_stall.argtypes = [P, I64, P, P, I64, I64, P, P, P, I32, I32]
        L.tq2_test_gemm_stall.argtypes = [P, I64, P, P, I64, I64, P, F, P, P, I32, I32]
        L.tq2_matvec_workspace_size.argtypes = [I64, I64, I64]
        L.tq2_trace_size.argtypes = []
        L.tq2_trace_size.restype = SZ
        L.tq2_trace_read.argtypes = [P, SZ]
        L.tq2_matvec_workspace_size.restype = SZ
        L.tq2_gemm_workspace_size.argtypes = [I64, I64, I64]
        L.tq2_gemm_static_ws.argtypes = [P, I64, P, P, I64, I64, P, I32, F, F, P, P, I32]
        L.tq2_gemm_workspace_size.restype = SZ
        L.tq2_status_string.argtypes = [I32]
        L.tq2_status_string.restype = ctypes.c_char_p
        L.tq2_version.argtypes = []
        L.tq2_last_cuda_error.argtypes = []
        L.tq2_last_cuda_error.restype = ctypes.c_char_p
        for fn in ("tq2_pack", "tq2_unpack", "tq2_from_dense", "tq2_matvec", "tq2_matvec_impl",
                   "tq2_matvec_requant", "tq2_matvec_grouped", "tq2_matvec_grouped_requant", "tq2_gemm",
                   "tq2_gemm_static_ws", "tq2_affine4_matvec",
                   "tq2_test_matvec_stall", "tq2_test_gemm_stall", "tq2_trace_read", "tq2_version"):
            getattr(L, fn).restype = ctypes.c_int
        _lib = L
        return L


def lib() -> ctypes.CDLL:
    return load()


def declared_symbols() -> list[str]:
    """Function names declared by include/tq2.h (the ABI this library exports)."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"TQ2_API\s+[\w\s\*]*?\b(tq2_\w+)\s*\(", text)))


def status_string(status: int) -> str:
    return load().tq2_status_string(int(status)).decode()


def version() -> int:
    return int(load().tq2_version())


# ------------------------------------------------------------------ helpers
def _torch():
    import torch
    return torch


def _stream_ptr(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr() if t is not None else 0)


def _check(status: int, where: str):
    if status != 0:
        raise TQ2Error(status, where)


def _workspace(workspace, act_scale, nbytes_fn, device, stream):
    """(pointer, bytes) of the scratch a call may use for the prologue as a
    pass of its own: "auto" allocates what the library asks for (nothing
    without the prologue, or where the library would not use it), None
    passes none (each kernel then converts x itself), a tensor is passed
    as is.  Returns the tensor too, to keep it alive for the call."""
    if workspace is None or (isinstance(workspace, str) and (act_scale == 0.0)):
        return ctypes.c_void_p(0), 0, None
    if isinstance(workspace, str):
        if workspace != "auto":
            raise ValueError("workspace must be 'auto', None or a CUDA tensor")
        nbytes = int(nbytes_fn())
        if nbytes == 0:
            return ctypes.c_void_p(0), 0, None
        torch = _torch()
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
        if stream is not None and not isinstance(stream, int):
            workspace.record_stream(stream)  # freed for reuse only after that stream's work
    _need_cuda(workspace)
    return _ptr(workspace), workspace.numel() * workspace.element_size(), workspace


def _need_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


# ------------------------------------------------------------------ ops
def pack(codes, qs=None, status=None, stream=None):
    """int8 codes [N,K] -> packed uint8 [N,K/4] (tq2_pack)."""
    torch = _torch()
    N, K = codes.shape
    if codes.dtype != torch.int8:
        raise TypeError("codes must be int8")
    if qs is None:
        qs = torch.empty((N, K // 4), dtype=torch.uint8, device=codes.device)
    _need_cuda(codes, qs, status)
    _check(load().tq2_pack(_ptr(codes), N, K, _ptr(qs), _ptr(status), _stream_ptr(stream)),
           "tq2_pack")
    return qs


def unpack(qs, K, codes=None, stream=None):
    """packed uint8 [N,K/4] -> int8 codes [N,K] (tq2_unpack)."""
    torch = _torch()
    N = qs.shape[0]
    if codes is None:
        codes = torch.empty((N, K), dtype=torch.int8, device=qs.device)
    _need_cuda(codes, qs)
    _check(load().tq2_unpack(_ptr(qs), N, K, _ptr(codes), _stream_ptr(stream)), "tq2_unpack")
    return codes


def from_dense(W, qs=None, d=None, status=None, stream=None):
    """Dequantised W [N,K] (float32/float16) -> (qs uint8 [N,K/4], d float16 [N,K/256])."""
    torch = _torch()
    N, K = W.shape
    if W.dtype == torch.float32:
        wd = F32
    elif W.dtype == torch.float16:
        wd = F16
    else:
        raise TypeError("W must be float32 or float16")
    if qs is None:
        qs = torch.empty((N, K // 4), dtype=torch.uint8, device=W.device)
    if d is None:
        d = torch.empty((N, K // 256), dtype=torch.float16, device=W.device)
    _need_cuda(W, qs, d, status)
    _check(load().tq2_from_dense(_ptr(W), wd, N, K, _ptr(qs), _ptr(d), _ptr(status),
                                 _stream_ptr(stream)), "tq2_from_dense")
    return qs, d


def matvec(x, qs, d, K=None, y=None, y_dtype=None, act_scale: float = 0.0, status=None,
           stream=None, impl: int = IMPL_AUTO, workspace="auto", out_scale: float = 0.0):
    """y [M,N] = ternary matvec of x [M,K] fp16 with packed qs/d (tq2_matvec);
    out_scale > 0 requantises y to int8 at store (tq2_matvec_requant).
    workspace: scratch for the prologue as a pass of its own ("auto": what
    tq2_matvec_workspace_size asks for; None: none; or a CUDA tensor)."""
    torch = _torch()
    if x.dim() == 1:
        x = x.view(1, -1)
    M = x.shape[0]
    N = qs.shape[0]
    if K is None:
        K = x.shape[1]
    if x.dtype != torch.float16 or d.dtype != torch.float16 or qs.dtype != torch.uint8:
        raise TypeError("x and d must be float16, qs uint8")
    if y is None:
        dt = torch.float32 if (y_dtype in (None, F32, torch.float32)) else torch.float16
        y = torch.empty((M, N), dtype=dt, device=qs.device)
    ycode = F32 if y.dtype == torch.float32 else F16
    _need_cuda(x, qs, d, y, status)
    L = load()
    ws_ptr, ws_bytes, _ws = _workspace(workspace, act_scale, lambda: L.tq2_matvec_workspace_size(M, N, K),
                                       qs.device, stream)
    if out_scale != 0.0:
        st = L.tq2_matvec_requant(_ptr(x), M, _ptr(qs), _ptr(d), N, K, _ptr(y), ycode,
                                  float(act_scale), float(out_scale), ws_ptr, ws_bytes, _ptr(status),
                                  _stream_ptr(stream), int(impl))
    elif impl == IMPL_AUTO:
        st = L.tq2_matvec(_ptr(x), M, _ptr(qs), _ptr(d), N, K, _ptr(y), ycode, float(act_scale),
                          ws_ptr, ws_bytes, _ptr(status), _stream_ptr(stream))
    else:
        st = L.tq2_matvec_impl(_ptr(x), M, _ptr(qs), _ptr(d), N, K, _ptr(y), ycode,
                               float(act_scale), ws_ptr, ws_bytes, _ptr(status),
                               _stream_ptr(stream), int(impl))
    _check(st, "tq2_matvec")
    return y


def matvec_grouped(x, qs_list, d_list, y_list=None, y_dtype=None, act_scale: float = 0.0,
                   status=None, stream=None, out_scales=None, workspace="auto"):
    """[y_j] = ternary matvecs of one shared x [M,K] with several packed
    matrices (tq2_matvec_grouped): one launch when the library can group them.
    out_scales (one float per matrix) requantises each y_j to int8 at store
    with its own scale (tq2_matvec_grouped_requant).  workspace as for matvec
    (tq2_matvec_grouped_workspace_size: x converted once for the group)."""
    torch = _torch()
    if x.dim() == 1:
        x = x.view(1, -1)
    M, K = x.shape
    n = len(qs_list)
    if n != len(d_list) or (y_list is not None and len(y_list) != n):
        raise ValueError("qs_list, d_list and y_list must have the same length")
    if x.dtype != torch.float16 or any(d.dtype != torch.float16 for d in d_list) or \
            any(q.dtype != torch.uint8 for q in qs_list):
        raise TypeError("x and d must be float16, qs uint8")
    if y_list is None:
        dt = torch.float32 if (y_dtype in (None, F32, torch.float32)) else torch.float16
        y_list = [torch.empty((M, q.shape[0]), dtype=dt, device=q.device) for q in qs_list]
    ycode = F32 if y_list[0].dtype == torch.float32 else F16
    _need_cuda(x, *qs_list, *d_list, *y_list, status)
    Pn = ctypes.c_void_p * n
    qa = Pn(*[_ptr(q).value for q in qs_list])
    da = Pn(*[_ptr(d).value for d in d_list])
    ya = Pn(*[_ptr(y).value for y in y_list])
    na = (ctypes.c_int64 * n)(*[q.shape[0] for q in qs_list])
    L = load()
    ws_ptr, ws_bytes, _ws = _workspace(
        workspace, act_scale,
        lambda: L.tq2_matvec_grouped_workspace_size(M, K, n, ctypes.cast(na, ctypes.c_void_p)), x.device, stream)
    common = (_ptr(x), M, K, n, ctypes.cast(qa, ctypes.c_void_p), ctypes.cast(da, ctypes.c_void_p),
              ctypes.cast(na, ctypes.c_void_p), ctypes.cast(ya, ctypes.c_void_p), ycode, float(act_scale))
    if out_scales is None:
        st = L.tq2_matvec_grouped(*common, ws_ptr, ws_bytes, _ptr(status), _stream_ptr(stream))
        _check(st, "tq2_matvec_grouped")
    else:
        if len(out_scales) != n:
            raise ValueError("out_scales needs one scale per matrix")
        sa = (ctypes.c_float * n)(*[float(v) for v in out_scales])
        st = L.tq2_matvec_grouped_requant(*common, ctypes.cast(sa, ctypes.c_void_p), ws_ptr, ws_bytes,
                                          _ptr(status), _stream_ptr(stream))
        _check(st, "tq2_matvec_grouped_requant")
    return y_list


def gemm(x, qs, d, y=None, y_dtype=None, act_scale: float = 0.0, out_scale: float = 0.0, status=None,
         stream=None, impl: int = 0, workspace="auto"):
    """y [M,N] for any M (prefill): tq2_gemm; impl 0 auto, 1 the tcgen05 GEMM,
    2 the matvec kernels on 16-row slices.  workspace as for matvec
    (tq2_gemm_workspace_size)."""
    torch = _torch()
    M, K = x.shape
    N = qs.shape[0]
    if x.dtype != torch.float16 or d.dtype != torch.float16 or qs.dtype != torch.uint8:
        raise TypeError("x and d must be float16, qs uint8")
    if y is None:
        dt = torch.float32 if (y_dtype in (None, F32, torch.float32)) else torch.float16
        y = torch.empty((M, N), dtype=dt, device=qs.device)
    ycode = F32 if y.dtype == torch.float32 else F16
    _need_cuda(x, qs, d, y, status)
    L = load()
    ws_ptr, ws_bytes, _ws = _workspace(workspace, act_scale, lambda: L.tq2_gemm_workspace_size(M, N, K),
                                       qs.device, stream)
    _check(L.tq2_gemm(_ptr(x), M, _ptr(qs), _ptr(d), N, K, _ptr(y), ycode, float(act_scale),
                      float(out_scale), ws_ptr, ws_bytes, _ptr(status), _stream_ptr(stream), int(impl)),
           "tq2_gemm")
    return y


def gemm_static_ws(x, qs, d, y=None, y_dtype=None, act_scale: float = 0.0, out_scale: float = 0.0, status=None,
                   stream=None, impl: int = 0):
    """tq2_gemm_static_ws: gemm whose prologue pass uses the library's static
    scratch (M * K <= 2**23 with the prologue) instead of a workspace."""
    torch = _torch()
    M, K = x.shape
    N = qs.shape[0]
    if x.dtype != torch.float16 or d.dtype != torch.float16 or qs.dtype != torch.uint8:
        raise TypeError("x and d must be float16, qs uint8")
    if y is None:
        dt = torch.float32 if (y_dtype in (None, F32, torch.float32)) else torch.float16
        y = torch.empty((M, N), dtype=dt, device=qs.device)
    ycode = F32 if y.dtype == torch.float32 else F16
    _need_cuda(x, qs, d, y, status)
    _check(load().tq2_gemm_static_ws(_ptr(x), M, _ptr(qs), _ptr(d), N, K, _ptr(y), ycode, float(act_scale),
                                     float(out_scale), _ptr(status), _stream_ptr(stream), int(impl)),
           "tq2_gemm_static_ws")
    return y


def affine4_matvec(x, qs, s, z, G: int, y=None, y_dtype=None, status=None, stream=None):
    """Affine-int4 matvec y [M,N] = W x with W = s (q - z) per group of G codes
    (tq2_affine4_matvec): qs uint8 [N, K/2] (low nibble first), s and z fp16
    [N, K/G], x fp16 [M, K] with M <= 16."""
    torch = _torch()
    M, K = x.shape
    N = qs.shape[0]
    if (x.dtype != torch.float16 or s.dtype != torch.float16 or z.dtype != torch.float16
            or qs.dtype != torch.uint8):
        raise TypeError("x, s and z must be float16, qs uint8")
    if y is None:
        dt = torch.float32 if (y_dtype in (None, F32, torch.float32)) else torch.float16
        y = torch.empty((M, N), dtype=dt, device=qs.device)
    ycode = F32 if y.dtype == torch.float32 else F16
    _need_cuda(x, qs, s, z, y, status)
    _check(load().tq2_affine4_matvec(_ptr(x), M, _ptr(qs), _ptr(s), _ptr(z), N, K, int(G), _ptr(y), ycode,
                                     _ptr(status), _stream_ptr(stream)), "tq2_affine4_matvec")
    return y


def test_matvec_stall(x, qs, d, status, stall_stage: int, wait_limit_us: int, y=None, stream=None):
    """Test hook (tq2_test_matvec_stall): the class-column kernel (impl 1,
    fp32 y) with the weight copy of one pipeline stage skipped and every
    device wait limited to wait_limit_us, so that the timeout path runs and
    sets TQ2_FLAG_TIMEOUT in status.  Not part of the product."""
    torch = _torch()
    if x.dim() == 1:
        x = x.view(1, -1)
    M, K = x.shape
    N = qs.shape[0]
    if x.dtype != torch.float16 or d.dtype != torch.float16 or qs.dtype != torch.uint8:
        raise TypeError("x and d must be float16, qs uint8")
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=qs.device)
    if y.dtype != torch.float32:
        raise TypeError("y must be float32")
    _need_cuda(x, qs, d, y, status)
    _check(load().tq2_test_matvec_stall(_ptr(x), M, _ptr(qs), _ptr(d), N, K, _ptr(y), _ptr(status),
                                        _stream_ptr(stream), int(stall_stage), int(wait_limit_us)),
           "tq2_test_matvec_stall")
    return y


def test_gemm_stall(x, qs, d, status, stall_stage: int, wait_limit_us: int, act_scale: float = 0.0, y=None,
                    stream=None):
    """Test hook (tq2_test_gemm_stall): the tcgen05 GEMM with one x stage's
    copy skipped in every CTA and the stage-ring waits limited to
    wait_limit_us, so that its timeout path runs.  Not part of the product."""
    torch = _torch()
    M, K = x.shape
    N = qs.shape[0]
    if x.dtype != torch.float16 or d.dtype != torch.float16 or qs.dtype != torch.uint8:
        raise TypeError("x and d must be float16, qs uint8")
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=qs.device)
    if y.dtype != torch.float32:
        raise TypeError("y must be float32")
    _need_cuda(x, qs, d, y, status)
    _check(load().tq2_test_gemm_stall(_ptr(x), M, _ptr(qs), _ptr(d), N, K, _ptr(y), float(act_scale), _ptr(status),
                                      _stream_ptr(stream), int(stall_stage), int(wait_limit_us)),
           "tq2_test_gemm_stall")
    return y


def trace_read():
    """The trace build's phase stamps (tq2_trace_read) as a numpy uint64
    array [2 slots, 1024 CTAs, 8 phases]; raises outside the trace build."""
    import numpy as np
    L = load()
    n = int(L.tq2_trace_size())
    if n == 0:
        raise RuntimeError("not the trace build (set TQ2_TRACE=1 before the first load)")
    buf = np.zeros(n // 8, dtype=np.uint64)
    _check(L.tq2_trace_read(buf.ctypes.data_as(ctypes.c_void_p), n), "tq2_trace_read")
    return buf.reshape(2, -1, 8)


def matvec_workspace_size(M: int, N: int, K: int) -> int:
    return int(load().tq2_matvec_workspace_size(M, N, K))


def gemm_workspace_size(M: int, N: int, K: int) -> int:
    return int(load().tq2_gemm_workspace_size(M, N, K))
