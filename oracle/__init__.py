"""Plain CPU oracle for the TQ2_0-style ternary matvec (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It wraps ``tq2_oracle.c`` (plain C,
one element at a time, fp64 accumulation, an exact __int128 variant) with
numpy-friendly functions.  It shares no code with the CUDA library.

The C source cites the passages it follows:
* "BitCPM-CANN-8B -> Core AI, ternary 1.58-bit" page: the TQ2_0 format, the
  recovery of d and the codes from a dequantised W, the linear factoring of
  the matvec;
* "Custom Metal kernels" page, the note on asymmetric (zero-point) int4:
  the affine-int4 matvec with the zero point factored out,
  acc += s * (dot - z * sum x);
* "gemma4 wNa8o8 requires int8 activations" page: the static int8
  fake-quant of the activations and its reciprocal-multiply form, and the
  same fake-quant of a linear's output at store (requantisation).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tq2_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_tq2.so")

FLAG_BAD_CODE = 1
FLAG_NONFINITE = 2
FLAG_INEXACT = 4

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into ``oracle/_build`` (if stale)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=gnu99", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        F = ctypes.c_float
        lib.tq2o_half_to_double.argtypes = [ctypes.c_uint16]
        lib.tq2o_half_to_double.restype = ctypes.c_double
        lib.tq2o_double_to_half.argtypes = [ctypes.c_double]
        lib.tq2o_double_to_half.restype = ctypes.c_uint16
        lib.tq2o_pack.argtypes = [P, I64, I64, P]
        lib.tq2o_pack.restype = ctypes.c_uint32
        lib.tq2o_unpack.argtypes = [P, I64, I64, P]
        lib.tq2o_unpack.restype = None
        lib.tq2o_dequant.argtypes = [P, P, I64, I64, P]
        lib.tq2o_dequant.restype = None
        lib.tq2o_from_dense_f32.argtypes = [P, I64, I64, P, P]
        lib.tq2o_from_dense_f32.restype = ctypes.c_uint32
        lib.tq2o_from_dense_f16.argtypes = [P, I64, I64, P, P]
        lib.tq2o_from_dense_f16.restype = ctypes.c_uint32
        lib.tq2o_fakequant_codes.argtypes = [P, I64, F, ctypes.c_int, P]
        lib.tq2o_fakequant_codes.restype = None
        lib.tq2o_fakequant.argtypes = [P, I64, F, ctypes.c_int, P]
        lib.tq2o_fakequant.restype = None
        lib.tq2o_requant.argtypes = [P, I64, F, P, P]
        lib.tq2o_requant.restype = None
        lib.tq2o_matvec_f64.argtypes = [P, I64, P, P, I64, I64, F, P, P]
        lib.tq2o_matvec_f64.restype = None
        lib.tq2o_matvec_rows_f64.argtypes = [P, I64, P, P, I64, I64, F, P, I64, P, P]
        lib.tq2o_matvec_rows_f64.restype = None
        lib.tq2o_matvec_exact.argtypes = [P, I64, P, P, I64, I64, F, P]
        lib.tq2o_matvec_exact.restype = ctypes.c_int64
        lib.tq2o_affine4_f64.argtypes = [P, I64, P, P, P, I64, I64, I64, P, P]
        lib.tq2o_affine4_f64.restype = None
        lib.tq2o_affine4_rows_f64.argtypes = [P, I64, P, P, P, I64, I64, I64, P, I64, P, P]
        lib.tq2o_affine4_rows_f64.restype = None
        lib.tq2o_affine4_exact.argtypes = [P, I64, P, P, P, I64, I64, I64, P]
        lib.tq2o_affine4_exact.restype = ctypes.c_int64
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _bits16(a) -> np.ndarray:
    """fp16 array (or its uint16 bit patterns) as contiguous uint16 bits."""
    a = np.asarray(a)
    if a.dtype == np.float16:
        return np.ascontiguousarray(a).view(np.uint16)
    return _c(a, np.uint16)


def _check_shape(N, K):
    if K % 256 or N < 0 or K < 0:
        raise ValueError("K must be a non-negative multiple of 256")


# ---------------------------------------------------------------- scalars
def half_to_double(h: int) -> float:
    return _load().tq2o_half_to_double(int(h) & 0xFFFF)


def double_to_half(v: float) -> int:
    return int(_load().tq2o_double_to_half(float(v)))


def half_bits_to_f64(bits) -> np.ndarray:
    """Decode an array of binary16 bit patterns (the oracle's own decoder)."""
    b = _bits16(bits)
    lib = _load()
    flat = b.reshape(-1)
    out = np.fromiter((lib.tq2o_half_to_double(int(v)) for v in flat),
                      dtype=np.float64, count=flat.size)
    return out.reshape(b.shape)


# ---------------------------------------------------------------- layout
def pack(codes: np.ndarray):
    """codes [N,K] int8 -> (qs [N,K/4] uint8, flags)."""
    c = _c(codes, np.int8)
    N, K = c.shape
    if K % 4:
        raise ValueError("K must be a multiple of 4")
    qs = np.zeros((N, K // 4), dtype=np.uint8)
    flags = _load().tq2o_pack(_ptr(c), N, K, _ptr(qs))
    return qs, int(flags)


def unpack(qs: np.ndarray, K: int) -> np.ndarray:
    """qs [N,K/4] uint8 -> codes [N,K] int8."""
    q = _c(qs, np.uint8)
    N = q.shape[0]
    assert q.shape[1] * 4 == K
    out = np.zeros((N, K), dtype=np.int8)
    _load().tq2o_unpack(_ptr(q), N, K, _ptr(out))
    return out


def dequant(qs: np.ndarray, d: np.ndarray, K: int) -> np.ndarray:
    """W = d_b * (q - 1) as fp32 [N,K]."""
    q = _c(qs, np.uint8)
    db = _bits16(d)
    N = q.shape[0]
    _check_shape(N, K)
    W = np.zeros((N, K), dtype=np.float32)
    _load().tq2o_dequant(_ptr(q), _ptr(db), N, K, _ptr(W))
    return W


def from_dense(W: np.ndarray):
    """Dequantised W [N,K] (fp32 or fp16) -> (qs, d fp16, flags)."""
    W = np.asarray(W)
    N, K = W.shape
    _check_shape(N, K)
    qs = np.zeros((N, K // 4), dtype=np.uint8)
    d = np.zeros((N, K // 256), dtype=np.uint16)
    lib = _load()
    if W.dtype == np.float16:
        w = np.ascontiguousarray(W).view(np.uint16)
        flags = lib.tq2o_from_dense_f16(_ptr(w), N, K, _ptr(qs), _ptr(d))
    else:
        w = _c(W, np.float32)
        flags = lib.tq2o_from_dense_f32(_ptr(w), N, K, _ptr(qs), _ptr(d))
    return qs, d.view(np.float16), int(flags)


# ---------------------------------------------------------------- fake-quant
def fakequant_codes(x: np.ndarray, s: float, mode: int = 0) -> np.ndarray:
    """Integer fake-quant codes of fp16 x (mode 0: fp32 x*(1/s); 1: fp64 x/s)."""
    xb = _bits16(x)
    q = np.zeros(xb.shape, dtype=np.int8)
    _load().tq2o_fakequant_codes(_ptr(xb), xb.size, float(np.float32(s)), int(mode), _ptr(q))
    return q


def fakequant(x: np.ndarray, s: float, mode: int = 0) -> np.ndarray:
    """x' = q * s in fp64."""
    xb = _bits16(x)
    out = np.zeros(xb.shape, dtype=np.float64)
    _load().tq2o_fakequant(_ptr(xb), xb.size, float(np.float32(s)), int(mode), _ptr(out))
    return out


def requant(y, s: float):
    """Output requantisation at store: (codes int8, y' = code * s fp64) of
    fp64 y, the decision taken as rint(fp32(y) * fp32(1/s)) in fp32."""
    yv = np.ascontiguousarray(np.asarray(y, dtype=np.float64))
    codes = np.zeros(yv.shape, dtype=np.int8)
    out = np.zeros(yv.shape, dtype=np.float64)
    _load().tq2o_requant(_ptr(yv), yv.size, float(np.float32(s)), _ptr(codes), _ptr(out))
    return codes, out


# ---------------------------------------------------------------- matvec
def matvec(x: np.ndarray, qs: np.ndarray, d: np.ndarray, K: int, act_scale: float = 0.0):
    """fp64 matvec: returns (y [M,N], tol_sum [M,N]) with
    tol_sum = sum_b |d_b| sum_{k in b} |x'_k|."""
    xb = _bits16(x)
    if xb.ndim == 1:
        xb = xb.reshape(1, -1)
    M = xb.shape[0]
    q = _c(qs, np.uint8)
    db = _bits16(d)
    N = q.shape[0]
    _check_shape(N, K)
    y = np.zeros((M, N), dtype=np.float64)
    t = np.zeros((M, N), dtype=np.float64)
    _load().tq2o_matvec_f64(_ptr(xb), M, _ptr(q), _ptr(db), N, K,
                            float(np.float32(act_scale)), _ptr(y), _ptr(t))
    return y, t


_executor = None


def _pool(n):
    """A persistent pool of at least n host threads (ctypes calls drop the GIL)."""
    global _executor
    from concurrent.futures import ThreadPoolExecutor
    with _lock:
        if _executor is None or _executor._max_workers < n:
            if _executor is not None:
                _executor.shutdown(wait=True)
            _executor = ThreadPoolExecutor(max_workers=n)
        return _executor


def matvec_threads(x: np.ndarray, qs: np.ndarray, d: np.ndarray, K: int, act_scale: float = 0.0,
                   threads: int = 1):
    """The same fp64 matvec (``matvec``) on ``threads`` host threads: the
    output rows are split into contiguous ranges and each range is one call
    of the C oracle (ctypes releases the GIL during the call).  The arithmetic
    per element is unchanged; only the rows run concurrently."""
    xb = _bits16(x)
    if xb.ndim == 1:
        xb = xb.reshape(1, -1)
    M = xb.shape[0]
    q = _c(qs, np.uint8)
    db = _bits16(d)
    N = q.shape[0]
    _check_shape(N, K)
    threads = max(1, min(int(threads), N if N > 0 else 1))
    lib = _load()
    bounds = [N * i // threads for i in range(threads + 1)]
    parts = [None] * threads

    def run(i):
        r0, r1 = bounds[i], bounds[i + 1]
        y = np.zeros((M, r1 - r0), dtype=np.float64)
        t = np.zeros((M, r1 - r0), dtype=np.float64)
        if r1 > r0:
            lib.tq2o_matvec_f64(_ptr(xb), M, _ptr(q[r0:r1]), _ptr(db[r0:r1]), r1 - r0, K,
                                float(np.float32(act_scale)), _ptr(y), _ptr(t))
        parts[i] = (y, t)

    if threads == 1:
        run(0)
    else:
        list(_pool(threads).map(run, range(threads)))
    return (np.concatenate([p_[0] for p_ in parts], axis=1),
            np.concatenate([p_[1] for p_ in parts], axis=1))


def matvec_rows(x, qs, d, K, rows, act_scale: float = 0.0):
    """fp64 matvec for the output rows ``rows`` only: (y, tol) [M, len(rows)]."""
    xb = _bits16(x)
    if xb.ndim == 1:
        xb = xb.reshape(1, -1)
    M = xb.shape[0]
    q = _c(qs, np.uint8)
    db = _bits16(d)
    N = q.shape[0]
    r = _c(rows, np.int64)
    assert r.size == 0 or (r.min() >= 0 and r.max() < N)
    y = np.zeros((M, r.size), dtype=np.float64)
    t = np.zeros((M, r.size), dtype=np.float64)
    _load().tq2o_matvec_rows_f64(_ptr(xb), M, _ptr(q), _ptr(db), N, K,
                                 float(np.float32(act_scale)), _ptr(r), r.size,
                                 _ptr(y), _ptr(t))
    return y, t


def matvec_exact(x, qs, d, K, act_scale: float = 0.0) -> np.ndarray:
    """Exact matvec (__int128 accumulation), rounded once to fp64."""
    xb = _bits16(x)
    if xb.ndim == 1:
        xb = xb.reshape(1, -1)
    M = xb.shape[0]
    q = _c(qs, np.uint8)
    db = _bits16(d)
    N = q.shape[0]
    y = np.zeros((M, N), dtype=np.float64)
    _load().tq2o_matvec_exact(_ptr(xb), M, _ptr(q), _ptr(db), N, K,
                              float(np.float32(act_scale)), _ptr(y))
    return y


def tolerance(tol_sum: np.ndarray) -> np.ndarray:
    """Per-element parity bound: 1e-3 * sum_k |d_b x_k| + 1e-6."""
    return 1e-3 * tol_sum + 1e-6


# ---------------------------------------------------------------- affine int4
def _affine4_args(x, qs, s, z, K, G):
    xb = _bits16(x)
    if xb.ndim == 1:
        xb = xb.reshape(1, -1)
    q = _c(qs, np.uint8)
    sb, zb = _bits16(s), _bits16(z)
    N = q.shape[0]
    if G < 1 or K % G or q.shape[1] * 2 != K or sb.shape != (N, K // G) or zb.shape != (N, K // G):
        raise ValueError("affine int4: qs [N, K/2], s and z [N, K/G], G | K")
    return xb, q, sb, zb, N


def affine4(x, qs, s, z, K: int, G: int):
    """fp64 affine-int4 matvec, zero point factored per group:
    (y [M,N], tol_sum [M,N]) with tol_sum = sum_g |s_g| sum_k |x_k| (q_k + |z_g|)."""
    xb, q, sb, zb, N = _affine4_args(x, qs, s, z, K, G)
    M = xb.shape[0]
    y = np.zeros((M, N), dtype=np.float64)
    t = np.zeros((M, N), dtype=np.float64)
    _load().tq2o_affine4_f64(_ptr(xb), M, _ptr(q), _ptr(sb), _ptr(zb), N, K, G, _ptr(y), _ptr(t))
    return y, t


def affine4_rows(x, qs, s, z, K: int, G: int, rows):
    """fp64 affine-int4 matvec for the output rows ``rows`` only."""
    xb, q, sb, zb, N = _affine4_args(x, qs, s, z, K, G)
    M = xb.shape[0]
    r = _c(rows, np.int64)
    assert r.size == 0 or (r.min() >= 0 and r.max() < N)
    y = np.zeros((M, r.size), dtype=np.float64)
    t = np.zeros((M, r.size), dtype=np.float64)
    _load().tq2o_affine4_rows_f64(_ptr(xb), M, _ptr(q), _ptr(sb), _ptr(zb), N, K, G, _ptr(r), r.size,
                                  _ptr(y), _ptr(t))
    return y, t


def affine4_exact(x, qs, s, z, K: int, G: int) -> np.ndarray:
    """Exact dense-form affine-int4 matvec (sum_k s(q - z) x_k in __int128),
    rounded once to fp64; NaN where a term could overflow the exact sum."""
    xb, q, sb, zb, N = _affine4_args(x, qs, s, z, K, G)
    M = xb.shape[0]
    y = np.zeros((M, N), dtype=np.float64)
    _load().tq2o_affine4_exact(_ptr(xb), M, _ptr(q), _ptr(sb), _ptr(zb), N, K, G, _ptr(y))
    return y
