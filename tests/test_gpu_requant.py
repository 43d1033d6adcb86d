"""GPU parity of tq2_matvec_requant: the matvec followed by the static int8
requantisation of y at store (gemma4 wNa8o8 page, "Implemented": fake-quant
at every linear boundary, output at store), against the CPU oracle.

The stored value must be code * out_scale (rounded to fp32, then to the y
dtype) with an int8 code; the code must be the oracle's requantisation of
some value within the matvec tolerance of the oracle's y, i.e. it may differ
from the oracle's own code only where y lies within that tolerance of a
rounding boundary (the kernel decides on its fp32 sum, the oracle on the
fp64 one)."""
import numpy as np
import pytest

import oracle
from gpu_util import Case, GuardedOutput, check_requant, host, sample_rows

pytestmark = pytest.mark.gpu

IMPLS = {"auto": 0, "mma": 1, "simt": 2, "ps": 4, "gemm": 6, "smalln": 7}


@pytest.fixture(scope="module")
def T():
    import torch
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    import quantized_gemv_tq2_gb300 as tq2
    tq2.load()
    return torch


def _impls_for(M):
    return ["auto", "mma", "ps", "gemm", "smalln", "simt"] if M <= 2 else ["auto", "ps", "gemm", "simt"]


def _run(T, case, impl, out_scale, y_dtype=0):
    import quantized_gemv_tq2_gb300 as tq2
    x, qs, d = case.device()
    st = T.zeros(1, dtype=T.int32, device="cuda")
    out = GuardedOutput(case.M, case.N, y_dtype)  # canaries on both sides of y
    try:
        tq2.matvec(x, qs, d, y=out.y, act_scale=case.s, status=st, impl=impl, out_scale=out_scale)
    except tq2.TQ2Error as e:
        if e.status == 5 and impl in (1, 4, 6, 7):
            return None  # that kernel does not take this shape
        raise
    T.cuda.synchronize()
    assert int(st.item()) == 0
    out.check(f"requant impl={impl} M={case.M} N={case.N} K={case.K}")
    return host(out.y)


@pytest.mark.parametrize("M,N,K", [
    (1, 32, 512), (1, 257, 4352), (2, 33, 1024), (1, 300, 4096), (2, 100, 8448),
    (3, 40, 512), (4, 100, 2048), (9, 20, 768), (16, 50, 16384),
])
@pytest.mark.parametrize("prologue", [False, True])
def test_requant_small_shapes(T, M, N, K, prologue):
    case = Case(seed=7 * M + N + K, M=M, N=N, K=K, heavy=prologue, prologue=prologue)
    y_ref, tol = case.reference()
    amax = float(np.abs(y_ref).max())
    for frac in (100.0, 300.0):  # codes up to ~100, and a third of them saturated
        s_o = float(np.float32(amax / frac))
        for name in _impls_for(M):
            for yd in (0, 1):
                y = _run(T, case, IMPLS[name], s_o, y_dtype=yd)
                if y is None:
                    continue
                check_requant(y, y_ref, tol, s_o, yd, f"{name} yd={yd} M={M} N={N} K={K} s_o=amax/{frac}")


def test_requant_saturates_and_zero_scale_is_plain(T):
    import quantized_gemv_tq2_gb300 as tq2
    case = Case(seed=3, M=1, N=64, K=1024)
    x, qs, d = case.device()
    y0 = host(tq2.matvec(x, qs, d))
    # out_scale 0 is the plain call, bit for bit
    assert np.array_equal(host(tq2.matvec(x, qs, d, out_scale=0.0)), y0)
    # a tiny scale saturates every nonzero result to the ends of the int8 range
    s = np.float32(1e-30)
    y = host(tq2.matvec(x, qs, d, out_scale=float(s)))
    expect = np.where(y0 > 0, np.float32(127) * s, np.where(y0 < 0, np.float32(-128) * s, np.float32(0)))
    assert np.array_equal(y, expect.astype(np.float32))


def test_requant_k_zero_stores_zero(T):
    import quantized_gemv_tq2_gb300 as tq2
    x = T.zeros((1, 0), dtype=T.float16, device="cuda")
    qs = T.zeros((8, 0), dtype=T.uint8, device="cuda")
    d = T.zeros((8, 0), dtype=T.float16, device="cuda")
    y = T.full((1, 8), 7.0, dtype=T.float32, device="cuda")
    tq2.matvec(x, qs, d, K=0, y=y, out_scale=0.25)
    T.cuda.synchronize()
    assert np.array_equal(host(y), np.zeros((1, 8), dtype=np.float32))


@pytest.mark.parametrize("N,K", [(16384, 4096), (4096, 16384)])
def test_requant_big_shapes_sampled(T, N, K):
    """The wNa8o8 path at the benchmark's big shapes, M = 1, prologue on,
    the launch configuration the benchmark times; sampled rows."""
    case = Case(seed=21, M=1, N=N, K=K, heavy=True, prologue=True)
    rows = sample_rows(N, 128, seed=5)
    y_ref, tol = case.reference(rows)
    s_o = float(np.float32(np.abs(y_ref).max() / 120.0))
    for yd in (0, 1):
        y = _run(T, case, 0, s_o, y_dtype=yd)
        check_requant(y[:, rows], y_ref, tol, s_o, yd, f"N={N} K={K} yd={yd}")
