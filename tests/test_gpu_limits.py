"""tq2_matvec at the edges of its shape range, against the CPU oracle: a long
K (65536: x no longer fits the tensor-core kernels' shared-memory staging
for two rows), a very tall N (200,000 rows: hundreds of rows per CTA), the
largest M (16) at the longest layer K, and each explicit kernel that takes
the shape either matching the oracle or refusing it with TQ2_ERR_ARG."""
import numpy as np
import pytest

import oracle
from gpu_util import Case, assert_within_tolerance, host, sample_rows

pytestmark = pytest.mark.gpu

IMPLS = {"auto": 0, "mma": 1, "simt": 2, "ps": 4, "gemm": 6, "smalln": 7}


@pytest.fixture(scope="module")
def T():
    import torch
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    import quantized_gemv_tq2_gb300 as tq2
    tq2.load()
    return torch


def _run(T, case, impl):
    import quantized_gemv_tq2_gb300 as tq2
    x, qs, d = case.device()
    st = T.zeros(1, dtype=T.int32, device="cuda")
    try:
        y = tq2.matvec(x, qs, d, act_scale=case.s, status=st, impl=impl)
    except tq2.TQ2Error as e:
        assert e.status == 5 and impl != 0, f"impl {impl}: {e}"
        return None  # that kernel does not take this shape
    T.cuda.synchronize()
    assert int(st.item()) == 0
    return host(y).astype(np.float64)


@pytest.mark.parametrize("M", [1, 2])
def test_long_k(T, M):
    case = Case(seed=31 + M, M=M, N=40, K=65536, heavy=True)
    y_ref, tol = case.reference()
    ran = 0
    for name, impl in IMPLS.items():
        y = _run(T, case, impl)
        if y is None:
            continue
        ran += 1
        assert_within_tolerance(y, y_ref, tol, f"{name} M={M} K=65536")
    assert ran >= 2


def test_tall_n_sampled(T):
    N, K = 200000, 256
    case = Case(seed=33, M=1, N=N, K=K)
    rows = sample_rows(N, 96, seed=4)
    y_ref, tol = case.reference(rows)
    for name in ("auto", "mma", "ps", "simt"):
        y = _run(T, case, IMPLS[name])
        if y is None:
            continue
        assert_within_tolerance(y[:, rows], y_ref, tol, f"{name} N={N}")


@pytest.mark.parametrize("prologue", [False, True])
def test_max_m_longest_layer_k(T, prologue):
    case = Case(seed=35, M=16, N=300, K=16384, heavy=prologue, prologue=prologue)
    y_ref, tol = case.reference()
    for name in ("auto", "ps", "gemm", "simt"):
        y = _run(T, case, IMPLS[name])
        if y is None:
            continue
        assert_within_tolerance(y, y_ref, tol, f"{name} M=16 K=16384 prologue={prologue}")
