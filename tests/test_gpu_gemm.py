"""GPU parity of tq2_gemm (any number of activation rows: prefill) against the
CPU oracle: element by element within |dy| <= 1e-3 * sum_k |d_b x'_k| + 1e-6,
bit-exact on one-hot x (every product and sum exact, with and without the
int8 prologue), ragged tiles in both dimensions, the prologue and the
requantisation at store on both paths (tcgen05 GEMM and 16-row slices),
determinism, and sampled rows at prefill-sized layer shapes."""
import numpy as np
import pytest

import oracle
import tq2_synth as syn
from gpu_util import Case, GuardedOutput, assert_within_tolerance, dev, host, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def T():
    import torch
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    import quantized_gemv_tq2_gb300 as tq2
    tq2.load()
    return torch


def _gemm(T, case, impl, y_dtype=0, out_scale=0.0, workspace="auto"):
    import quantized_gemv_tq2_gb300 as tq2
    x, qs, d = case.device()
    st = T.zeros(1, dtype=T.int32, device="cuda")
    out = GuardedOutput(case.M, case.N, y_dtype)  # canaries on both sides of y
    tq2.gemm(x, qs, d, y=out.y, act_scale=case.s, out_scale=out_scale, status=st, impl=impl, workspace=workspace)
    T.cuda.synchronize()
    assert int(st.item()) == 0
    out.check(f"gemm impl={impl} M={case.M} N={case.N} K={case.K}")
    return host(out.y).astype(np.float64)


@pytest.mark.parametrize("M,N,K", [
    (17, 128, 256),     # one k-block, a ragged activation tile
    (1, 64, 256),       # a single activation row through the GEMM
    (64, 100, 512),     # ragged weight tile
    (130, 257, 768),    # ragged in both, K not a multiple of 512
    (300, 300, 1024),
    (256, 128, 4096),
    (512, 96, 2048),
    (64, 256, 4096),    # 64-column tile (two A slots, two accumulators), K split over 8-CTA clusters
    (32, 512, 2048),    # 32-column tile, K split over 8 (one 256-block per CTA)
    (9, 640, 8448),     # 16-column tile, two accumulators, split K, K not a multiple of 512
])
def test_gemm_small_shapes(T, M, N, K):
    case = Case(seed=M + 3 * N + K, M=M, N=N, K=K)
    y_ref, tol = case.reference()
    for impl in (1, 0, 2):
        for yd in (0, 1):
            y = _gemm(T, case, impl, y_dtype=yd)
            assert_within_tolerance(y, y_ref, tol, f"impl={impl} yd={yd} M={M} N={N} K={K}")


def test_gemm_one_hot_is_exact(T):
    """x[m] = e_k for a k that walks every position of a 16-code k-step and
    both 8-value halves: y[m][n] = (q[n][k] - 1) * d[n][k // 256] exactly."""
    M, N, K = 160, 256, 1024
    case = Case(seed=5, M=M, N=N, K=K)
    ks = (np.arange(M) * 37 + 11) % K
    x = np.zeros((M, K), dtype=np.float16)
    x[np.arange(M), ks] = np.float16(1.0)
    case.x = x
    ye = oracle.matvec_exact(x, case.qs, case.d, K)
    direct = (case.codes[:, ks].T.astype(np.float64) - 1.0) * case.d[:, ks // 256].T.astype(np.float64)
    assert np.array_equal(ye, direct)  # the oracle agrees with the closed form
    for impl in (1, 2):
        y = _gemm(T, case, impl)
        assert np.array_equal(y, ye), f"impl={impl}: {int((y != ye).sum())} elements differ"


@pytest.mark.parametrize("M,N,K", [(40, 200, 2048), (130, 257, 768), (300, 128, 4096), (24, 1100, 1024)])
def test_gemm_prologue_and_requant(T, M, N, K):
    """The int8 prologue -- x fake-quantised in shared memory in every tile
    of the tcgen05 path (no workspace), or converted once by a pass of its
    own where that pays (a workspace: M > 64 or N > 512) -- and the
    requantisation at store, both paths; the two prologue plans give the
    same bits."""
    from test_gpu_requant import check_requant
    case = Case(seed=9 + M, M=M, N=N, K=K, heavy=True, prologue=True)
    y_ref, tol = case.reference()
    s_o = float(np.float32(np.abs(y_ref).max() / 100.0))
    for impl in (1, 0, 2):
        y = _gemm(T, case, impl)
        assert_within_tolerance(y, y_ref, tol, f"prologue impl={impl}")
        assert np.array_equal(y, _gemm(T, case, impl, workspace=None)), f"plans differ, impl={impl}"
        for yd in (0, 1):
            yq = _gemm(T, case, impl, y_dtype=yd, out_scale=s_o)
            check_requant(yq.astype(np.float32 if yd == 0 else np.float16), y_ref, tol, s_o, yd,
                          f"prologue+requant impl={impl} yd={yd}")


def test_gemm_prologue_one_hot_is_exact(T):
    """With the prologue, x' = s * code: one-hot x of value 3 s gives
    y = s * 3 * (q - 1) * d exactly (codes, products and the sum are exact)."""
    M, N, K = 64, 128, 512
    case = Case(seed=6, M=M, N=N, K=K, prologue=True)
    ks = (np.arange(M) * 53 + 5) % K
    x = np.zeros((M, K), dtype=np.float16)
    x[np.arange(M), ks] = np.float16(3.0 * case.s)
    case.x = x
    ye = oracle.matvec_exact(x, case.qs, case.d, K, case.s)
    y = _gemm(T, case, 1)
    assert np.array_equal(y.astype(np.float32), ye.astype(np.float32))


def test_gemm_is_deterministic(T):
    import quantized_gemv_tq2_gb300 as tq2
    case = Case(seed=4, M=200, N=384, K=4096)
    x, qs, d = case.device()
    a = host(tq2.gemm(x, qs, d, impl=1))
    b = host(tq2.gemm(x, qs, d, impl=1))
    assert np.array_equal(a, b)


@pytest.mark.parametrize("N,K", [(4096, 4096), (16384, 4096), (4096, 16384)])
def test_gemm_prefill_layer_shapes_sampled(T, N, K):
    """M = 512 activation rows (a prompt chunk) through a layer's shapes, in
    the launch configuration the benchmark times; sampled weight rows."""
    M = 512
    case = Case(seed=N + K, M=M, N=N, K=K)
    rows = sample_rows(N, 48, seed=3)
    y_ref, tol = case.reference(rows)
    y = _gemm(T, case, 0)
    assert_within_tolerance(y[:, rows], y_ref, tol, f"N={N} K={K}")
