"""tq2_gemm_static_ws: tq2_gemm whose prologue pass writes the library's
static device scratch instead of a caller's workspace.  On the GPU, two
calls in a row on one stream (different x, so the second overwrites the
first's codes in the shared scratch) give the same bits as tq2_gemm with a
workspace of its own, and match the oracle; the size limit (M * K <= 2^23
with the prologue) holds at its edge.  On the host, a call past the limit is
rejected before any CUDA call."""
import ctypes

import numpy as np
import pytest

import quantized_gemv_tq2_gb300 as tq2

P = ctypes.c_void_p
A16 = P(0x10000)


def test_static_ws_rejects_past_the_limit_on_the_host():
    L = tq2.load()
    # 4097 x 2048 activations: 2^23 + 2048 codes, one row past the scratch
    assert L.tq2_gemm_static_ws(A16, 4097, A16, A16, 32, 2048, A16, 0, 0.5, 0.0, P(0), P(0), 0) == 2
    assert L.tq2_gemm_static_ws(A16, 1 << 20, A16, A16, 32, 4096, A16, 0, 0.25, 0.0, P(0), P(0), 1) == 2
    # the other checks of tq2_gemm stand
    assert L.tq2_gemm_static_ws(A16, 64, A16, A16, 32, 300, A16, 0, 0.5, 0.0, P(0), P(0), 0) == 2
    assert L.tq2_gemm_static_ws(A16, 64, A16, A16, 32, 512, A16, 0, -1.0, 0.0, P(0), P(0), 0) == 5
    assert L.tq2_gemm_static_ws(P(0), 64, A16, A16, 32, 512, A16, 0, 0.0, 0.0, P(0), P(0), 0) == 1


@pytest.mark.gpu
@pytest.mark.parametrize("M,N,K,impl", [
    (40, 1000, 2048, 1),    # the pass runs (N > 512)
    (130, 257, 768, 0),     # the pass runs (M > 64), ragged tiles
    (16, 300, 4096, 0),     # 16-row slices: no pass at this shape, the scratch unused
    (2048, 640, 4096, 1),   # exactly 2^23 codes: the whole scratch
])
def test_static_ws_equals_tq2_gemm_two_calls_in_a_row(M, N, K, impl):
    import torch
    import oracle
    from gpu_util import Case, assert_within_tolerance, dev, host, sample_rows
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    cases = [Case(seed=M + N + K + i, M=M, N=N, K=K, heavy=True, prologue=True) for i in range(2)]
    _, qs, d = cases[0].device()
    xs = [dev(c.x) for c in cases]
    ys = [tq2.gemm_static_ws(x, qs, d, act_scale=c.s, impl=impl) for x, c in zip(xs, cases)]
    refs = [tq2.gemm(x, qs, d, act_scale=c.s, impl=impl,
                     workspace=torch.empty(tq2.gemm_workspace_size(M, N, K), dtype=torch.uint8, device="cuda"))
            for x, c in zip(xs, cases)]
    torch.cuda.synchronize()
    rows = sample_rows(N, 40, seed=M) if N > 512 else np.arange(N)
    for i, (c, y, r) in enumerate(zip(cases, ys, refs)):
        assert torch.equal(y.view(torch.int32), r.view(torch.int32)), f"call {i}"
        y_ref, tol = oracle.matvec_rows(c.x, cases[0].qs, cases[0].d, K, rows, c.s)
        assert_within_tolerance(host(y)[:, rows], y_ref, tol, f"static scratch call {i} M={M} N={N} K={K}")


@pytest.mark.gpu
def test_static_ws_past_the_limit_and_without_the_prologue():
    import torch
    from gpu_util import Case
    c = Case(seed=1, M=2049, N=64, K=4096, prologue=True)
    x, qs, d = c.device()
    with pytest.raises(tq2.TQ2Error) as e:
        tq2.gemm_static_ws(x, qs, d, act_scale=c.s)
    assert e.value.status == 2
    # without the prologue there is no scratch and no limit
    y = tq2.gemm_static_ws(x, qs, d)
    r = tq2.gemm(x, qs, d)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int32), r.view(torch.int32))
