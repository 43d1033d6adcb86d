"""The bounded-wait timeout path of the class-column kernel (impl 1), made to
run without faulting anything: the test hook tq2_test_matvec_stall skips the
weight copy of one pipeline stage in every CTA and shortens every device wait
to a few milliseconds, so the consumers' wait for that stage runs out.  The
kernel must report TQ2_FLAG_TIMEOUT, drain the copies it did issue, leave y
unwritten, and leave the context usable: the next ordinary call on the same
stream is correct."""
import numpy as np
import pytest

from gpu_util import Case, GuardedOutput, assert_within_tolerance, dev, host, sample_rows

pytestmark = pytest.mark.gpu

TQ2_FLAG_TIMEOUT = 8
LIMIT_US = 2000


@pytest.fixture(scope="module")
def T():
    import torch
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    import quantized_gemv_tq2_gb300 as tq2
    tq2.load()
    return torch


# (M, N, K, stall stages): K = 4096 runs the one-stage-per-row-group path,
# K = 16384 the general path over 4096-code chunks with 2-D tensor boxes.
@pytest.mark.parametrize("M,N,K,stages", [
    (1, 16384, 4096, (0, 1, 2)),
    (2, 16384, 4096, (0, 1)),
    (1, 4096, 16384, (0, 1, 3, 5)),
    (2, 4096, 16384, (0, 2)),
])
def test_stall_reports_timeout_then_recovers(T, M, N, K, stages):
    import quantized_gemv_tq2_gb300 as tq2
    case = Case(seed=7000 + M * 100 + K // 256, M=M, N=N, K=K)
    x, qs, d = case.device()
    rows = sample_rows(N, 64, seed=M)
    y_ref, tol = case.reference(rows)
    for stall in stages:
        st = T.zeros(1, dtype=T.int32, device="cuda")
        out = GuardedOutput(M, N)
        tq2.test_matvec_stall(x, qs, d, st, stall_stage=stall, wait_limit_us=LIMIT_US, y=out.y)
        T.cuda.synchronize()  # raises if the context was lost
        assert int(st.item()) & TQ2_FLAG_TIMEOUT, f"stage {stall}: no timeout reported"
        out.check(f"stall {stall}")
        if stall == 0:  # every CTA has a stage 0: no CTA may have stored y
            assert bool(T.all(out.y.view(T.int32) == out.canary)), "y written after a timeout"
        # the same stream, the ordinary kernel: correct, no flag
        st2 = T.zeros(1, dtype=T.int32, device="cuda")
        y = tq2.matvec(x, qs, d, status=st2, impl=1)
        T.cuda.synchronize()
        assert int(st2.item()) == 0
        assert_within_tolerance(host(y).astype(np.float64)[:, rows], y_ref, tol,
                                f"M={M} {N}x{K} after stall {stall}")


def test_stall_past_last_stage_is_ordinary(T):
    """A stall stage no CTA reaches skips nothing: no flag, a correct y."""
    import quantized_gemv_tq2_gb300 as tq2
    M, N, K = 1, 4096, 4096
    case = Case(seed=7100, M=M, N=N, K=K)
    x, qs, d = case.device()
    y_ref, tol = case.reference()
    st = T.zeros(1, dtype=T.int32, device="cuda")
    y = tq2.test_matvec_stall(x, qs, d, st, stall_stage=1 << 30, wait_limit_us=LIMIT_US)
    T.cuda.synchronize()
    assert int(st.item()) == 0
    assert_within_tolerance(host(y).astype(np.float64), y_ref, tol, "stall past the end")


def test_stall_argument_checks(T):
    import quantized_gemv_tq2_gb300 as tq2
    case = Case(seed=7200, M=1, N=64, K=512)
    x, qs, d = case.device()
    st = T.zeros(1, dtype=T.int32, device="cuda")
    for kw in (dict(stall_stage=-1, wait_limit_us=100), dict(stall_stage=0, wait_limit_us=0),
               dict(stall_stage=0, wait_limit_us=200001)):
        with pytest.raises(tq2.TQ2Error) as e:
            tq2.test_matvec_stall(x, qs, d, st, **kw)
        assert e.value.status == 5
    with pytest.raises(tq2.TQ2Error) as e:
        tq2.test_matvec_stall(dev(case.x).view(1, -1).repeat(3, 1), qs, d, st, stall_stage=0,
                              wait_limit_us=100)
    assert e.value.status == 5  # M = 3: impl 1 takes M <= 2


# The tcgen05 GEMM: (M, N, K, stall stages) with the CTA's x stages counted
# within its share of K -- one CTA per 128-row tile and all of K (160 tiles:
# more than two CTAs per SM hold, so no split; 8 stages), K split over CTA
# pairs (two CTAs per SM for a 16-row activation tile; 4 stages each), split
# K over clusters of 8 CTAs (the partial-sum hand-off; 4 stages each), and
# two activation tiles over clusters of 4 (2 stages each).
@pytest.mark.parametrize("M,N,K,stages", [
    (16, 20480, 1024, (0, 1, 7)),
    (16, 16384, 1024, (0, 1, 3)),
    (16, 512, 4096, (0, 1, 3)),
    (200, 2048, 1024, (0, 1)),
])
@pytest.mark.parametrize("prologue", [False, True])
def test_gemm_stall_reports_timeout_then_recovers(T, M, N, K, stages, prologue):
    import quantized_gemv_tq2_gb300 as tq2
    case = Case(seed=7300 + M + K // 256, M=M, N=N, K=K, heavy=prologue, prologue=prologue)
    x, qs, d = case.device()
    rows = sample_rows(N, 64, seed=M)
    y_ref, tol = case.reference(rows)
    for stall in stages:
        st = T.zeros(1, dtype=T.int32, device="cuda")
        out = GuardedOutput(M, N)
        tq2.test_gemm_stall(x, qs, d, st, stall_stage=stall, wait_limit_us=LIMIT_US, act_scale=case.s, y=out.y)
        T.cuda.synchronize()  # raises if the context was lost
        assert int(st.item()) & TQ2_FLAG_TIMEOUT, f"stage {stall}: no timeout reported"
        out.check(f"gemm stall {stall}")
        if stall == 0:  # every CTA has a stage 0: no CTA may have stored y
            assert bool(T.all(out.y.view(T.int32) == out.canary)), "y written after a timeout"
        st2 = T.zeros(1, dtype=T.int32, device="cuda")
        y = tq2.gemm(x, qs, d, act_scale=case.s, status=st2, impl=1)
        T.cuda.synchronize()
        assert int(st2.item()) == 0
        assert_within_tolerance(host(y).astype(np.float64)[:, rows], y_ref, tol,
                                f"gemm M={M} {N}x{K} after stall {stall}")
