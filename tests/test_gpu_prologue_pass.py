"""The static int8 prologue (gemma4 wNa8o8 page, "Implemented": x replaced by
s * clamp(rint(x / s), -128, 127) at a linear's input) run as a pass of its
own: given a workspace, a call whose kernel gains from it converts x once
into the workspace and the kernel reads the codes instead of converting x in
every CTA.  Checked against the CPU oracle:
  * the codes the pass leaves in the workspace are the oracle's fake-quant
    codes (the fp32 decision rint(x * (1/s)), ties to even, clamped to
    [-128, 127], NaN -> 0) bit for bit, on edge values: exact ties, +-0,
    the ends of the range and beyond, +-Inf, NaN;
  * y is the same bits as the same kernel converting x in each CTA, and
    within the oracle's tolerance: the tcgen05 GEMM (N > 512 or M > 64,
    ragged tiles, split K), the pre-scaled kernel at M >= 9 with K >= 8192,
    the automatic choice at M = 8 with down-sized K, fp32 and fp16 y, the
    output requantisation;
  * where the pass does not pay the workspace is left untouched; a
    workspace too small for the pass is TQ2_ERR_ARG with nothing written,
    a misaligned one TQ2_ERR_ALIGN;
  * one workspace reused by consecutive calls on a stream, and inside a
    CUDA graph, with different x."""
import numpy as np
import pytest

import oracle
from gpu_util import Case, assert_within_tolerance, check_requant, dev, host

pytestmark = pytest.mark.gpu

SENTINEL = 0x5A


@pytest.fixture(scope="module")
def T():
    import torch
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    import quantized_gemv_tq2_gb300 as tq2
    tq2.load()
    return torch


def _ws(T, nbytes, extra=256):
    buf = T.full((nbytes + extra,), SENTINEL, dtype=T.uint8, device="cuda")
    return buf


def _codes_in(ws, M, K):
    """The fp16 codes the pass wrote, as float64 [M, K]."""
    return host(ws[:2 * M * K].view(dtype=__import__("torch").float16)).astype(np.float64).reshape(M, K)


def _bits(t):
    import torch
    return host(t.view(torch.int32) if t.dtype == torch.float32 else t.view(torch.int16))


def _edge_x(M, K, s, seed):
    """Heavy random activations with edge values planted: exact ties at
    +-0.5, +-1.5, +-126.5, +-127.5, +-128.5 (s a power of two, so x / s is
    exact), +-0, beyond the range, +-Inf and NaN."""
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((M, K)) * 40.0 * s).astype(np.float16)
    t = np.array([0.5, -0.5, 1.5, -1.5, 2.5, -2.5, 126.5, -126.5, 127.5, -127.5, 128.5, -128.5,
                  127.0, -128.0, 129.0, -129.0, 1000.0, -1000.0, 0.0], dtype=np.float64)
    special = np.concatenate([(t * s).astype(np.float16),
                              np.array([-0.0, np.inf, -np.inf, np.nan], dtype=np.float16)])
    flat = x.reshape(-1)
    pos = rng.choice(flat.size, size=4 * special.size, replace=False)
    flat[pos] = np.tile(special, 4)
    return x


def test_pass_codes_are_the_oracles(T):
    """The GEMM (N > 512) with a workspace: its codes and y."""
    import quantized_gemv_tq2_gb300 as tq2
    M, N, K = 20, 600, 1024
    s = 2.0 ** -6
    case = Case(seed=31, M=M, N=N, K=K, prologue=True)
    case.x, case.s = _edge_x(M, K, s, 31), s
    x, qs, d = case.device()
    ws = _ws(T, 2 * M * K)
    st = T.zeros(1, dtype=T.int32, device="cuda")
    y = tq2.gemm(x, qs, d, act_scale=s, status=st, impl=1, workspace=ws)
    T.cuda.synchronize()
    assert int(st.item()) == 0
    want = oracle.fakequant_codes(case.x, s, mode=0).astype(np.float64)
    got = _codes_in(ws, M, K)
    assert np.array_equal(got, want), f"{int((got != want).sum())} codes differ"
    assert np.all(host(ws[2 * M * K:]) == SENTINEL)  # nothing past the codes
    y_ref, tol = case.reference()
    assert_within_tolerance(host(y), y_ref, tol, "gemm with the pass, edge x")
    y_f = tq2.gemm(x, qs, d, act_scale=s, impl=1, workspace=None)
    assert np.array_equal(_bits(y), _bits(y_f))


@pytest.mark.parametrize("M,N,K,impl,call", [
    (9, 700, 1024, 1, "gemm"),      # N > 512: ragged weight tile
    (17, 513, 768, 1, "gemm"),      # one row past 4 weight tiles, ragged activation tile
    (65, 100, 512, 1, "gemm"),      # M > 64: the pass pays even on one weight tile
    (20, 600, 256, 1, "gemm"),      # K = 256: one block, split K impossible
    (70, 16, 1024, 0, "gemm"),      # M > 64 on a 16-row matrix: 128-column tile, two MMA issuers
    (130, 257, 2048, 1, "gemm"),
    (300, 96, 4096, 0, "gemm"),
    (40, 1000, 8448, 1, "gemm"),    # K not a multiple of 512, split K
    (16, 600, 4096, 6, "matvec"),   # the GEMM through tq2_matvec_impl
    (9, 300, 8192, 4, "matvec"),    # the pre-scaled kernel at M >= 9, K >= 8192
    (16, 70, 8448, 4, "matvec"),
    (8, 640, 8192, 0, "matvec"),    # the automatic choice takes the GEMM, given the pass
    (12, 4096, 4096, 0, "matvec"),
])
def test_pass_equals_in_kernel_conversion(T, M, N, K, impl, call):
    # the kernel the call runs with the pass; without a workspace the
    # automatic choice at M = 8 would run the pre-scaled kernel instead
    same = 6 if (call, impl) == ("matvec", 0) else impl
    import quantized_gemv_tq2_gb300 as tq2
    case = Case(seed=M * 7 + N + K, M=M, N=N, K=K, heavy=True, prologue=True)
    x, qs, d = case.device()
    y_ref, tol = case.reference()
    s_o = float(np.float32(np.abs(y_ref).max() / 100.0))
    f = tq2.gemm if call == "gemm" else tq2.matvec
    for yd in (0, 1):
        for so in (0.0, s_o):
            ws = _ws(T, 2 * M * K)
            st = T.zeros(1, dtype=T.int32, device="cuda")
            kw = dict(act_scale=case.s, impl=impl, y_dtype=yd, out_scale=so)
            y_p = f(x, qs, d, status=st, workspace=ws, **kw)
            y_f = f(x, qs, d, workspace=None, **dict(kw, impl=same))
            T.cuda.synchronize()
            assert int(st.item()) == 0
            what = f"{call} impl={impl} M={M} N={N} K={K} yd={yd} so={so}"
            # the pass ran: the workspace holds the oracle's codes
            want = oracle.fakequant_codes(case.x, case.s, mode=0).astype(np.float64)
            assert np.array_equal(_codes_in(ws, M, K), want), what
            assert np.array_equal(_bits(y_p), _bits(y_f)), what
            if so == 0.0:
                assert_within_tolerance(host(y_p), y_ref, tol, what)
            else:
                check_requant(host(y_p), y_ref, tol, so, yd, what)


@pytest.mark.parametrize("M,N,K,impl", [
    (1, 4096, 4096, 0), (2, 16384, 4096, 1), (2, 256, 4096, 7), (6, 4096, 16384, 0), (8, 600, 4096, 4),
    (16, 256, 4096, 0), (16, 2048, 4096, 4), (12, 300, 2048, 2),
])
def test_workspace_untouched_where_the_pass_does_not_pay(T, M, N, K, impl):
    import quantized_gemv_tq2_gb300 as tq2
    case = Case(seed=M + N, M=M, N=N, K=K, heavy=True, prologue=True)
    x, qs, d = case.device()
    ws = _ws(T, 2 * M * K)
    y = tq2.matvec(x, qs, d, act_scale=case.s, impl=impl, workspace=ws)
    y_f = tq2.matvec(x, qs, d, act_scale=case.s, impl=impl, workspace=None)
    T.cuda.synchronize()
    assert np.all(host(ws) == SENTINEL)
    assert np.array_equal(_bits(y), _bits(y_f))
    rows = np.arange(0, N, max(1, N // 64))
    y_ref, tol = case.reference(rows)
    assert_within_tolerance(host(y)[:, rows], y_ref, tol, f"M={M} N={N} K={K} impl={impl}")


def test_workspace_errors(T):
    import quantized_gemv_tq2_gb300 as tq2
    M, N, K = 24, 1024, 2048
    case = Case(seed=2, M=M, N=N, K=K, prologue=True)
    x, qs, d = case.device()
    y = T.full((M, N), 7.0, dtype=T.float32, device="cuda")
    small = _ws(T, 2 * M * K - 16, extra=0)
    with pytest.raises(tq2.TQ2Error) as e:
        tq2.gemm(x, qs, d, y=y, act_scale=case.s, impl=1, workspace=small)
    assert e.value.status == 5
    # the automatic matvec choice at M = 8 with down-sized K runs the pass with the GEMM
    c8 = Case(seed=3, M=8, N=640, K=8192, prologue=True)
    x8, q8, d8 = c8.device()
    with pytest.raises(tq2.TQ2Error) as e:
        tq2.matvec(x8, q8, d8, act_scale=c8.s, workspace=_ws(T, 2 * 8 * 8192 - 16, extra=0))
    assert e.value.status == 5
    T.cuda.synchronize()
    assert np.all(host(y) == 7.0) and np.all(host(small) == SENTINEL)  # nothing was enqueued
    buf = _ws(T, 2 * M * K + 64)
    with pytest.raises(tq2.TQ2Error) as e:
        tq2.gemm(x, qs, d, y=y, act_scale=case.s, impl=1, workspace=buf[8:])
    assert e.value.status == 3
    # without the prologue a workspace is never used
    ws = _ws(T, 2 * M * K)
    tq2.gemm(x, qs, d, y=y, impl=1, workspace=ws)
    T.cuda.synchronize()
    assert np.all(host(ws) == SENTINEL)


def test_one_workspace_for_consecutive_calls_and_a_graph(T):
    """Each call's pass waits for the previous kernel on the stream before
    it writes the workspace, so consecutive calls may share it."""
    import quantized_gemv_tq2_gb300 as tq2
    M, N, K = 96, 768, 4096
    cases = [Case(seed=50 + i, M=M, N=N, K=K, heavy=True, prologue=True) for i in range(3)]
    W = cases[0].device()[1:]
    xs = [dev(c.x) for c in cases]
    ss = [c.s for c in cases]
    ws = _ws(T, 2 * M * K)
    ref = [tq2.gemm(xx, *W, act_scale=s, impl=1, workspace=None) for xx, s in zip(xs, ss)]
    stream = T.cuda.Stream()
    stream.wait_stream(T.cuda.current_stream())
    with T.cuda.stream(stream):
        ys = [tq2.gemm(xx, *W, act_scale=s, impl=1, workspace=ws) for xx, s in zip(xs, ss)]
        stream.synchronize()
        for a, b in zip(ys, ref):
            assert np.array_equal(_bits(a), _bits(b))
        outs = [T.empty(M, N, device="cuda") for _ in xs]
        g = T.cuda.CUDAGraph()
        with T.cuda.graph(g, stream=stream):
            for xx, s, yy in zip(xs, ss, outs):
                tq2.gemm(xx, *W, y=yy, act_scale=s, impl=1, workspace=ws)
        for _ in range(2):
            for yy in outs:
                yy.fill_(0.0)
            g.replay()
        stream.synchronize()
    for a, b in zip(outs, ref):
        assert np.array_equal(_bits(a), _bits(b))
    rows = np.arange(0, N, 13)
    for c, y in zip(cases, outs):  # every call used the first case's weights
        y_ref, tol = oracle.matvec_rows(c.x, cases[0].qs, cases[0].d, K, rows, c.s)
        assert_within_tolerance(host(y)[:, rows], y_ref, tol, "graph replay")
