"""GPU parity of tq2_matvec_grouped and tq2_matvec_grouped_requant (several
matrices sharing x) against the CPU oracle, per matrix: one launch of the
class-column kernel (M <= 2, any K) and of the pre-scaled kernel (M up to 16,
K = 4096 and longer), decoder layer shapes, odd sizes and the prologue; the
fallback to consecutive calls where a matrix would take the GEMM, with one
prologue pass for the whole group given a workspace; each matrix's own
output requantisation; guard bands around every y; and the back-to-back
graph configuration the benchmark times."""
import ctypes

import numpy as np
import pytest

import oracle
import tq2_synth as syn
from gpu_util import GuardedOutput, assert_within_tolerance, check_requant, dev, host, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def T():
    import torch
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    import quantized_gemv_tq2_gb300 as tq2
    tq2.load()
    return torch


def _mats(seed, Ns, K):
    out = []
    for j, N in enumerate(Ns):
        codes = syn.codes(seed, N, K, linear=j)
        qs, _ = oracle.pack(codes)
        d = syn.scales(seed, N, K // 256, linear=j)
        out.append((qs, d))
    return out


@pytest.mark.parametrize("M,K,Ns", [
    (1, 4096, (4096, 256, 256)),      # q, k, v: class-column kernel, one launch
    (1, 4096, (16384, 16384)),        # gate, up
    (2, 4096, (4096, 256, 256)),
    (1, 1024, (33, 1, 300)),
    (2, 256, (17, 17)),
    (1, 512, (5, 7, 11, 13)),         # four matrices
    (1, 8448, (50, 70)),              # K > 4096: 2-D boxes, one tensor map per matrix
    (2, 16384, (300, 41)),
    (3, 1024, (40, 24)),              # M > 2: pre-scaled kernel, one launch
    (4, 4096, (4096, 256, 256)),      # q, k, v at M = 4 (one 16-row group x 16 blocks per stage)
    (8, 4096, (16384, 16384)),        # gate, up at M = 8
    (16, 4096, (1000, 3000)),         # M >= 12, every N > 512: consecutive calls
    (10, 4096, (1000, 3000)),         # M = 9..11: one pre-scaled launch (two n-tiles)
    (5, 8448, (100, 60)),             # M > 2, K > 4096
    (12, 4096, (4096, 256, 256)),     # q/k/v at M = 12: one pre-scaled launch
    (13, 8448, (100, 600)),           # K >= 8192 at M >= 9: consecutive calls (the GEMM)
])
@pytest.mark.parametrize("prologue", [False, True])
@pytest.mark.parametrize("yd", [0, 1])
def test_grouped_matches_oracle(T, M, K, Ns, prologue, yd):
    import quantized_gemv_tq2_gb300 as tq2
    seed = 11 + M + K + len(Ns)
    x = syn.activations(seed, M, K, heavy=prologue)
    s = float(syn.act_scale(seed)) if prologue else 0.0
    mats = _mats(seed, Ns, K)
    st = T.zeros(1, dtype=T.int32, device="cuda")
    outs = [GuardedOutput(M, N, yd) for N in Ns]
    tq2.matvec_grouped(dev(x), [dev(q) for q, _ in mats], [dev(d) for _, d in mats], y_list=[o.y for o in outs],
                       act_scale=s, status=st)
    T.cuda.synchronize()
    assert int(st.item()) == 0
    for j, ((qs, d), out) in enumerate(zip(mats, outs)):
        N = Ns[j]
        out.check(f"matrix {j} N={N}")
        rows = sample_rows(N, 128, seed=j) if N > 2048 else np.arange(N)
        y_ref, tol = oracle.matvec_rows(x, qs, d, K, rows, act_scale=s)
        assert_within_tolerance(host(out.y)[:, rows].astype(np.float64), y_ref, tol, f"matrix {j} N={N}")


@pytest.mark.parametrize("M,K,Ns", [
    (1, 4096, (4096, 256, 256)),
    (2, 8448, (70, 50)),
    (4, 4096, (4096, 256, 256)),
    (8, 4096, (16384, 16384)),
    (12, 4096, (4096, 256, 256)),     # one pre-scaled launch at M = 12
    (14, 4096, (1000, 700)),          # consecutive calls, each with its own scale
])
@pytest.mark.parametrize("yd", [0, 1])
def test_grouped_requant_per_matrix(T, M, K, Ns, yd):
    """Each matrix's y is requantised with its own out_scale (0 for one of
    them: stored as computed), with and without the int8 prologue."""
    import quantized_gemv_tq2_gb300 as tq2
    for prologue in (False, True):
        seed = 70 + M + len(Ns) + int(prologue)
        x = syn.activations(seed, M, K, heavy=prologue)
        s = float(syn.act_scale(seed)) if prologue else 0.0
        mats = _mats(seed, Ns, K)
        scales = [0.37 * (j + 1) for j in range(len(Ns))]
        scales[-1] = 0.0
        st = T.zeros(1, dtype=T.int32, device="cuda")
        outs = [GuardedOutput(M, N, yd) for N in Ns]
        tq2.matvec_grouped(dev(x), [dev(q) for q, _ in mats], [dev(d) for _, d in mats],
                           y_list=[o.y for o in outs], act_scale=s, status=st, out_scales=scales)
        T.cuda.synchronize()
        assert int(st.item()) == 0
        for j, ((qs, d), out) in enumerate(zip(mats, outs)):
            N = Ns[j]
            out.check(f"requant matrix {j}")
            rows = sample_rows(N, 128, seed=j) if N > 2048 else np.arange(N)
            y_ref, tol = oracle.matvec_rows(x, qs, d, K, rows, act_scale=s)
            yg = host(out.y)[:, rows]
            what = f"M={M} matrix {j} N={N} s_o={scales[j]} prologue={prologue}"
            if scales[j] == 0.0:
                assert_within_tolerance(yg.astype(np.float64), y_ref, tol, what)
            else:
                check_requant(yg, y_ref, tol, scales[j], yd, what)


def test_grouped_prescaled_equals_single_calls(T):
    """One pre-scaled launch over q/k/v agrees with the single-matrix
    pre-scaled launches to fp32 rounding.  (The group's rows per CTA differ
    from a single call's, so the shared-memory plan, and with it whether x
    stays resident or is staged per K range, can differ; that changes the
    order of the fp32 block sums, not the result beyond rounding.)"""
    import quantized_gemv_tq2_gb300 as tq2
    K, Ns = 4096, (4096, 256, 256)
    for M in (3, 4, 8, 9, 12, 16):
        xh = syn.activations(M, M, K)
        x = dev(xh)
        mh = _mats(M, Ns, K)
        mats = [(dev(q), dev(d)) for q, d in mh]
        ys = tq2.matvec_grouped(x, [q for q, _ in mats], [d for _, d in mats])
        for (qh, dh), (q, d), y in zip(mh, mats, ys):
            single = tq2.matvec(x, q, d, impl=tq2.IMPL_PS)
            T.cuda.synchronize()
            rows = sample_rows(qh.shape[0], 256, seed=M)
            _, tol_sum = oracle.matvec_rows(xh, qh, dh, K, rows)
            diff = np.abs(host(y)[:, rows].astype(np.float64) - host(single)[:, rows].astype(np.float64))
            # reordered fp32 sums: a few units of 2^-24 of sum |d_b x_k|, far below the parity bound
            assert np.all(diff <= 1e-6 * tol_sum + 1e-7), (M, float((diff / (tol_sum + 1e-30)).max()))


def test_grouped_equals_single_calls(T):
    """The grouped launch computes each row like the single-matrix launch of
    the same kernel (impl 1; automatic dispatch may pick the small-N kernel
    for the k/v shapes, whose summation order differs)."""
    import quantized_gemv_tq2_gb300 as tq2
    K, Ns = 4096, (4096, 256, 256)
    x = dev(syn.activations(3, 1, K))
    mats = [(dev(q), dev(d)) for q, d in _mats(3, Ns, K)]
    ys = tq2.matvec_grouped(x, [q for q, _ in mats], [d for _, d in mats])
    for (q, d), y in zip(mats, ys):
        single = tq2.matvec(x, q, d, impl=tq2.IMPL_MMA)
        T.cuda.synchronize()
        assert np.allclose(host(y), host(single), rtol=1e-6, atol=1e-6)


def test_grouped_zero_rows_and_graph(T):
    """A matrix with N = 0 is skipped; grouped calls replay back to back in a
    CUDA graph (programmatic dependent launches between them)."""
    import quantized_gemv_tq2_gb300 as tq2
    K = 4096
    groups = [(4096, 256, 256), (16384, 16384)]
    data = []
    for gi, Ns in enumerate(groups):
        x = syn.activations(40 + gi, 1, K)
        mats = _mats(40 + gi, Ns, K)
        data.append((x, mats, [dev(q) for q, _ in mats], [dev(d) for _, d in mats],
                     [T.empty((1, N), dtype=T.float32, device="cuda") for N in Ns]))
    s = T.cuda.Stream()
    with T.cuda.stream(s):
        for x, _, qd, dd, ys in data:
            tq2.matvec_grouped(dev(x), qd, dd, y_list=ys)
        xs = [dev(x) for x, *_ in data]
        s.synchronize()
        g = T.cuda.CUDAGraph()
        with T.cuda.graph(g, stream=s):
            for xdev, (_, _, qd, dd, ys) in zip(xs, data):
                tq2.matvec_grouped(xdev, qd, dd, y_list=ys)
        for y in [y for *_, ys in data for y in ys]:
            y.zero_()
        for _ in range(3):
            g.replay()
    s.synchronize()
    for x, mats, _, _, ys in data:
        for (qs, d), y in zip(mats, ys):
            rows = sample_rows(qs.shape[0], 64)
            y_ref, tol = oracle.matvec_rows(x, qs, d, K, rows)
            assert_within_tolerance(host(y)[:, rows].astype(np.float64), y_ref, tol, "graph")
    # N = 0 in the middle of a group
    x = dev(syn.activations(5, 1, 512))
    mats = _mats(5, (8, 8), 512)
    empty_q = T.zeros((0, 128), dtype=T.uint8, device="cuda")
    empty_d = T.zeros((0, 2), dtype=T.float16, device="cuda")
    ys = tq2.matvec_grouped(x, [dev(mats[0][0]), empty_q, dev(mats[1][0])],
                            [dev(mats[0][1]), empty_d, dev(mats[1][1])])
    T.cuda.synchronize()
    assert ys[1].shape == (1, 0)
    for j, (qs, d) in ((0, mats[0]), (2, mats[1])):
        y_ref, tol = oracle.matvec(host(x), qs, d, 512)
        assert_within_tolerance(host(ys[j]).astype(np.float64), y_ref, tol, f"zero-row group {j}")


@pytest.mark.parametrize("M,K,Ns", [
    (13, 4096, (2048, 1024)),         # consecutive calls (the GEMM each)
    (16, 4096, (1000, 3000)),
    (12, 8448, (600, 70, 70)),        # GEMM for q, k and v
    (8, 8448, (640, 300)),            # M = 8: a matrix takes the GEMM given the pass
])
@pytest.mark.parametrize("requant", [False, True])
def test_grouped_one_prologue_pass(T, M, K, Ns, requant):
    """With the prologue and a workspace, a group run as consecutive calls
    converts x once: the workspace then holds the oracle's codes, and each
    matrix's y is the same bits as its single call (with a workspace of its
    own) and as the group without a workspace where that runs the same
    kernel; all within the oracle's tolerance."""
    import quantized_gemv_tq2_gb300 as tq2
    seed = 90 + M + K + len(Ns)
    xh = syn.activations(seed, M, K, heavy=True)
    s = float(syn.act_scale(seed))
    mh = _mats(seed, Ns, K)
    x = dev(xh)
    mats = [(dev(q), dev(d)) for q, d in mh]
    scales = [0.21 * (j + 1) for j in range(len(Ns))] if requant else None
    wsz = tq2.load().tq2_matvec_grouped_workspace_size(
        M, K, len(Ns), ctypes.cast((ctypes.c_int64 * len(Ns))(*Ns), ctypes.c_void_p))
    assert wsz == 2 * M * K
    ws = T.full((wsz + 256,), 0x5A, dtype=T.uint8, device="cuda")
    st = T.zeros(1, dtype=T.int32, device="cuda")
    ys = tq2.matvec_grouped(x, [q for q, _ in mats], [d for _, d in mats], act_scale=s, status=st,
                            out_scales=scales, workspace=ws)
    singles = [tq2.matvec(x, q, d, act_scale=s, out_scale=(scales[j] if scales else 0.0),
                          workspace=T.empty(2 * M * K, dtype=T.uint8, device="cuda"))
               for j, (q, d) in enumerate(mats)]
    T.cuda.synchronize()
    assert int(st.item()) == 0
    codes = host(ws[:2 * M * K].view(T.float16)).astype(np.float64).reshape(M, K)
    assert np.array_equal(codes, oracle.fakequant_codes(xh, s, mode=0).astype(np.float64))
    assert np.all(host(ws[2 * M * K:]) == 0x5A)
    for j, ((qh, dh), y, y1) in enumerate(zip(mh, ys, singles)):
        what = f"M={M} K={K} matrix {j} N={Ns[j]} requant={requant}"
        assert np.array_equal(host(y).view(np.int32), host(y1).view(np.int32)), what
        rows = sample_rows(Ns[j], 96, seed=j) if Ns[j] > 2048 else np.arange(Ns[j])
        y_ref, tol = oracle.matvec_rows(xh, qh, dh, K, rows, act_scale=s)
        if requant:
            check_requant(host(y)[:, rows], y_ref, tol, scales[j], 0, what)
        else:
            assert_within_tolerance(host(y)[:, rows].astype(np.float64), y_ref, tol, what)
    if M >= 9:  # without a workspace the same kernels run, each converting x itself
        ys0 = tq2.matvec_grouped(x, [q for q, _ in mats], [d for _, d in mats], act_scale=s,
                                 out_scales=scales, workspace=None)
        T.cuda.synchronize()
        for j, (y, y0) in enumerate(zip(ys, ys0)):
            assert np.array_equal(host(y).view(np.int32), host(y0).view(np.int32)), f"no workspace, matrix {j}"


def test_grouped_workspace_too_small(T):
    import quantized_gemv_tq2_gb300 as tq2
    M, K, Ns = 12, 4096, (600, 700)
    mats = [(dev(q), dev(d)) for q, d in _mats(5, Ns, K)]
    x = dev(syn.activations(5, M, K))
    ys = [T.full((M, N), 3.0, device="cuda") for N in Ns]
    with pytest.raises(tq2.TQ2Error) as e:
        tq2.matvec_grouped(x, [q for q, _ in mats], [d for _, d in mats], y_list=ys, act_scale=0.05,
                           workspace=T.empty(2 * M * K - 16, dtype=T.uint8, device="cuda"))
    assert e.value.status == 5
    T.cuda.synchronize()
    assert all(np.all(host(y) == 3.0) for y in ys)  # nothing was enqueued
