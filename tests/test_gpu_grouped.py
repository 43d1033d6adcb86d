"""GPU parity of tq2_matvec_grouped (several matrices sharing x) against the
CPU oracle, per matrix: the one-launch path (M <= 2, K <= 4096) with decoder
layer shapes, odd sizes and the prologue; the fallback path (M > 2 or
K > 4096); and the back-to-back graph configuration the benchmark times."""
import numpy as np
import pytest

import oracle
import tq2_synth as syn
from gpu_util import assert_within_tolerance, dev, host, sample_rows

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
    (1, 4096, (4096, 256, 256)),      # q, k, v
    (1, 4096, (16384, 16384)),        # gate, up
    (2, 4096, (4096, 256, 256)),
    (1, 1024, (33, 1, 300)),
    (2, 256, (17, 17)),
    (1, 512, (5, 7, 11, 13)),         # four matrices
    (3, 1024, (40, 24)),              # M > 2: consecutive calls
    (1, 8448, (50, 70)),              # K > 4096: consecutive calls
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
    ys = tq2.matvec_grouped(dev(x), [dev(q) for q, _ in mats], [dev(d) for _, d in mats], y_dtype=yd,
                            act_scale=s, status=st)
    T.cuda.synchronize()
    assert int(st.item()) == 0
    for j, ((qs, d), y) in enumerate(zip(mats, ys)):
        N = Ns[j]
        rows = sample_rows(N, 128, seed=j) if N > 2048 else np.arange(N)
        y_ref, tol = oracle.matvec_rows(x, qs, d, K, rows, act_scale=s)
        assert_within_tolerance(host(y)[:, rows].astype(np.float64), y_ref, tol, f"matrix {j} N={N}")


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
