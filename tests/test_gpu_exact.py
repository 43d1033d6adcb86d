"""Exact parity at the full MiniCPM4-8B shapes.

Inputs are chosen so that every partial sum the product can form is an exact
fp32 value: x is an integer in [-2, 2] times 2^-2 and every block scale is a
power of two in [2^-4, 1], so each term d_b x_k (q_k - 1) is a multiple of
2^-6 and every sum of them stays below 2^13 (2^19 units, well inside fp32's
24 bits), whatever the order of summation.  Any correct kernel must then
reproduce the oracle's exact result (integer accumulation, one rounding) bit
for bit, on every element: a single mis-indexed code, scale or x value, or a
dropped term, changes some output.  This covers the full software-pipelined
K = 4096 stage loop and the 16-row boxes of every CTA (q/o, gate/up), the
4096-code chunks of K = 16384 (down) with its partial 2-D boxes, the pre-scaled small-M kernel
and the tcgen05 GEMM, with the output surrounded by guard bands that must
stay untouched.
"""
import numpy as np
import pytest

import oracle
import tq2_synth as syn
from gpu_util import GuardedOutput, dev, host

pytestmark = pytest.mark.gpu

SHAPES = {"qo": (4096, 4096), "gateup": (16384, 4096), "down": (4096, 16384)}
_cache = {}


@pytest.fixture(scope="module")
def T():
    import torch
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    import quantized_gemv_tq2_gb300 as tq2
    tq2.load()
    return torch


def _case(name, M):
    key = (name, M)
    if key not in _cache:
        N, K = SHAPES[name]
        codes = syn.codes(31, N, K, linear=len(_cache))
        qs, flags = oracle.pack(codes)
        assert flags == 0
        d = syn.pow2_scales(31, N, K // 256, linear=len(_cache))
        x = syn.small_int_activations(31, M, K, linear=len(_cache))
        y = oracle.matvec_exact(x, qs, d, K)
        if M <= 2:  # exact-sum inputs: the fp64 oracle agrees exactly too
            y64, _ = oracle.matvec(x, qs, d, K)
            assert np.array_equal(y, y64)
        _cache[key] = (x, qs, d, y)
    return _cache[key]


@pytest.mark.parametrize("shape", list(SHAPES))
@pytest.mark.parametrize("M,impl", [(1, 0), (2, 0), (1, 1), (2, 1), (4, 4), (8, 4), (16, 4), (8, 0), (16, 0), (16, 6)])
def test_exact_full_shape(T, shape, M, impl):
    import quantized_gemv_tq2_gb300 as tq2
    x, qs, d, y_exact = _case(shape, M)
    N, K = SHAPES[shape]
    xd, qd, dd = dev(x), dev(qs), dev(d)
    for yd in (0, 1):
        out = GuardedOutput(M, N, yd)
        st = T.zeros(1, dtype=T.int32, device="cuda")
        tq2.matvec(xd, qd, dd, y=out.y, status=st, impl=impl)
        T.cuda.synchronize()
        assert int(st.item()) == 0
        out.check(f"{shape} M={M} impl={impl} yd={yd}")
        got = host(out.y).astype(np.float64)
        want = y_exact if yd == 0 else y_exact.astype(np.float16).astype(np.float64)
        bad = got != want
        assert not bad.any(), (f"{shape} M={M} impl={impl} yd={yd}: {int(bad.sum())} of {bad.size} differ; "
                               f"first at {tuple(np.argwhere(bad)[0])}")


@pytest.mark.parametrize("shape", ["gateup", "down"])
def test_exact_back_to_back_graph(T, shape):
    """The benchmark's launch configuration: calls captured in a CUDA graph
    with programmatic dependent launches between them, replayed; the
    outputs of distinct weight sets must all be exact."""
    import quantized_gemv_tq2_gb300 as tq2
    N, K = SHAPES[shape]
    sets = []
    for j in range(3):
        codes = syn.codes(40 + j, N, K)
        qs, _ = oracle.pack(codes)
        d = syn.pow2_scales(40 + j, N, K // 256)
        x = syn.small_int_activations(40 + j, 1, K)
        sets.append((dev(x), dev(qs), dev(d), oracle.matvec_exact(x, qs, d, K)))
    ys = [T.empty((1, N), dtype=T.float32, device="cuda") for _ in sets]
    s = T.cuda.Stream()
    with T.cuda.stream(s):
        for (x, qs, d, _), y in zip(sets, ys):
            tq2.matvec(x, qs, d, y=y)
        s.synchronize()
        for y in ys:
            y.fill_(float("nan"))
        g = T.cuda.CUDAGraph()
        with T.cuda.graph(g, stream=s):
            for (x, qs, d, _), y in zip(sets, ys):
                tq2.matvec(x, qs, d, y=y)
        for _ in range(3):
            g.replay()
    s.synchronize()
    for (_, _, _, want), y in zip(sets, ys):
        assert np.array_equal(host(y).astype(np.float64), want)
