"""GPU parity of tq2_affine4_matvec (the affine-int4 sibling: W = s (q - z)
per group of G codes, zero point factored out) against the CPU oracle,
element by element within |dy| <= 1e-3 * sum_g |s_g| sum_k |x_k| (q_k + |z_g|)
+ 1e-6; one-hot x exact to one fp32 rounding; ragged rows and K chunks,
every group size, M up to 16, both y dtypes, determinism, and sampled rows
at layer shapes in the launch configuration the benchmark times."""
import numpy as np
import pytest

import oracle
import tq2_synth as syn
from gpu_util import GuardedOutput, assert_within_tolerance, dev, host, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def T():
    import torch
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    import quantized_gemv_tq2_gb300 as tq2
    tq2.load()
    return torch


def _case(seed, M, N, K, G, heavy=False):
    qs, s, z = syn.affine4_weights(seed, N, K, G)
    x = syn.activations(seed, M, K, heavy=heavy)
    return x, qs, s, z


def _run(T, x, qs, s, z, G, y_dtype=0):
    import quantized_gemv_tq2_gb300 as tq2
    st = T.zeros(1, dtype=T.int32, device="cuda")
    out = GuardedOutput(x.shape[0], qs.shape[0], y_dtype)  # canaries on both sides of y
    tq2.affine4_matvec(dev(x), dev(qs), dev(s), dev(z), G, y=out.y, status=st)
    T.cuda.synchronize()
    assert int(st.item()) == 0
    out.check(f"affine4 M={x.shape[0]} N={qs.shape[0]} K={x.shape[1]} G={G}")
    return host(out.y)


@pytest.mark.parametrize("M,N,K,G", [
    (1, 1, 256, 256), (1, 16, 256, 64), (1, 17, 512, 128), (2, 33, 768, 64),
    (1, 100, 2048, 128), (2, 257, 2304, 256), (1, 300, 4096, 64), (2, 40, 4352, 128),
    (3, 50, 1024, 64), (5, 19, 2560, 256), (16, 70, 1280, 128), (1, 24, 16384, 64),
])
@pytest.mark.parametrize("heavy", [False, True])
def test_affine4_small_shapes(T, M, N, K, G, heavy):
    x, qs, s, z = _case(M * 1000 + N + K + G, M, N, K, G, heavy)
    y_ref, tol = oracle.affine4(x, qs, s, z, K, G)
    for yd in (0, 1):
        y = _run(T, x, qs, s, z, G, y_dtype=yd)
        assert_within_tolerance(y.astype(np.float64), y_ref, tol, f"yd={yd} M={M} N={N} K={K} G={G}")


@pytest.mark.parametrize("G", [64, 128, 256])
def test_affine4_one_hot_is_exact(T, G):
    """x = e_k: y[n] = s (q - z), which the kernel forms as one fused
    multiply-add of exact products, so it equals fp32(s (q - z)) exactly.
    k walks both nibbles of a byte, every word of a 64-code slice and group
    and chunk boundaries."""
    N, K = 40, 4096
    _, qs, s, z = _case(11, 1, N, K, G)
    ks = [0, 1, 2, 7, 8, 15, 16, 63, 64, 127, 128, 255, 256, 2047, 2048, 4095]
    x = np.zeros((len(ks), K), dtype=np.float16)
    x[np.arange(len(ks)), ks] = 1.0
    exact = oracle.affine4_exact(x, qs, s, z, K, G)
    for i in range(0, len(ks), 2):  # two activation rows per launch, M = 2
        y = _run(T, x[i:i + 2], qs, s, z, G)
        assert np.array_equal(y, exact[i:i + 2].astype(np.float32)), ks[i:i + 2]


def test_affine4_integer_zero_point_equal_codes_cancel(T):
    """Every code equal to an integer zero point: W = 0, so y = 0 (the
    oracle's value, exact).  The factored form subtracts two fp32 sums, dot
    and z * sum x, rounded separately: the kernel lands within the tolerance
    of 0, not on it."""
    N, K, G = 48, 2048, 128
    x = syn.activations(3, 2, K, heavy=True)
    v = np.arange(N) % 16
    qs = np.repeat((v | (v << 4)).astype(np.uint8)[:, None], K // 2, axis=1)
    s = syn.scales(3, N, K // G)
    z = np.repeat(v.astype(np.float16)[:, None], K // G, axis=1)
    y_ref, tol = oracle.affine4(x, qs, s, z, K, G)
    assert np.all(y_ref == 0.0)
    y = _run(T, x, qs, s, z, G)
    assert_within_tolerance(y.astype(np.float64), y_ref, tol, "codes == zero point")


def test_affine4_is_deterministic(T):
    x, qs, s, z = _case(4, 2, 1000, 4096, 64, heavy=True)
    a = _run(T, x, qs, s, z, 64)
    b = _run(T, x, qs, s, z, 64)
    assert np.array_equal(a, b)


def test_affine4_k_zero_and_empty(T):
    import quantized_gemv_tq2_gb300 as tq2
    x = T.zeros((2, 0), dtype=T.float16, device="cuda")
    qs = T.zeros((8, 0), dtype=T.uint8, device="cuda")
    s = T.zeros((8, 0), dtype=T.float16, device="cuda")
    y = T.full((2, 8), 7.0, dtype=T.float32, device="cuda")
    tq2.affine4_matvec(x, qs, s, s, 64, y=y)
    T.cuda.synchronize()
    assert np.array_equal(host(y), np.zeros((2, 8), dtype=np.float32))


@pytest.mark.parametrize("N,K,G", [(16384, 4096, 128), (4096, 16384, 128), (4096, 4096, 64),
                                   (4096, 4096, 256)])
def test_affine4_layer_shapes_sampled(T, N, K, G):
    """M = 1 at a decoder layer's shapes, the launch configuration the
    benchmark times; sampled rows against the oracle."""
    x, qs, s, z = _case(N + K + G, 1, N, K, G)
    rows = sample_rows(N, 64, seed=2)
    y_ref, tol = oracle.affine4_rows(x, qs, s, z, K, G, rows)
    y = _run(T, x, qs, s, z, G)
    assert_within_tolerance(y[:, rows].astype(np.float64), y_ref, tol, f"N={N} K={K} G={G}")


def test_affine4_long_k(T):
    """K = 32768 (128 blocks of x staged per CTA; two activation rows need
    the one-CTA-per-SM plan): full compare against the oracle."""
    x, qs, s, z = _case(21, 2, 40, 32768, 256, heavy=True)
    y_ref, tol = oracle.affine4(x, qs, s, z, 32768, 256)
    y = _run(T, x, qs, s, z, 256)
    assert_within_tolerance(y.astype(np.float64), y_ref, tol, "K=32768")


def test_affine4_k_too_long_is_an_argument_error(T):
    """x of two rows at K = 131072 cannot be staged in shared memory: the
    call returns TQ2_ERR_ARG before launching anything."""
    import quantized_gemv_tq2_gb300 as tq2
    K, N = 131072, 16
    x = T.zeros((2, K), dtype=T.float16, device="cuda")
    qs = T.zeros((N, K // 2), dtype=T.uint8, device="cuda")
    s = T.zeros((N, K // 64), dtype=T.float16, device="cuda")
    with pytest.raises(tq2.TQ2Error) as e:
        tq2.affine4_matvec(x, qs, s, s, 64)
    assert e.value.status == 5
