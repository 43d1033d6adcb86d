"""Sweep run by tests/test_gpu_bounds.py in a child process whose environment
selects the bounds-checked debug library (TQ2_BOUNDS_CHECK=1): every call
must leave the status word clear (no TQ2_FLAG_BOUNDS: no kernel computed an
index outside its buffer) and match the CPU oracle within the parity
tolerance.  Prints one line per group of cases; exits non-zero on the first
failure."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

import torch  # noqa: E402

import oracle  # noqa: E402
import quantized_gemv_tq2_gb300 as tq2  # noqa: E402
import tq2_synth as syn  # noqa: E402
from gpu_util import assert_within_tolerance, dev, host, sample_rows  # noqa: E402

IMPL_FOR = {1: (0, 1, 2, 4, 7), 2: (0, 1, 2, 4, 7)}  # M <= 2; larger M: 0, 2, 4


def run(x, qs, d, K, impl, M, N, st):
    try:
        y = tq2.matvec(x, qs, d, K=K, status=st, impl=impl)
    except tq2.TQ2Error as e:
        if e.status == 5 and impl != 0:
            return None  # this kernel does not take the shape
        raise
    return y


def check_status(st, what):
    torch.cuda.synchronize()
    v = int(st.item())
    assert v == 0, f"{what}: status {v:#x} (bounds flag {bool(v & tq2.FLAG_BOUNDS)})"


def tiny_sweep():
    n_calls = 0
    for K in (256, 512, 768):
        for N in range(1, 71):
            seed = 100 * K + N
            codes = syn.codes(seed, N, K)
            qs_h, _ = oracle.pack(codes)
            d_h = syn.scales(seed, N, K // 256)
            x_all = syn.activations(seed, 16, K)
            qs, d = dev(qs_h), dev(d_h)
            for M in range(1, 17):
                x_h = x_all[:M]
                y_ref, tol = oracle.matvec(x_h, qs_h, d_h, K)
                x = dev(x_h)
                for impl in IMPL_FOR.get(M, (0, 2, 4)):
                    st = torch.zeros(1, dtype=torch.int32, device="cuda")
                    y = run(x, qs, d, K, impl, M, N, st)
                    if y is None:
                        continue
                    check_status(st, f"K={K} N={N} M={M} impl={impl}")
                    assert_within_tolerance(host(y).astype(np.float64), y_ref, tol, f"K={K} N={N} M={M} impl={impl}")
                    n_calls += 1
        print(f"tiny sweep K={K}: clear, parity green ({n_calls} calls so far)", flush=True)


def layer_shapes():
    for name, N, K in (("q/o", 4096, 4096), ("k/v", 256, 4096), ("gate/up", 16384, 4096), ("down", 4096, 16384)):
        codes = syn.codes(7, N, K)
        qs_h, _ = oracle.pack(codes)
        d_h = syn.scales(7, N, K // 256)
        qs, d = dev(qs_h), dev(d_h)
        rows = sample_rows(N, 48, seed=N)
        for M in (1, 2, 3, 4, 8, 9, 16):
            x_h = syn.activations(7 + M, M, K)
            y_ref, tol = oracle.matvec_rows(x_h, qs_h, d_h, K, rows)
            for impl in IMPL_FOR.get(M, (0, 2, 4)):
                st = torch.zeros(1, dtype=torch.int32, device="cuda")
                y = run(dev(x_h), qs, d, K, impl, M, N, st)
                if y is None:
                    continue
                check_status(st, f"{name} M={M} impl={impl}")
                assert_within_tolerance(host(y).astype(np.float64)[:, rows], y_ref, tol, f"{name} M={M} impl={impl}")
        print(f"layer shape {name} {N}x{K}: clear, parity green", flush=True)


def grouped():
    for M, K, Ns in ((1, 4096, (4096, 256, 256)), (2, 8448, (70, 50)), (4, 4096, (4096, 256, 256)),
                     (8, 4096, (1000, 3000)), (5, 8448, (100, 60)),
                     (12, 4096, (4096, 256, 256)), (10, 4096, (1000, 3000)), (16, 2048, (300, 70, 45))):
        mats = []
        for j, N in enumerate(Ns):
            qs_h, _ = oracle.pack(syn.codes(11, N, K, linear=j))
            mats.append((qs_h, syn.scales(11, N, K // 256, linear=j)))
        x_h = syn.activations(11, M, K)
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        ys = tq2.matvec_grouped(dev(x_h), [dev(q) for q, _ in mats], [dev(d) for _, d in mats], status=st)
        check_status(st, f"grouped M={M} K={K} {Ns}")
        for (qs_h, d_h), y in zip(mats, ys):
            rows = sample_rows(qs_h.shape[0], 48)
            y_ref, tol = oracle.matvec_rows(x_h, qs_h, d_h, K, rows)
            assert_within_tolerance(host(y).astype(np.float64)[:, rows], y_ref, tol, f"grouped M={M} K={K}")
    print("grouped calls: clear, parity green", flush=True)


def affine4():
    n_calls = 0
    cases = [(M, N, K, G) for K in (256, 512, 2048) for N in (1, 15, 16, 17, 33, 70) for M in (1, 2, 3, 16)
             for G in (64, 128, 256)]
    cases += [(M, 16384, 4096, 128) for M in (1, 2)] + [(1, 4096, 16384, 64), (2, 4096, 4096, 256)]
    for M, N, K, G in cases:
        qs_h, s_h, z_h = syn.affine4_weights(M + N + K + G, N, K, G)
        x_h = syn.activations(M + N, M, K)
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        y = tq2.affine4_matvec(dev(x_h), dev(qs_h), dev(s_h), dev(z_h), G, status=st)
        check_status(st, f"affine4 M={M} N={N} K={K} G={G}")
        if N > 2048:
            rows = sample_rows(N, 32, seed=N)
            y_ref, tol = oracle.affine4_rows(x_h, qs_h, s_h, z_h, K, G, rows)
            yg = host(y).astype(np.float64)[:, rows]
        else:
            y_ref, tol = oracle.affine4(x_h, qs_h, s_h, z_h, K, G)
            yg = host(y).astype(np.float64)
        assert_within_tolerance(yg, y_ref, tol, f"affine4 M={M} N={N} K={K} G={G}")
        n_calls += 1
    print(f"affine-int4: clear, parity green ({n_calls} calls)", flush=True)


def gemm():
    n_calls = 0
    cases = [(17, 128, 256), (64, 100, 512), (130, 257, 768), (300, 300, 1024), (16, 512, 4096),
             (16, 16384, 1024), (200, 2048, 1024), (2048, 256, 4096), (512, 4096, 4096),
             (64, 256, 4096), (32, 512, 2048), (9, 20480, 1024)]
    for M, N, K in cases:
        # prologue in every tile (no workspace), or as a pass of its own where it pays
        for prologue, ws in ((False, None), (True, None), (True, "auto")):
            seed = M + N + K + int(prologue)
            codes = syn.codes(seed, N, K)
            qs_h, _ = oracle.pack(codes)
            d_h = syn.scales(seed, N, K // 256)
            x_h = syn.activations(seed, M, K, heavy=prologue)
            s = float(syn.act_scale(seed)) if prologue else 0.0
            st = torch.zeros(1, dtype=torch.int32, device="cuda")
            y = tq2.gemm(dev(x_h), dev(qs_h), dev(d_h), act_scale=s, status=st, impl=1, workspace=ws)
            check_status(st, f"gemm M={M} N={N} K={K} prologue={prologue} workspace={ws}")
            rows = sample_rows(N, 48, seed=M) if N > 512 else np.arange(N)
            y_ref, tol = oracle.matvec_rows(x_h, qs_h, d_h, K, rows, act_scale=s)
            assert_within_tolerance(host(y).astype(np.float64)[:, rows], y_ref, tol,
                                    f"gemm M={M} N={N} K={K} prologue={prologue} workspace={ws}")
            n_calls += 1
    print(f"tcgen05 GEMM: clear, parity green ({n_calls} calls)", flush=True)


if __name__ == "__main__":
    assert tq2.bounds_checked(), "run with TQ2_BOUNDS_CHECK=1"
    tq2.load()
    tiny_sweep()
    layer_shapes()
    grouped()
    affine4()
    gemm()
    print("OK")
