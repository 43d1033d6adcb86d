"""GPU parity of pack / unpack / from_dense against the CPU oracle: bit-exact."""
import os

import numpy as np
import pytest

import oracle
import tq2_synth as syn
from gpu_util import dev, host

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    import quantized_gemv_tq2_gb300 as tq2
    tq2.load()
    return torch


def _status(torch):
    return torch.zeros(1, dtype=torch.int32, device="cuda")


@pytest.mark.parametrize("N,K", [(1, 256), (3, 768), (33, 512), (257, 1024), (4096, 4096),
                                 (16384, 4096), (4096, 16384)])
def test_pack_unpack_bit_exact(torch_cuda, N, K):
    torch = torch_cuda
    import quantized_gemv_tq2_gb300 as tq2
    codes = syn.codes(N + K, N, K)
    qs_ref, fl = oracle.pack(codes)
    st = _status(torch)
    qs = tq2.pack(dev(codes), status=st)
    back = tq2.unpack(qs, K)
    torch.cuda.synchronize()
    assert np.array_equal(host(qs), qs_ref)
    assert np.array_equal(host(back), codes)
    assert int(st.item()) == 0 == fl


def test_pack_bad_codes_and_unaligned_buffers(torch_cuda):
    torch = torch_cuda
    import quantized_gemv_tq2_gb300 as tq2
    N, K = 5, 512
    codes = syn.codes(3, N, K)
    codes[1, 7] = 3
    codes[4, 300] = -1
    codes[2, 0] = 9
    qs_ref, fl = oracle.pack(codes)
    assert fl == oracle.FLAG_BAD_CODE
    # offset views: not 16-byte aligned -> the byte-wise kernels
    big = torch.zeros(N * K + 3, dtype=torch.int8, device="cuda")
    cview = big[3:].view(N, K)
    cview.copy_(dev(codes))
    qbig = torch.zeros(N * K // 4 + 1, dtype=torch.uint8, device="cuda")
    qview = qbig[1:].view(N, K // 4)
    st = _status(torch)
    tq2.pack(cview, qs=qview, status=st)
    back_big = torch.zeros(N * K + 5, dtype=torch.int8, device="cuda")
    bview = back_big[5:].view(N, K)
    tq2.unpack(qview, K, codes=bview)
    torch.cuda.synchronize()
    assert np.array_equal(host(qview), qs_ref)
    assert int(st.item()) == oracle.FLAG_BAD_CODE
    assert np.array_equal(host(bview), oracle.unpack(qs_ref, K))
    assert host(qbig)[0] == 0 and np.all(host(back_big)[:5] == 0)  # no writes outside


def _from_dense_both(torch, W):
    import quantized_gemv_tq2_gb300 as tq2
    st = _status(torch)
    qs, d = tq2.from_dense(dev(W), status=st)
    torch.cuda.synchronize()
    qs_ref, d_ref, fl = oracle.from_dense(W)
    assert np.array_equal(host(qs), qs_ref)
    assert np.array_equal(host(d).view(np.uint16), d_ref.view(np.uint16))
    assert int(st.item()) == fl
    return fl


@pytest.mark.parametrize("wdtype", [np.float32, np.float16])
@pytest.mark.parametrize("N,K", [(7, 256), (129, 1024), (4096, 4096)])
def test_from_dense_round_trip_bit_exact(torch_cuda, wdtype, N, K):
    codes = syn.codes(N, N, K)
    d = syn.scales(N, N, K // 256)
    d[0, :] = np.float16(2.0 ** -20)  # subnormal scales too
    qs, _ = oracle.pack(codes)
    W = oracle.dequant(qs, d, K).astype(wdtype)
    fl = _from_dense_both(torch_cuda, W)
    assert fl == 0


def test_from_dense_generic_and_edge_blocks(torch_cuda):
    W = syn.dense_normal(2, 64, 2048)
    assert _from_dense_both(torch_cuda, W) == oracle.FLAG_INEXACT
    W16 = W.astype(np.float16)
    _from_dense_both(torch_cuda, W16)
    # the hand-derived blocks of tests/golden/from_dense_blocks.txt, one per row
    rows = []
    with open(os.path.join(GOLDEN, "from_dense_blocks.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append([float(v) for v in line.split("->")[0].split()])
    E = np.zeros((len(rows), 256), dtype=np.float32)
    for i, r in enumerate(rows):
        E[i, :len(r)] = r
    _from_dense_both(torch_cuda, E)
    # ties at +-0.5 and +-1.5 of d, -0.0, zero blocks, one NaN block
    T = np.zeros((4, 512), dtype=np.float32)
    T[0, :4] = [1.0, 0.5, -0.5, -0.0]
    T[1, 256:260] = [2.0, 3.0, -3.0, 1.0]
    T[2, 10] = np.nan
    T[2, 11] = 0.25
    T[3, 300] = 7e4
    _from_dense_both(torch_cuda, T)
