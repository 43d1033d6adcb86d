"""The C-ABI library loads, exports every declared symbol, and rejects bad
arguments on the host (no GPU needed: every check below returns before any
CUDA call; the fake pointers are never dereferenced)."""
import ctypes

import pytest

import quantized_gemv_tq2_gb300 as tq2

OK, NULL, SHAPE, ALIGN, DTYPE, ARG = 0, 1, 2, 3, 4, 5
P = ctypes.c_void_p
A16 = P(0x10000)   # 16-byte aligned fake device pointer
A2 = P(0x10002)    # 2-byte aligned only
NUL = P(0)
S = P(0)           # stream


@pytest.fixture(scope="module")
def L():
    return tq2.load()


def test_every_declared_symbol_is_exported(L):
    names = tq2.declared_symbols()
    assert set(names) >= {"tq2_pack", "tq2_unpack", "tq2_from_dense", "tq2_matvec", "tq2_matvec_grouped",
                          "tq2_matvec_impl", "tq2_matvec_requant", "tq2_gemm",
                          "tq2_affine4_matvec", "tq2_matvec_workspace_size", "tq2_status_string", "tq2_version",
                          "tq2_test_matvec_stall", "tq2_matvec_grouped_requant", "tq2_test_gemm_stall",
                          "tq2_trace_size", "tq2_trace_read", "tq2_gemm_workspace_size"}
    for n in names:
        assert hasattr(L, n), n  # dlsym succeeds


def test_trace_entry_points_outside_the_trace_build(L):
    assert L.tq2_trace_size() == 0
    buf = ctypes.create_string_buffer(64)
    assert L.tq2_trace_read(ctypes.cast(buf, P), 64) == ARG


def test_version_and_status_strings(L):
    assert tq2.version() >= 100
    for st in range(8):
        assert tq2.status_string(st).startswith("TQ2_")
    assert "unknown" in tq2.status_string(99)
    assert tq2.matvec_workspace_size(1, 4096, 4096) == 0


def test_workspace_sizes():
    """2 M K bytes (the prologue's codes as fp16) where the automatic plan
    runs the prologue as a pass of its own: with the tcgen05 GEMM when it
    has more than 4 weight tiles (N > 512) -- down-sized K from M = 8, the
    other GEMM-preferred shapes -- else 0; tq2_gemm_workspace_size is 2 M K
    for every valid shape (enough for every plan)."""
    ws = tq2.matvec_workspace_size
    assert ws(1, 16384, 4096) == 0 and ws(2, 4096, 16384) == 0   # the M <= 2 kernels
    assert ws(6, 4096, 16384) == 0                               # the pre-scaled kernel
    assert ws(8, 4096, 16384) == 2 * 8 * 16384                   # the GEMM, given the pass
    assert ws(9, 4096, 16384) == 2 * 9 * 16384
    assert ws(12, 4096, 4096) == 2 * 12 * 4096
    assert ws(11, 4096, 4096) == 0                               # the pre-scaled kernel at K = 4096
    assert ws(16, 256, 4096) == 0                                # the GEMM on two weight tiles
    assert ws(16, 16384, 4096) == 0                              # the pre-scaled kernel
    assert ws(0, 32, 256) == 0 and ws(17, 32, 256) == 0 and ws(8, 4096, 300) == 0
    gs = tq2.gemm_workspace_size
    assert gs(1, 32, 256) == 512 and gs(2048, 16384, 4096) == 2 * 2048 * 4096
    assert gs(0, 32, 256) == 0 and gs(5, 32, 300) == 0 and gs(5, 0, 256) == 0 and gs(2 ** 31, 32, 256) == 0


def mv(L, x=A16, M=1, qs=A16, d=A16, N=32, K=512, y=A16, yd=0, s=0.0, st=NUL, impl=None, ws=NUL, wsb=0):
    if impl is None:
        return L.tq2_matvec(x, M, qs, d, N, K, y, yd, s, ws, wsb, st, S)
    return L.tq2_matvec_impl(x, M, qs, d, N, K, y, yd, s, ws, wsb, st, S, impl)


def test_grouped_workspace_sizes(L):
    """2 M K where the group runs as consecutive calls with one prologue pass
    (M >= 12 with every N_j > 512, or K >= 8192 at M >= 9, or a matrix that
    would take the GEMM at 3 <= M <= 8), else 0 (one launch)."""
    def gs(M, K, Ns):
        a = (ctypes.c_int64 * len(Ns))(*Ns)
        return L.tq2_matvec_grouped_workspace_size(M, K, len(Ns), ctypes.cast(a, P))
    assert gs(1, 4096, (4096, 256, 256)) == 0 and gs(2, 4096, (16384, 16384)) == 0
    assert gs(8, 4096, (4096, 256, 256)) == 0        # one pre-scaled launch
    assert gs(9, 4096, (4096, 256, 256)) == 0        # one pre-scaled launch up to M = 16 with k/v in it
    assert gs(16, 4096, (4096, 256, 256)) == 0
    assert gs(11, 4096, (16384, 16384)) == 0         # one launch up to M = 11
    assert gs(12, 4096, (16384, 16384)) == 2 * 12 * 4096
    assert gs(16, 4096, (16384, 16384)) == 2 * 16 * 4096
    assert gs(9, 16384, (4096, 256)) == 2 * 9 * 16384  # K >= 8192: the GEMM's single calls
    assert gs(8, 16384, (4096, 4096)) == 2 * 8 * 16384  # down-sized K takes the GEMM at M = 8 given the pass
    assert gs(12, 4096, (4096,)) == 0                  # one matrix: a single call
    assert gs(9, 300, (64,)) == 0 and gs(9, 4096, (-1,)) == 0 and gs(17, 4096, (64,)) == 0
    assert gs(9, 4096, ()) == 0 and gs(9, 4096, (1, 2, 3, 4, 5)) == 0
    assert L.tq2_matvec_grouped_workspace_size(9, 4096, 1, NUL) == 0


def test_workspace_arguments_are_checked(L):
    """A workspace of > 0 bytes must be a non-NULL, 16-byte aligned pointer
    (0 bytes: none, whatever the pointer)."""
    assert mv(L, ws=NUL, wsb=64, s=0.5) == NULL
    assert mv(L, ws=A2, wsb=64, s=0.5) == ALIGN
    assert mv(L, ws=NUL, wsb=64) == NULL       # checked with or without the prologue
    assert mv(L, ws=A2, wsb=64, impl=4, M=9) == ALIGN
    assert rq(L, ws=A2, wsb=64) == ALIGN
    assert gm(L, ws=NUL, wsb=64) == NULL
    assert gm(L, ws=A2, wsb=64, s=0.5) == ALIGN
    assert gm(L, ws=A2, wsb=0, M=0, x=NUL, y=NUL) == OK  # an empty call checks nothing more


def test_matvec_rejects_bad_shapes(L):
    assert mv(L, K=300) == SHAPE
    assert mv(L, K=-256) == SHAPE
    assert mv(L, N=-1) == SHAPE
    assert mv(L, M=17) == SHAPE
    assert mv(L, M=-1) == SHAPE
    assert mv(L, N=2 ** 62, K=2 ** 20) == SHAPE  # N*K overflows


def test_matvec_rejects_bad_dtype_and_args(L):
    assert mv(L, yd=2) == DTYPE
    assert mv(L, s=-0.5) == ARG
    assert mv(L, s=float("nan")) == ARG
    assert mv(L, s=float("inf")) == ARG
    assert mv(L, impl=8) == ARG
    assert mv(L, impl=7, M=3) == ARG  # the small-N kernel takes M <= 2
    assert mv(L, impl=5) == ARG  # retired numbers
    assert mv(L, impl=3) == ARG
    assert mv(L, impl=-1) == ARG
    assert mv(L, impl=1, M=3) == ARG  # the class-column tensor-core kernels take M <= 2
    assert mv(L, impl=4, M=17) == SHAPE  # the pre-scaled kernel takes M <= 16, as the API


def rq(L, x=A16, M=1, qs=A16, d=A16, N=32, K=512, y=A16, yd=0, s=0.0, so=0.5, st=NUL, impl=0, ws=NUL, wsb=0):
    return L.tq2_matvec_requant(x, M, qs, d, N, K, y, yd, s, so, ws, wsb, st, S, impl)


def test_requant_rejects_bad_arguments(L):
    assert rq(L, so=-0.5) == ARG
    assert rq(L, so=float("nan")) == ARG
    assert rq(L, so=float("inf")) == ARG
    assert rq(L, s=-1.0) == ARG
    assert rq(L, K=300) == SHAPE
    assert rq(L, M=17) == SHAPE
    assert rq(L, yd=3) == DTYPE
    assert rq(L, impl=8) == ARG
    assert rq(L, impl=1, M=3) == ARG
    assert rq(L, x=NUL) == NULL
    assert rq(L, y=A2) == ALIGN
    assert rq(L, M=0, x=NUL, y=NUL) == OK
    assert rq(L, N=0, qs=NUL, d=NUL, y=NUL, so=0.0) == OK


def gm(L, x=A16, M=64, qs=A16, d=A16, N=32, K=512, y=A16, yd=0, s=0.0, so=0.0, st=NUL, impl=0, ws=NUL, wsb=0):
    return L.tq2_gemm(x, M, qs, d, N, K, y, yd, s, so, ws, wsb, st, S, impl)


def test_gemm_rejects_bad_arguments(L):
    assert gm(L, K=300) == SHAPE
    assert gm(L, M=-1) == SHAPE
    assert gm(L, M=2 ** 31) == SHAPE
    assert gm(L, yd=2) == DTYPE
    assert gm(L, s=-1.0) == ARG
    assert gm(L, so=float("nan")) == ARG
    assert gm(L, impl=3) == ARG
    assert gm(L, impl=-1) == ARG
    assert gm(L, x=NUL) == NULL
    assert gm(L, y=NUL) == NULL
    assert gm(L, x=A2) == ALIGN
    assert gm(L, M=0, x=NUL, y=NUL) == OK
    assert gm(L, N=0, qs=NUL, d=NUL, y=NUL) == OK


def test_matvec_empty_shapes_are_noops(L):
    assert mv(L, M=0, x=NUL, y=NUL) == OK
    assert mv(L, N=0, qs=NUL, d=NUL, y=NUL) == OK


def test_matvec_rejects_null_and_misaligned(L):
    assert mv(L, x=NUL) == NULL
    assert mv(L, qs=NUL) == NULL
    assert mv(L, d=NUL) == NULL
    assert mv(L, y=NUL) == NULL
    assert mv(L, x=A2) == ALIGN
    assert mv(L, qs=A2) == ALIGN
    assert mv(L, d=P(0x10001)) == ALIGN
    assert mv(L, y=A2, yd=0) == ALIGN
    assert mv(L, st=P(0x10002)) == ALIGN


def test_stall_hook_rejects_bad_arguments(L):
    def stall(x=A16, M=1, qs=A16, d=A16, N=32, K=512, y=A16, st=A16, stage=0, lim=100):
        return L.tq2_test_matvec_stall(x, M, qs, d, N, K, y, st, S, stage, lim)
    assert stall(stage=-1) == ARG
    assert stall(lim=0) == ARG
    assert stall(lim=200001) == ARG
    assert stall(st=NUL) == NULL
    assert stall(K=300) == SHAPE
    assert stall(M=17) == SHAPE
    assert stall(M=3) == ARG      # impl 1 takes M <= 2
    assert stall(y=A2) == ALIGN   # fp32 y
    assert stall(M=0, x=NUL, y=NUL) == OK


def test_gemm_stall_hook_rejects_bad_arguments(L):
    def stall(x=A16, M=16, qs=A16, d=A16, N=128, K=512, y=A16, s=0.0, st=A16, stage=0, lim=100):
        return L.tq2_test_gemm_stall(x, M, qs, d, N, K, y, s, st, S, stage, lim)
    assert stall(stage=-1) == ARG
    assert stall(lim=0) == ARG
    assert stall(lim=200001) == ARG
    assert stall(st=NUL) == NULL
    assert stall(K=300) == SHAPE
    assert stall(s=-1.0) == ARG
    assert stall(y=A2) == ALIGN
    assert stall(M=0, x=NUL, y=NUL) == OK


def test_layout_calls_reject_bad_arguments(L):
    assert L.tq2_pack(A16, 4, 100, A16, NUL, S) == SHAPE
    assert L.tq2_pack(NUL, 4, 256, A16, NUL, S) == NULL
    assert L.tq2_pack(A16, 0, 256, A16, NUL, S) == OK
    assert L.tq2_unpack(A16, -1, 256, A16, S) == SHAPE
    assert L.tq2_unpack(A16, 4, 256, NUL, S) == NULL
    assert L.tq2_from_dense(A16, 0, 4, 255, A16, A16, NUL, S) == SHAPE
    assert L.tq2_from_dense(A16, 7, 4, 256, A16, A16, NUL, S) == DTYPE
    assert L.tq2_from_dense(A16, 0, 4, 256, A16, NUL, NUL, S) == NULL
    assert L.tq2_from_dense(A2, 0, 4, 256, A16, A16, NUL, S) == ALIGN  # fp32 W needs 4 bytes
    assert L.tq2_from_dense(A16, 1, 0, 256, A16, A16, NUL, S) == OK


def test_grouped_rejects_bad_arguments(L):
    n = 3
    Pn = ctypes.c_void_p * n
    good = Pn(0x10000, 0x20000, 0x30000)
    ys = Pn(0x40000, 0x50000, 0x60000)
    Ns = (ctypes.c_int64 * n)(64, 32, 16)
    cast = lambda a: ctypes.cast(a, ctypes.c_void_p)
    G = lambda **k: L.tq2_matvec_grouped(k.get("x", A16), k.get("M", 1), k.get("K", 512), k.get("n", n),
                                         cast(k.get("qs", good)), cast(k.get("d", good)), cast(k.get("N", Ns)),
                                         cast(k.get("y", ys)), k.get("yd", 0), k.get("s", 0.0),
                                         k.get("ws", NUL), k.get("wsb", 0), NUL, S)
    assert G(n=0) == ARG
    assert G(n=5) == ARG                          # more than TQ2_MAX_GROUP
    assert L.tq2_matvec_grouped(A16, 1, 512, n, NUL, cast(good), cast(Ns), cast(ys), 0, 0.0, NUL, 0, NUL, S) == NULL
    assert G(K=300) == SHAPE
    assert G(M=17) == SHAPE
    assert G(N=(ctypes.c_int64 * n)(64, -1, 16)) == SHAPE
    assert G(yd=3) == DTYPE
    assert G(s=-1.0) == ARG
    assert G(qs=Pn(0x10000, 0x20002, 0x30000)) == ALIGN
    assert G(y=Pn(0x40000, 0, 0x60000)) == NULL
    assert G(x=A2) == ALIGN
    assert G(M=0) == OK                           # nothing to do
    assert G(ws=NUL, wsb=64) == NULL              # workspace: non-NULL and 16-byte aligned when given
    assert G(ws=A2, wsb=64, M=9, s=0.5) == ALIGN
    # the requantising variant: one finite, non-negative scale per matrix
    F3 = ctypes.c_float * n
    R = lambda sc, **k: L.tq2_matvec_grouped_requant(k.get("x", A16), k.get("M", 1), 512, n, cast(good), cast(good),
                                                     cast(Ns), cast(ys), 0, 0.0, sc, NUL, 0, NUL, S)
    assert R(NUL) == NULL
    assert R(cast(F3(0.5, -0.1, 0.2))) == ARG
    assert R(cast(F3(0.5, float("inf"), 0.2))) == ARG
    assert R(cast(F3(0.5, float("nan"), 0.2))) == ARG
    assert R(cast(F3(0.5, 0.0, 0.2)), M=0) == OK
    assert R(cast(F3(0.5, 0.1, 0.2)), x=A2) == ALIGN
    assert G(N=(ctypes.c_int64 * n)(0, 0, 0)) == OK


def a4(L, x=A16, M=1, qs=A16, s=A16, z=A16, N=64, K=512, G=128, y=A16, yd=0, st=NUL):
    return L.tq2_affine4_matvec(x, M, qs, s, z, N, K, G, y, yd, st, S)


def test_affine4_rejects_bad_arguments(L):
    assert a4(L, K=300) == SHAPE
    assert a4(L, K=-256) == SHAPE
    assert a4(L, M=17) == SHAPE
    assert a4(L, M=-1) == SHAPE
    assert a4(L, yd=2) == DTYPE
    for g in (0, 32, 100, 512, -64):
        assert a4(L, G=g) == ARG
    assert a4(L, x=NUL) == NULL
    assert a4(L, qs=NUL) == NULL
    assert a4(L, s=NUL) == NULL
    assert a4(L, z=NUL) == NULL
    assert a4(L, y=NUL) == NULL
    assert a4(L, x=A2) == ALIGN
    assert a4(L, qs=A2) == ALIGN
    assert a4(L, s=A2) == ALIGN
    assert a4(L, z=A2) == ALIGN
    assert a4(L, y=A2, yd=0) == ALIGN
    assert a4(L, st=P(0x10002)) == ALIGN
    assert a4(L, M=0, x=NUL, y=NUL) == OK
    assert a4(L, N=0, qs=NUL, s=NUL, z=NUL, y=NUL) == OK
