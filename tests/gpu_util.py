"""Helpers for the GPU parity tests: seeded cases, device transfer, and the
element-wise comparison against the CPU oracle."""
import numpy as np

import oracle
import tq2_synth as syn


def dev(a, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def host(t):
    return t.detach().cpu().numpy()


class Case:
    """Seeded inputs of one linear plus the oracle's packed weights."""

    def __init__(self, seed, M, N, K, heavy=False, prologue=False, linear=0):
        self.M, self.N, self.K = M, N, K
        self.codes = syn.codes(seed, N, K, linear=linear)
        self.d = syn.scales(seed, N, K // 256, linear=linear)
        self.x = syn.activations(seed, M, K, linear=linear, heavy=heavy)
        self.s = syn.act_scale(seed, linear=linear) if prologue else 0.0
        self.qs, flags = oracle.pack(self.codes)
        assert flags == 0

    def device(self):
        return dev(self.x), dev(self.qs), dev(self.d)

    def reference(self, rows=None):
        if rows is None:
            return oracle.matvec(self.x, self.qs, self.d, self.K, self.s)
        return oracle.matvec_rows(self.x, self.qs, self.d, self.K, rows, self.s)


def assert_within_tolerance(y_gpu, y_ref, tol_sum, what=""):
    """|y_gpu - y_ref| <= 1e-3 * sum_k |d_b x'_k| + 1e-6, element by element."""
    y = np.asarray(y_gpu, dtype=np.float64)
    assert y.shape == y_ref.shape, (y.shape, y_ref.shape)
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    err = np.abs(y - y_ref)
    bound = oracle.tolerance(tol_sum)
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; first at {tuple(i)}: "
            f"gpu={y[tuple(i)]!r} ref={y_ref[tuple(i)]!r} bound={bound[tuple(i)]!r}; "
            f"max err/bound={float((err / bound).max()):.3g}")
    return float((err / bound).max()) if err.size else 0.0


def sample_rows(N, count, seed=0):
    """Sorted distinct rows: the first/last few, every tile edge pattern, random."""
    rng = np.random.default_rng(seed)
    base = {0, 1, 15, 16, 17, N // 2, N - 17, N - 16, N - 2, N - 1}
    r = set(int(v) for v in base if 0 <= v < N)
    r.update(int(v) for v in rng.choice(N, size=min(count, N), replace=False))
    return np.array(sorted(r), dtype=np.int64)


class GuardedOutput:
    """An output tensor [M, N] inside a larger buffer whose PAD elements on
    each side hold a canary bit pattern, to catch writes outside [M, N]."""

    PAD = 256

    def __init__(self, M, N, dtype_code=0):
        import torch
        self.M, self.N = M, N
        if dtype_code == 0:
            self.buf = torch.empty(M * N + 2 * self.PAD, dtype=torch.int32, device="cuda")
            self.buf.fill_(0x7F8DEAD5)  # a NaN pattern no kernel writes
            self.y = self.buf[self.PAD:self.PAD + M * N].view(torch.float32).view(M, N)
        else:
            self.buf = torch.empty(M * N + 2 * self.PAD, dtype=torch.int16, device="cuda")
            self.buf.fill_(0x7E5B)
            self.y = self.buf[self.PAD:self.PAD + M * N].view(torch.float16).view(M, N)
        self.canary = self.buf[0].item()

    def check(self, what=""):
        import torch
        lo = self.buf[:self.PAD]
        hi = self.buf[self.PAD + self.M * self.N:]
        assert bool(torch.all(lo == self.canary)), f"{what}: write below y"
        assert bool(torch.all(hi == self.canary)), f"{what}: write above y"


def check_requant(y_gpu, y_ref, tol_sum, s_o, y_dtype, what):
    """Codes within the tolerance band, stored values exactly code * s_o."""
    s32 = np.float32(s_o)
    yg = np.asarray(y_gpu)
    code = np.rint(yg.astype(np.float64) / np.float64(s32))
    assert np.all(np.abs(code) <= 128), what
    assert np.all((code >= -128) & (code <= 127)), what
    stored = code.astype(np.float32) * s32  # one fp32 rounding, as the kernel
    if y_dtype == 1:
        stored = stored.astype(np.float16)
    assert np.array_equal(yg, stored.astype(yg.dtype)), what + ": stored value is not code * s"
    bound = oracle.tolerance(tol_sum)
    lo, _ = oracle.requant(y_ref - bound, s_o)
    hi, _ = oracle.requant(y_ref + bound, s_o)
    ref, _ = oracle.requant(y_ref, s_o)
    bad = (code < lo) | (code > hi)
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} codes outside the band; first at {i}: "
                             f"gpu={code[i]} band=[{lo[i]}, {hi[i]}] y_ref={y_ref[i]!r}")
    # the kernel's sums are far more accurate than the bound: it almost
    # always lands on the oracle's own code
    assert np.mean(code == ref) > 0.9, what
