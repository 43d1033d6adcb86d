"""CPU enumeration of the number-format facts the tensor-core unpacks rest on
(BitCPM ternary page, linear-factoring paragraph: y is the per-block sum of
x times q - 1, scaled once by d_b; the kernels reach the q - 1 values without
a conversion instruction).  The masks and constants are read from the kernel
sources, so a change to them is checked here:

  * class unpack (tq2_matvec_mma.cu, tq2_matvec_ps.cu): a 16-bit lane ANDed
    with 3 << 2c is the fp16 bit pattern q * 4^c, i.e. exactly q * 2^(2c-24),
    for every lane value and class; the word shifted right by 8 gives the
    codes of the odd bytes;
  * class-column combination (tq2_matvec_mma.cu): the class sums scaled by
    2^(24 - 2c), less the block's sum of x, are sum_k x_k (q_k - 1) exactly;
  * pre-scaled B (tq2_matvec_ps.cu): x * 4^(3 - c) is exact in fp16 while
    |x| <= 1023.5, each lane times its B is q * x * 2^-18 exactly (an fp32
    product), the test on the bit pattern of |x| (>= 0x6400) picks exactly
    the blocks holding |x| >= 1024, Inf or NaN, and there x * 4^-c loses at
    most 2^-19 of x; the scale-back constants are the powers of two;
  * tcgen05 GEMM expand (tq2_gemm_tc05.cu): OR-ing a code into 0x6400 gives
    fp16 1024 + q, adding -1025 gives q - 1 exactly, and (q - 1) * d is exact
    for every finite fp16 d;
  * affine int4 (tq2_matvec_affine4.cu): the nibble masks give q * 2^-24 and
    q * 2^-20 exactly, and the class and zero-point combination is the
    affine group sum.
"""
import os
import re

import numpy as np
import pytest

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "quantized_gemv_tq2_gb300", "csrc")


def _src(name):
    with open(os.path.join(CSRC, name)) as f:
        return f.read()


def _f16(bits):
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


ALL16 = np.arange(1 << 16, dtype=np.uint32)
FINITE = _f16(ALL16)[np.isfinite(_f16(ALL16))]


def test_class_masks_in_the_sources():
    mma, ps = _src("tq2_matvec_mma.cu"), _src("tq2_matvec_ps.cu")
    assert "0x00030003u << (2 * cl)" in mma
    # the pre-scaled kernel spells the four class masks out
    for c in range(4):
        m = 0x00030003 << (2 * c)
        assert f"w0 & 0x{m:08X}u" in ps, f"class {c} mask changed"
    assert re.search(r"s0 = w0 >> 8, s1 = w1 >> 8", ps)


@pytest.mark.parametrize("c", range(4))
def test_lane_mask_is_q_times_4c_subnormal(c):
    """Lane bits 0-7 hold codes 0..3 of one byte (code j at bits 2j), bits
    8-15 the next byte: the mask keeps code c, the shift by 8 code 4 + c."""
    lane = ALL16
    got = _f16(lane & (3 << (2 * c)))
    q = (lane >> (2 * c)) & 3
    assert np.array_equal(got, q * 2.0 ** (2 * c - 24))
    got_hi = _f16((lane >> 8) & (3 << (2 * c)))
    q_hi = (lane >> (8 + 2 * c)) & 3
    assert np.array_equal(got_hi, q_hi * 2.0 ** (2 * c - 24))


def test_class_column_combination_is_the_block_sum():
    """Per 256-block: sum_c 2^(24-2c) * sum_k lane_c(k) x_k - sum_k x_k equals
    sum_k x_k (q_k - 1), with the combination constants of the kernel."""
    mma = _src("tq2_matvec_mma.cu")
    consts = re.search(r"acc\[2\]\[0\] \* ([0-9.]+)f \+ acc\[3\]\[0\] \* ([0-9.]+)f\)\s*"
                       r":\s*\(acc\[0\]\[0\] \* ([0-9.]+)f \+ acc\[1\]\[0\] \* ([0-9.]+)f\)", mma)
    assert consts, "the class combination changed: update this check"
    c2, c3, c0, c1 = (float(v) for v in consts.groups())
    scale = [c0, c1, c2, c3]
    assert scale == [2.0 ** (24 - 2 * c) for c in range(4)]
    rng = np.random.default_rng(7)
    for _ in range(20):
        q = rng.integers(0, 3, size=256)
        x = rng.standard_normal(256).astype(np.float16).astype(np.float64)
        # 16 words of 16 codes: code j of a word at bits 2j (j < 8) or 16 + 2(j - 8)
        words = np.zeros(16, dtype=np.uint64)
        for k in range(256):
            w, j = divmod(k, 16)
            words[w] |= np.uint64(int(q[k]) << (2 * j if j < 8 else 16 + 2 * (j - 8)))
        words = words.astype(np.uint32)
        total = -x.sum()
        for c in range(4):
            s = 0.0
            for w in range(16):
                for src, base in ((words[w], 0), (words[w] >> np.uint32(8), 4)):
                    m = np.uint32(0x00030003 << (2 * c))
                    v = int(src & m)
                    lo, hi = _f16(v & 0xFFFF), _f16(v >> 16)
                    s += lo * x[16 * w + base + c] + hi * x[16 * w + 8 + base + c]
            total += scale[c] * s
        assert total == float(np.dot(x, q - 1))


def test_prescale_constants():
    ps = _src("tq2_matvec_ps.cu")
    s01 = re.search(r"s01 = big \? __floats2half2_rn\(([0-9.]+)f, ([0-9.]+)f\) : __floats2half2_rn\(([0-9.]+)f, ([0-9.]+)f\)", ps)
    s23 = re.search(r"s23 = big \? __floats2half2_rn\(([0-9.]+)f, ([0-9.]+)f\) : __floats2half2_rn\(([0-9.]+)f, ([0-9.]+)f\)", ps)
    sc = re.search(r"sc = big \? ([0-9.e+-]+)f : ([0-9.e+-]+)f;", ps)
    rs = re.search(r"rs = big \? ([0-9.]+)f : ([0-9.]+)f;", ps)
    thr = re.search(r"\(mx & 0xFFFFu\) >= (0x[0-9A-Fa-f]+)u\) \|\| \(\(mx >> 16\) >= (0x[0-9A-Fa-f]+)u", ps)
    assert s01 and s23 and sc and rs and thr, "the pre-scaled constants changed: update this check"
    b01, b23 = [float(v) for v in s01.groups()], [float(v) for v in s23.groups()]
    big = [b01[0], b01[1], b23[0], b23[1]]
    small = [b01[2], b01[3], b23[2], b23[3]]
    assert small == [4.0 ** (3 - c) for c in range(4)]
    assert big == [4.0 ** -c for c in range(4)]
    assert [float(v) for v in sc.groups()] == [2.0 ** -24, 2.0 ** -18]
    assert [float(v) for v in rs.groups()] == [2.0 ** 24, 2.0 ** 18]
    assert int(thr.group(1), 16) == int(thr.group(2), 16) == 0x6400
    assert _f16(0x6400) == 1024.0


def test_prescale_exact_below_1024():
    x = FINITE[np.abs(FINITE) <= 1023.5]
    assert x.size == 2 * 0x6400  # every fp16 pattern below 1024, both signs
    for c in range(4):
        s = 4.0 ** (3 - c)
        b = (x.astype(np.float16) * np.float16(s)).astype(np.float64)  # fp16 multiply, round to nearest
        assert np.array_equal(b, x * s)
        for q in (0, 1, 2):
            prod = (q * 2.0 ** (2 * c - 24)) * b        # exact in fp64
            assert np.array_equal(prod.astype(np.float32).astype(np.float64), prod)  # exact in fp32
            assert np.array_equal(prod, q * x * 2.0 ** -18)
    # the first value past the range overflows x * 64
    with np.errstate(over="ignore"):
        assert np.isinf(np.float16(1024.0) * np.float16(64.0))


def test_big_test_on_bit_patterns():
    """|x| bits >= 0x6400 exactly when |x| >= 1024, Inf or NaN."""
    a = ALL16 & 0x7FFF
    v = _f16(a)
    assert np.array_equal(a >= 0x6400, (v >= 1024.0) | np.isnan(v))


def test_big_blocks_lose_at_most_2_to_minus_19():
    x = FINITE
    for c in range(4):
        s = 4.0 ** -c
        b = (x.astype(np.float16) * np.float16(s)).astype(np.float64)
        err = np.abs(b / s - x)
        assert err.max() <= 2.0 ** -19
        # only where x * 4^-c falls below the normal range (2^-14)
        assert err[np.abs(x) * s >= 2.0 ** -14].max() == 0.0
        # products q * 4^c * 2^-24 * b are exact in fp32; scaled back by 2^24 they are q * b / s
        for q in (1, 2):
            prod = (q * 2.0 ** (2 * c - 24)) * b
            assert np.array_equal(prod.astype(np.float32).astype(np.float64), prod)


def test_gemm_expand_is_exact():
    g = _src("tq2_gemm_tc05.cu")
    assert "(t & 0x00030003u) | 0x64006400u" in g and "__float2half2_rn(-1025.0f)" in g
    d = FINITE.astype(np.float16)
    bias = np.float16(-1025.0)
    for q in (0, 1, 2):
        f = np.array([0x6400 | q], dtype=np.uint16).view(np.float16)[0]
        assert float(f) == 1024.0 + q
        qm1 = f + bias                       # fp16 add, round to nearest
        assert float(qm1) == q - 1
        prod = (np.full_like(d, qm1) * d).astype(np.float64)
        assert np.array_equal(prod, (q - 1) * d.astype(np.float64))


def test_affine4_nibble_unpack_and_combination():
    """Affine int4 (tq2_matvec_affine4.cu): w & 0x000F000F leaves q * 2^-24,
    w & 0x00F000F0 leaves 16 q = q * 2^-20, both exact (subnormal) for every
    lane; the high-nibble class is brought to units of 2^-24 by 1/16 and the
    group sum back by 2^24, and s * (sum q x - z * sum x) is the affine
    group's sum_k s (q_k - z) x_k."""
    a4 = _src("tq2_matvec_affine4.cu")
    m = re.search(r"kLo = (0x[0-9A-Fa-f]+)u, kHi = (0x[0-9A-Fa-f]+)u;", a4)
    comb = re.search(r"\(c\[0\]\[0\] \+ c\[1\]\[1\] \* ([0-9.]+)f\)", a4)
    back = re.search(r"acc_lo = fmaf\(slo \* ([0-9.]+)f, dlo, acc_lo\);", a4)
    assert m and comb and back, "the affine-int4 unpack changed: update this check"
    lo, hi = int(m.group(1), 16), int(m.group(2), 16)
    assert (lo, hi) == (0x000F000F, 0x00F000F0)
    inv16, two24 = float(comb.group(1)), float(back.group(1))
    assert (inv16, two24) == (2.0 ** -4, 2.0 ** 24)
    lane = ALL16
    assert np.array_equal(_f16(lane & (lo & 0xFFFF)), (lane & 15) * 2.0 ** -24)
    assert np.array_equal(_f16(lane & (hi & 0xFFFF)), ((lane >> 4) & 15) * 2.0 ** -20)
    rng = np.random.default_rng(11)
    for G in (64, 128, 256):
        q = rng.integers(0, 16, size=G)
        x = rng.standard_normal(G).astype(np.float16).astype(np.float64)
        s = float(np.float16(rng.uniform(0.01, 0.1)))
        z = float(np.float16(rng.integers(0, 16)))
        # two codes per byte, code k at bits 4 (k % 2) of byte k / 2; 8 per 32-bit word
        cls = [0.0] * 4
        for k in range(G):
            byte, nib = divmod(k, 2)
            c = 2 * (byte % 2) + nib  # bytes 0 / 2 of a word: classes 0, 1; bytes 1 / 3 (after >> 8): 2, 3
            shift = 4 * nib
            cls[c] += _f16((int(q[k]) << shift) & (lo if nib == 0 else hi) & 0xFFFF) * x[k]
        dsum = cls[0] + cls[1] * inv16 + cls[2] + cls[3] * inv16
        y = s * two24 * dsum - s * z * x.sum()
        want = float(np.sum(s * (q - z) * x))
        assert abs(y - want) <= 1e-12 * max(1.0, float(np.sum(np.abs(s * (q - z) * x))))
