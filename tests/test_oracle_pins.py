"""Pins of the CPU oracle against things other than itself (no GPU needed).

Each test checks an oracle function against a closed form, an invariant,
hand-derived golden values (tests/golden/), brute force on a tiny case, or an
independent library (numpy), chosen so that a plausible slip in the oracle
(a dropped term, a wrong sign, index or bit order, a transposed operand)
fails at least one of them.
"""
import os

import numpy as np
import pytest

import oracle
import tq2_synth as syn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                yield line


# --------------------------------------------------------------------- fp16
def test_half_decode_matches_numpy_on_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.half_bits_to_f64(bits)
    ref = bits.view(np.float16).astype(np.float64)
    assert np.array_equal(ours, ref, equal_nan=True)


def test_half_encode_matches_numpy_round_to_nearest_even():
    rng = np.random.default_rng(0)
    # normals, subnormals, values around ties and the overflow edge
    vals = np.concatenate([
        rng.standard_normal(4000) * 10.0 ** rng.uniform(-9, 5, 4000),
        np.ldexp(rng.integers(0, 2048, 2000).astype(np.float64) + 0.5, -24),  # subnormal ties
        np.ldexp(1.0 + (2 * np.arange(1024) + 1) / 2048.0, 3),  # normal ties at 8..16
        [65504.0, 65519.99, 65520.0, -65520.0, 1e9, 0.0, -0.0, 2.0 ** -25,
         2.0 ** -25 * 1.0000001, 2.0 ** -26, 5.960464477539063e-08],
    ])
    ours = np.array([oracle.double_to_half(v) for v in vals], dtype=np.uint16)
    with np.errstate(over="ignore"):  # 65520 and beyond round to inf on purpose
        ref = vals.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)
    # hand-worked ties: 1 + 2^-11 is halfway between 1 and 1 + 2^-10 -> 1 (even)
    assert oracle.double_to_half(1.0 + 2.0 ** -11) == 0x3C00
    assert oracle.double_to_half(1.0 + 3 * 2.0 ** -11) == 0x3C02


# --------------------------------------------------------------------- pack
def test_pack_golden_layout():
    for line in _golden_lines("pack_layout.txt"):
        parts = line.split()
        codes = np.array([[int(c) for c in parts[:4]]], dtype=np.int8)
        want = int(parts[4], 16)
        qs, flags = oracle.pack(codes)
        assert qs[0, 0] == want, line
        assert flags == 0
        assert np.array_equal(oracle.unpack(qs, 4), codes)


def test_pack_unpack_all_valid_patterns_at_every_position():
    # the 81 valid bytes are the 4-digit base-4 numbers with digits in {0,1,2}
    pats = [c0 + 4 * c1 + 16 * c2 + 64 * c3
            for c3 in range(3) for c2 in range(3) for c1 in range(3) for c0 in range(3)]
    assert len(set(pats)) == 81
    nbytes = 81
    for shift in range(nbytes):  # pattern p lands at byte position (p + shift) % 81
        row = np.array([pats[(j - shift) % 81] for j in range(nbytes)], dtype=np.uint8)
        codes = np.array([[(row[k // 4] >> (2 * (k % 4))) & 3 for k in range(4 * nbytes)]],
                         dtype=np.int8)
        # closed form: code k = digit k%4 of byte k/4 in base 4
        assert np.array_equal(oracle.unpack(row[None, :], 4 * nbytes), codes)
        qs, flags = oracle.pack(codes)
        assert flags == 0 and np.array_equal(qs[0], row)


def test_pack_of_unpack_is_identity_on_every_byte_and_flags_code3():
    allb = np.arange(256, dtype=np.uint8)[None, :]
    codes = oracle.unpack(allb, 1024)
    qs, flags = oracle.pack(codes)
    assert np.array_equal(qs, allb)
    assert flags == oracle.FLAG_BAD_CODE  # some fields are 3
    valid = np.array([b for b in range(256) if all(((b >> (2 * i)) & 3) != 3 for i in range(4))],
                     dtype=np.uint8)[None, :]
    assert oracle.pack(oracle.unpack(valid, 4 * valid.size))[1] == 0


def test_pack_bad_codes_are_flagged_and_stored_masked():
    codes = np.array([[3, -1, 5, 1]], dtype=np.int8)
    qs, flags = oracle.pack(codes)
    assert flags == oracle.FLAG_BAD_CODE
    assert qs[0, 0] == (3 | (3 << 2) | (1 << 4) | (1 << 6))


# --------------------------------------------------------------------- recovery
def test_from_dense_golden_blocks():
    for line in _golden_lines("from_dense_blocks.txt"):
        lhs, rhs = line.split("->")
        head = [float(v) for v in lhs.split()]
        res, flags = rhs.split("|")
        res = res.split()
        d_want = float(res[0])
        codes_want = [int(c) for c in res[1:]]
        W = np.zeros((1, 256), dtype=np.float32)
        W[0, :len(head)] = head
        qs, d, fl = oracle.from_dense(W)
        assert fl == int(flags), line
        assert float(d[0, 0]) == d_want or (np.isinf(d_want) and np.isinf(float(d[0, 0]))), line
        codes = oracle.unpack(qs, 256)[0]
        assert list(codes[:len(codes_want)]) == codes_want, line
        assert np.all(codes[len(head):] == 1), line


@pytest.mark.parametrize("wdtype", [np.float32, np.float16])
def test_from_dense_round_trip_is_bit_exact(wdtype):
    N, K = 37, 1024
    codes = syn.codes(11, N, K)
    d = syn.scales(11, N, K // 256)
    # subnormal and tiny normal fp16 scales too
    d[0, :] = np.float16(2.0 ** -20)
    d[1, :] = np.float16(6.1035156e-05)
    d[2, :] = np.float16(3.0e-7)
    qs, fl = oracle.pack(codes)
    assert fl == 0
    W = oracle.dequant(qs, d, K)
    # W built independently from the codes: d * (code - 1)
    W_ind = (np.repeat(d.astype(np.float64), 256, axis=1) * (codes.astype(np.float64) - 1))
    assert np.array_equal(W.astype(np.float64), W_ind)
    qs2, d2, fl2 = oracle.from_dense(W.astype(wdtype))
    assert fl2 == 0
    assert np.array_equal(qs2, qs)
    assert np.array_equal(d2.view(np.uint16), d.view(np.uint16))
    assert np.array_equal(oracle.dequant(qs2, d2, K), W)


def test_from_dense_all_zero_block_gives_zero_scale_and_code_one():
    W = np.zeros((2, 512), dtype=np.float32)
    W[1, 256:] = 0.5 * np.sign(np.arange(256) % 3 - 1)
    qs, d, fl = oracle.from_dense(W)
    assert fl == 0
    assert float(d[0, 0]) == 0.0 and float(d[0, 1]) == 0.0 and float(d[1, 0]) == 0.0
    assert float(d[1, 1]) == 0.5
    c = oracle.unpack(qs, 512)
    assert np.all(c[0] == 1) and np.all(c[1, :256] == 1)
    assert np.array_equal(c[1, 256:], (np.arange(256) % 3).astype(np.int8))


def test_from_dense_generic_weights_flag_inexact_and_match_nearest_ternary():
    W = syn.dense_normal(5, 8, 512)
    qs, d, fl = oracle.from_dense(W)
    assert fl == oracle.FLAG_INEXACT
    c = oracle.unpack(qs, 512).astype(np.int64) - 1
    dd = np.repeat(d.astype(np.float32), 256, axis=1)
    r = W / dd  # numpy fp32 division, independent of the oracle's C
    assert np.array_equal(c, np.clip(np.rint(r), -1, 1).astype(np.int64))
    amax = np.abs(W.reshape(8, 2, 256)).max(axis=2)
    assert np.array_equal(d, amax.astype(np.float16))


# --------------------------------------------------------------------- fake-quant
def test_fakequant_golden_cases():
    for line in _golden_lines("fakequant_cases.txt"):
        xs, ss, qs = line.split()
        x = np.array([float(xs)], dtype=np.float16)
        for mode in (0, 1):
            q = oracle.fakequant_codes(x, float(ss), mode)
            assert int(q[0]) == int(qs), (line, mode)
        xq = oracle.fakequant(x, float(ss), 0)
        assert xq[0] == int(qs) * float(np.float32(ss))


def test_fakequant_idempotent_for_power_of_two_scale():
    x = syn.activations(3, 1, 4096, heavy=True)[0]
    for s in (0.25, 0.0625, 2.0 ** -10):
        q = oracle.fakequant_codes(x, s, 0)
        xq = (q.astype(np.float64) * s).astype(np.float16)  # exact: |q| <= 128, s = 2^-e
        assert np.array_equal(xq.astype(np.float64), q.astype(np.float64) * s)
        assert np.array_equal(oracle.fakequant_codes(xq, s, 0), q)


def test_fakequant_tiny_scale_saturates():
    x = np.array([1e-3, -1e-3, 5.0, -5.0, 0.0], dtype=np.float16)
    q = oracle.fakequant_codes(x, 1e-8, 0)
    assert list(q) == [127, -128, 127, -128, 0]


def test_fakequant_reciprocal_form_matches_definition_away_from_ties():
    x = syn.activations(4, 1, 200000, heavy=True)[0]
    mism = 0
    for lin in range(5):
        s = syn.act_scale(4, linear=lin)
        q0 = oracle.fakequant_codes(x, s, 0).astype(np.int64)
        q1 = oracle.fakequant_codes(x, s, 1).astype(np.int64)
        # the definition recomputed with numpy (fp64 x/s, half to even, clamp)
        t = x.astype(np.float64) / np.float64(np.float32(s))
        qd = np.clip(np.rint(t), -128, 127).astype(np.int64)
        assert np.array_equal(q1, qd)
        diff = q0 != q1
        mism += int(diff.sum())
        # every disagreement sits within a few fp32 ulps of a .5 tie
        frac = np.abs(np.abs(t[diff]) - np.floor(np.abs(t[diff])) - 0.5)
        assert np.all(frac <= 4 * 2.0 ** -23 * np.abs(t[diff]) + 1e-30)
        assert np.all(np.abs(q0[diff] - q1[diff]) == 1)
    assert mism < 50


# --------------------------------------------------------------------- output requantisation
def test_requant_golden_cases():
    for line in _golden_lines("requant_cases.txt"):
        ys, ss, cs, vs = line.split()
        codes, out = oracle.requant(np.array([float(ys)]), float(ss))
        assert int(codes[0]) == int(cs), line
        assert out[0] == float(vs), line


def test_requant_matches_definition_away_from_ties():
    # numpy restatement of the definition: clamp(round(y / s)) in fp64 on the
    # fp32 value of y, half to even; the reciprocal form may differ only
    # within a few fp32 ulps of a .5 tie
    rng = np.random.default_rng(11)
    y = (rng.standard_normal(100000) * 10.0 ** rng.uniform(-3, 2, 100000)).astype(np.float32)
    mism = 0
    for s in (0.013, 0.05, 0.0917, 1.7):
        codes, out = oracle.requant(y.astype(np.float64), s)
        t = y.astype(np.float64) / np.float64(np.float32(s))
        qd = np.clip(np.rint(t), -128, 127).astype(np.int64)
        c = codes.astype(np.int64)
        diff = c != qd
        mism += int(diff.sum())
        frac = np.abs(np.abs(t[diff]) - np.floor(np.abs(t[diff])) - 0.5)
        assert np.all(frac <= 4 * 2.0 ** -23 * np.abs(t[diff]) + 1e-30)
        assert np.all(np.abs(c[diff] - qd[diff]) == 1)
        assert np.array_equal(out, c * np.float64(np.float32(s)))
    assert mism < 50


def test_requant_is_the_activation_fakequant_on_fp16_values():
    # the same function at the other boundary: on values that are fp16 the
    # codes equal those of the (pinned) activation fake-quant
    x = syn.activations(5, 1, 20000, heavy=True)[0]
    for s in (0.02, 0.07, 0.25):
        codes, _ = oracle.requant(x.astype(np.float64), s)
        assert np.array_equal(codes, oracle.fakequant_codes(x, s, 0))


def test_requant_range_and_fixed_point():
    rng = np.random.default_rng(12)
    y = rng.standard_normal(5000) * 150.0
    for s in (0.125, 0.5, 2.0):  # powers of two: code * s is exact in fp32
        codes, out = oracle.requant(y, s)
        assert codes.min() >= -128 and codes.max() <= 127
        assert codes.min() == -128 and codes.max() == 127  # the clamp is reached
        codes2, out2 = oracle.requant(out, s)
        assert np.array_equal(codes2, codes) and np.array_equal(out2, out)


# --------------------------------------------------------------------- matvec
def _dense_from_codes(codes, d):
    return np.repeat(d.astype(np.float64), 256, axis=1) * (codes.astype(np.float64) - 1)


def test_matvec_golden_worked_example():
    x = np.zeros((1, 512), dtype=np.float16)
    d = np.zeros((2, 2), dtype=np.float16)
    codes = np.ones((2, 512), dtype=np.int8)
    want = {}
    for line in _golden_lines("matvec_small.txt"):
        p = line.split()
        if p[0] == "x":
            x[0, int(p[1])] = float(p[2])
        elif p[0] == "d":
            d[int(p[1])] = [float(v) for v in p[2:]]
        elif p[0] == "q":
            codes[int(p[1]), int(p[2])] = int(p[3])
        elif p[0] == "y":
            want[int(p[1])] = (float(p[2]), float(p[3]))
    qs, _ = oracle.pack(codes)
    y, t = oracle.matvec(x, qs, d, 512)
    ye = oracle.matvec_exact(x, qs, d, 512)
    for n, (yv, tv) in want.items():
        assert y[0, n] == yv and ye[0, n] == yv and t[0, n] == tv


@pytest.mark.parametrize("seed,M,N,K", [(0, 1, 32, 512), (1, 3, 65, 1024), (2, 2, 17, 4096)])
@pytest.mark.parametrize("prologue", [False, True])
def test_matvec_linearity_identity_against_numpy_dense(seed, M, N, K, prologue):
    """Factored per-block sum == dense dequantised W @ x (numpy), from the codes."""
    codes = syn.codes(seed, N, K)
    d = syn.scales(seed, N, K // 256)
    x = syn.activations(seed, M, K, heavy=prologue)
    s = syn.act_scale(seed) if prologue else 0.0
    qs, _ = oracle.pack(codes)
    y, t = oracle.matvec(x, qs, d, K, s)
    xv = (x.astype(np.float64) if not prologue else
          np.clip(np.rint(x.astype(np.float32) * (np.float32(1) / np.float32(s))), -128, 127)
          .astype(np.float64) * np.float64(np.float32(s)))
    W = _dense_from_codes(codes, d)
    y_np = xv @ W.T
    t_np = np.abs(xv) @ np.abs(W).T  # |W| = d wherever the code is not 1
    assert np.all(np.abs(y - y_np) <= 1e-12 * t + 1e-300)
    # tolerance sum counts zero codes too: it is >= the dense |W||x|
    assert np.all(t >= t_np * (1 - 1e-12))
    t_full = np.abs(xv) @ np.repeat(d.astype(np.float64), 256, axis=1).T
    assert np.allclose(t, t_full, rtol=1e-12, atol=0)


@pytest.mark.parametrize("prologue", [False, True])
def test_matvec_f64_within_rounding_of_exact_int128(prologue):
    for seed, (M, N, K) in [(0, (1, 32, 512)), (1, (1, 256, 4096)), (3, (2, 8, 16384))]:
        codes = syn.codes(seed, N, K)
        d = syn.scales(seed, N, K // 256)
        x = syn.activations(seed, M, K, heavy=True)
        s = syn.act_scale(seed) if prologue else 0.0
        qs, _ = oracle.pack(codes)
        y, t = oracle.matvec(x, qs, d, K, s)
        ye = oracle.matvec_exact(x, qs, d, K, s)
        assert np.all(np.abs(y - ye) <= K * 2.0 ** -52 * t + 1e-300)


def test_matvec_one_hot_rows_are_exact():
    N, K = 40, 768
    codes = syn.codes(7, N, K)
    d = syn.scales(7, N, K // 256)
    qs, _ = oracle.pack(codes)
    ks = [0, 1, 2, 3, 255, 256, 511, 513, 767]
    x = np.zeros((len(ks), K), dtype=np.float16)
    for i, k in enumerate(ks):
        x[i, k] = 1.0
    y, _ = oracle.matvec(x, qs, d, K)
    for i, k in enumerate(ks):
        want = d[:, k // 256].astype(np.float64) * (codes[:, k].astype(np.float64) - 1)
        assert np.array_equal(y[i], want)


def test_matvec_all_ones_block_counts_codes():
    N, K = 24, 1024
    codes = syn.codes(8, N, K)
    d = syn.scales(8, N, K // 256)
    qs, _ = oracle.pack(codes)
    for b in range(K // 256):
        x = np.zeros((1, K), dtype=np.float16)
        x[0, 256 * b:256 * (b + 1)] = 1.0
        y, _ = oracle.matvec(x, qs, d, K)
        blk = codes[:, 256 * b:256 * (b + 1)]
        want = d[:, b].astype(np.float64) * ((blk == 2).sum(1) - (blk == 0).sum(1))
        assert np.array_equal(y[0], want)


def test_matvec_single_block_is_textbook_dot_product():
    N, K = 9, 256
    codes = syn.codes(9, N, K)
    d = syn.scales(9, N, 1)
    x = syn.activations(9, 1, K)
    qs, _ = oracle.pack(codes)
    y, _ = oracle.matvec(x, qs, d, K)
    for n in range(N):
        w = float(d[n, 0]) * (codes[n].astype(np.float64) - 1)
        assert abs(y[0, n] - float(np.dot(w, x[0].astype(np.float64)))) <= 1e-13


def _exhaustive_pr1_codes(t):
    """qs[n][j] = P[(n + 32 t + 7 j) mod 81] over the 81 valid byte patterns."""
    pats = [c0 + 4 * c1 + 16 * c2 + 64 * c3
            for c3 in range(3) for c2 in range(3) for c1 in range(3) for c0 in range(3)]
    N, K = 32, 512
    qs = np.array([[pats[(n + 32 * t + 7 * j) % 81] for j in range(K // 4)] for n in range(N)],
                  dtype=np.uint8)
    return qs


def test_matvec_exhaustive_pr1_brute_force():
    """K=512, N=32: every valid byte pattern at every byte position (over the
    three code matrices), distinct exact scales, all 512 one-hot x and random x."""
    N, K = 32, 512
    d = np.array([[(1 + 2 * n + b) / 1024.0 for b in range(2)] for n in range(N)],
                 dtype=np.float16)
    seen = np.zeros((K // 4, 256), dtype=bool)
    for t in range(3):
        qs = _exhaustive_pr1_codes(t)
        for j in range(K // 4):
            seen[j, qs[:, j]] = True
        codes = oracle.unpack(qs, K)
        # brute-force definition, straight from the codes with Python integers
        onehot = np.eye(K, dtype=np.float16)
        y, _ = oracle.matvec(onehot, qs, d, K)
        for k in range(0, K, 37):
            for n in range(N):
                assert y[k, n] == float(d[n, k // 256]) * (int(codes[n, k]) - 1)
        W = _dense_from_codes(codes, d)
        assert np.array_equal(y, W.T)  # one-hot rows read W column by column
        for seed in range(4):
            x = syn.activations(seed, 1, K)
            y, tl = oracle.matvec(x, qs, d, K)
            ye = oracle.matvec_exact(x, qs, d, K)
            assert np.all(np.abs(y - ye) <= K * 2.0 ** -52 * tl)
            assert np.all(np.abs(ye - x.astype(np.float64) @ W.T) <= K * 2.0 ** -52 * tl)
    valid = {c0 + 4 * c1 + 16 * c2 + 64 * c3
             for c3 in range(3) for c2 in range(3) for c1 in range(3) for c0 in range(3)}
    assert all(set(np.nonzero(seen[j])[0]) == valid for j in range(K // 4))


def test_matvec_rows_matches_full():
    N, K = 50, 1024
    codes = syn.codes(12, N, K)
    d = syn.scales(12, N, K // 256)
    x = syn.activations(12, 2, K)
    qs, _ = oracle.pack(codes)
    y, t = oracle.matvec(x, qs, d, K, 0.05)
    rows = np.array([0, 7, 49, 13])
    yr, tr = oracle.matvec_rows(x, qs, d, K, rows, 0.05)
    assert np.array_equal(yr, y[:, rows]) and np.array_equal(tr, t[:, rows])


# --------------------------------------------------------------------- generator
def test_generator_is_deterministic_and_has_the_stated_distribution():
    a = syn.codes(1, 64, 4096)
    b = syn.codes(1, 64, 4096)
    assert np.array_equal(a, b)
    assert not np.array_equal(a, syn.codes(2, 64, 4096))
    assert not np.array_equal(a, syn.codes(1, 64, 4096, linear=1))
    n = a.size
    for v, p in ((0, 0.25), (1, 0.5), (2, 0.25)):
        frac = float((a == v).mean())
        assert abs(frac - p) < 5 * np.sqrt(p * (1 - p) / n)
    d = syn.scales(1, 64, 16).astype(np.float64)
    assert d.min() >= 0.0049 and d.max() <= 0.0501
    x = syn.activations(1, 4, 65536).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01
    xh = syn.activations(1, 4, 65536, heavy=True).astype(np.float64)
    assert 0.007 < (np.abs(xh) > 6).mean() < 0.011
    s = [syn.act_scale(1, linear=i) for i in range(100)]
    assert min(s) >= 0.01 and max(s) <= 0.1


def test_generator_words_equal_sequential_splitmix64():
    """Counter-based words equal the sequential SplitMix64 stream from base."""
    def mix(z):
        z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9 & (2 ** 64 - 1)
        z = (z ^ (z >> 27)) * 0x94D049BB133111EB & (2 ** 64 - 1)
        return z ^ (z >> 31)
    seed, tid = 5, 17
    base = mix(mix(seed) ^ (tid * 0xD1B54A32D192ED03 & (2 ** 64 - 1)))
    state, seq = base, []
    for _ in range(10):
        state = (state + 0x9E3779B97F4A7C15) & (2 ** 64 - 1)
        seq.append(mix(state))
    assert [int(w) for w in syn.words(seed, tid, 10)] == seq
    assert [int(w) for w in syn.words(seed, tid, 4, start=6)] == seq[6:]


def test_generator_torch_code_expansion_matches_numpy():
    import torch
    bits = syn.code_bits(3, syn.tensor_id(2, syn.SLOT_CODE_BITS), 64 * 512 // 4)
    a = syn.codes_from_bits(bits, 64, 512)
    b = syn.codes_from_bits_torch(torch.from_numpy(bits), 64, 512).numpy()
    assert np.array_equal(a, b)
    assert np.array_equal(a, syn.codes(3, 64, 512, linear=2))


# ------------------------------------------------------------- affine int4
def _nibbles(qs):
    """Codes [N, K] from packed bytes, written independently of the oracle:
    byte j holds code 2j in its low nibble and code 2j+1 in its high one."""
    q = np.asarray(qs, dtype=np.uint8)
    out = np.empty((q.shape[0], q.shape[1] * 2), dtype=np.int64)
    out[:, 0::2] = q & 15
    out[:, 1::2] = q >> 4
    return out


def _affine4_case(seed, M, N, K, G, heavy=False):
    qs, s, z = syn.affine4_weights(seed, N, K, G)
    x = syn.activations(seed, M, K, heavy=heavy)
    return x, qs, s, z


@pytest.mark.parametrize("seed,M,N,K,G", [(1, 1, 7, 256, 64), (2, 2, 33, 1024, 128),
                                          (3, 3, 16, 768, 256), (4, 1, 9, 4096, 64)])
def test_affine4_against_numpy_dense(seed, M, N, K, G):
    """The factored form equals the dense product W x with W = s (q - z)
    materialised element by element (numpy, fp64): pins the nibble order,
    the group index, the zero point's sign and the scale."""
    x, qs, s, z = _affine4_case(seed, M, N, K, G, heavy=(seed % 2 == 0))
    y, tol = oracle.affine4(x, qs, s, z, K, G)
    gi = np.arange(K) // G
    W = s.astype(np.float64)[:, gi] * (_nibbles(qs) - z.astype(np.float64)[:, gi])
    ref = x.astype(np.float64) @ W.T
    assert np.all(np.abs(y - ref) <= 1e-12 * tol + 1e-300)
    # the tolerance sum's closed form
    t_ref = np.abs(x.astype(np.float64)) @ (np.abs(s.astype(np.float64))[:, gi]
                                            * (_nibbles(qs) + np.abs(z.astype(np.float64))[:, gi])).T
    assert np.allclose(tol, t_ref, rtol=1e-12, atol=0)


def test_affine4_one_hot_is_exact():
    """x = e_k gives y[n] = s[n][k/G] * (q[n][k] - z[n][k/G]) exactly."""
    N, K, G = 12, 512, 64
    _, qs, s, z = _affine4_case(5, 1, N, K, G)
    q = _nibbles(qs)
    for k in (0, 1, 63, 64, 127, 200, 511):
        x = np.zeros((1, K), dtype=np.float16)
        x[0, k] = 1.0
        want = s.astype(np.float64)[:, k // G] * (q[:, k] - z.astype(np.float64)[:, k // G])
        y, _ = oracle.affine4(x, qs, s, z, K, G)
        assert np.array_equal(y[0], want), k
        assert np.array_equal(oracle.affine4_exact(x, qs, s, z, K, G)[0], want), k


def test_affine4_every_byte_value_in_both_nibble_positions():
    """Row v holds the byte v everywhere: x = e_0 reads its low nibble,
    x = e_1 its high nibble (brute force over all 256 byte values)."""
    N, K, G = 256, 256, 256
    qs = np.repeat(np.arange(256, dtype=np.uint8)[:, None], K // 2, axis=1)
    s = np.full((N, 1), 0.5, dtype=np.float16)
    z = np.full((N, 1), 3.0, dtype=np.float16)
    for k, nib in ((0, np.arange(256) & 15), (1, np.arange(256) >> 4), (255, np.arange(256) >> 4)):
        x = np.zeros((1, K), dtype=np.float16)
        x[0, k] = 1.0
        y, _ = oracle.affine4(x, qs, s, z, K, G)
        assert np.array_equal(y[0], 0.5 * (nib - 3.0)), k


def test_affine4_unit_scale_zero_point_zero_is_integer_dot():
    """s = 1, z = 0: y = sum_k q_k x_k, the textbook dot product (numpy)."""
    M, N, K, G = 2, 10, 512, 128
    x, qs, _, _ = _affine4_case(6, M, N, K, G)
    s = np.ones((N, K // G), dtype=np.float16)
    z = np.zeros((N, K // G), dtype=np.float16)
    y, _ = oracle.affine4(x, qs, s, z, K, G)
    ref = x.astype(np.float64) @ _nibbles(qs).T.astype(np.float64)
    assert np.array_equal(y, ref)  # every partial sum is exact in fp64


def test_affine4_code_equal_to_integer_zero_point_gives_zero():
    """Every code equal to an integer zero point: W = 0, so y = 0 exactly,
    whatever x and s are."""
    N, K, G = 6, 512, 64
    x = syn.activations(7, 2, K, heavy=True)
    v = np.arange(N) % 16
    qs = np.repeat((v | (v << 4)).astype(np.uint8)[:, None], K // 2, axis=1)
    s = syn.scales(7, N, K // G)
    z = np.repeat(v.astype(np.float16)[:, None], K // G, axis=1)
    y, _ = oracle.affine4(x, qs, s, z, K, G)
    assert np.all(y == 0.0)
    assert np.all(oracle.affine4_exact(x, qs, s, z, K, G) == 0.0)


def test_affine4_exact_against_fractions_and_f64_within_rounding():
    """The exact dense form equals rational arithmetic (Python fractions) on
    a tiny case, and the fp64 factored form is within K * 2^-52 * tol of it."""
    from fractions import Fraction
    M, N, K, G = 1, 3, 256, 64
    x, qs, s, z = _affine4_case(8, M, N, K, G, heavy=True)
    q = _nibbles(qs)
    ye = oracle.affine4_exact(x, qs, s, z, K, G)
    for n in range(N):
        acc = Fraction(0)
        for k in range(K):
            acc += (Fraction(float(s[n, k // G])) * (q[n, k] - Fraction(float(z[n, k // G])))
                    * Fraction(float(x[0, k])))
        assert ye[0, n] == float(acc)
    x, qs, s, z = _affine4_case(9, 2, 40, 4096, 128, heavy=True)
    y, tol = oracle.affine4(x, qs, s, z, 4096, 128)
    ye = oracle.affine4_exact(x, qs, s, z, 4096, 128)
    assert np.all(np.isfinite(ye))
    assert np.all(np.abs(y - ye) <= 4096 * 2.0 ** -52 * tol)


def test_affine4_rows_matches_full():
    x, qs, s, z = _affine4_case(10, 2, 50, 1024, 64)
    y, t = oracle.affine4(x, qs, s, z, 1024, 64)
    rows = np.array([0, 7, 49, 23])
    yr, tr = oracle.affine4_rows(x, qs, s, z, 1024, 64, rows)
    assert np.array_equal(yr, y[:, rows]) and np.array_equal(tr, t[:, rows])


def test_affine4_generator_distribution():
    qs, s, z = syn.affine4_weights(1, 64, 4096, 128)
    q = _nibbles(qs)
    counts = np.bincount(q.reshape(-1), minlength=16) / q.size
    assert np.all(np.abs(counts - 1 / 16) < 0.005)
    assert s.dtype == np.float16 and z.dtype == np.float16
    assert 0.0 <= float(z.min()) and float(z.max()) <= 15.0 and float(z.std()) > 3.0
    assert np.array_equal(syn.affine4_weights(1, 64, 4096, 128)[0], qs)
