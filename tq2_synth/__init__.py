"""Seeded synthetic inputs for the ternary (TQ2_0-style) matvec.

This module is shared by the CPU oracle side and the CUDA side of the test
suite and the benchmark.  It draws random numbers and nothing else: it holds
none of the method's arithmetic (no packing, no dequantisation, no
quantisation of activations, no matvec).

Random stream
-------------
Every tensor is a counter-based stream keyed by ``(seed, tensor_id)``.  Word
``i`` of a stream is the SplitMix64 output function ("mix") applied to
``base + (i + 1) * GAMMA`` where ``GAMMA = 0x9E3779B97F4A7C15`` and
``base = mix(mix(seed) ^ (tensor_id * 0xD1B54A32D192ED03))``; this equals the
i-th output of the sequential SplitMix64 generator started at state ``base``
(Steele, Lea, Flood, "Fast splittable pseudorandom number generators",
OOPSLA 2014).  Uniform doubles take the top 53 bits; normals use the
Box-Muller transform.

Distributions (the workloads of the BitCPM ternary page: MiniCPM4-8B shaped
linears, 2-bit codes in {0,1,2}, one fp16 scale per 256-element block)
------------------------------------------------------------------------------
* codes: i.i.d. with P(1) = 1/2 and P(0) = P(2) = 1/4, drawn as the sum of two
  fair random bits (so every byte of the packed weights is random);
* scales d_b: fp16(U[0.005, 0.05]);
* activations x: fp16(N(0, 1)); the heavy-tailed variant replaces each entry,
  with probability 0.01, by fp16(50 * z) with z ~ N(0, 1);
* static activation scale s: fp32(U[0.01, 0.1]), one per linear.

Tensor ids: a linear with index ``L`` uses ``8 * L + slot`` with the slots
below, so every linear of a multi-linear workload has its own streams.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "SLOT_CODE_BITS", "SLOT_SCALES", "SLOT_X", "SLOT_HEAVY_SEL", "SLOT_HEAVY_Z",
    "SLOT_ACT_SCALE", "SLOT_DENSE", "SLOT_OUT_SCALE",
    "tensor_id", "words", "uniform", "normal",
    "code_bits", "codes_from_bits", "codes_from_bits_torch", "codes", "scales", "activations",
    "act_scale", "dense_normal", "small_int_activations", "pow2_scales",
]

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_KEY = np.uint64(0xD1B54A32D192ED03)

SLOT_CODE_BITS = 0
SLOT_SCALES = 1
SLOT_X = 2
SLOT_HEAVY_SEL = 3
SLOT_HEAVY_Z = 4
SLOT_ACT_SCALE = 5
SLOT_DENSE = 6
SLOT_OUT_SCALE = 7
SLOT_ZERO_POINT = 8
SLOT_EXACT_X = 9
SLOT_EXACT_D = 10


def tensor_id(linear: int, slot: int) -> int:
    """Stream id of ``slot`` for the linear with index ``linear``."""
    return 8 * int(linear) + int(slot)


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _base(seed: int, tid: int) -> np.uint64:
    s = _mix(np.array([np.uint64(seed & 0xFFFFFFFFFFFFFFFF)], dtype=np.uint64))[0]
    t = np.uint64(tid & 0xFFFFFFFFFFFFFFFF) * _KEY
    return _mix(np.array([s ^ t], dtype=np.uint64))[0]


def words(seed: int, tid: int, n: int, start: int = 0) -> np.ndarray:
    """Words ``start .. start+n-1`` of stream ``(seed, tid)`` as uint64."""
    with np.errstate(over="ignore"):
        i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        return _mix(_base(seed, tid) + i * GAMMA)


def uniform(seed: int, tid: int, n: int) -> np.ndarray:
    """n doubles in [0, 1) from the top 53 bits of each word."""
    return (words(seed, tid, n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(seed: int, tid: int, n: int) -> np.ndarray:
    """n standard normals (Box-Muller on pairs of uniforms; cosine branch)."""
    u = uniform(seed, tid, 2 * n)
    u1 = 1.0 - u[0::2]  # (0, 1]
    u2 = u[1::2]
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


def code_bits(seed: int, tid: int, nbytes: int) -> np.ndarray:
    """``nbytes`` random bytes: bits 2j and 2j+1 of byte i feed code 4i+j."""
    nw = (nbytes + 7) // 8
    return words(seed, tid, nw).view(np.uint8)[:nbytes].copy()


def codes_from_bits(bits: np.ndarray, n: int, k: int) -> np.ndarray:
    """Codes [n, k] int8 in {0,1,2}: code 4i+j = bit(2j) + bit(2j+1) of byte i.

    The sum of two fair bits gives P(1) = 1/2, P(0) = P(2) = 1/4.
    """
    b = bits.reshape(n, k // 4)
    out = np.empty((n, k // 4, 4), dtype=np.int8)
    for j in range(4):
        out[:, :, j] = ((b >> (2 * j)) & 1) + ((b >> (2 * j + 1)) & 1)
    return out.reshape(n, k)


def codes_from_bits_torch(bits, n: int, k: int):
    """Same as ``codes_from_bits`` for a torch uint8 tensor (any device)."""
    import torch
    b = bits.reshape(n, k // 4)
    out = torch.empty((n, k // 4, 4), dtype=torch.int8, device=bits.device)
    for j in range(4):
        out[:, :, j] = (((b >> (2 * j)) & 1) + ((b >> (2 * j + 1)) & 1)).to(torch.int8)
    return out.reshape(n, k)


def codes(seed: int, n: int, k: int, linear: int = 0) -> np.ndarray:
    """Ternary codes [n, k] int8 for the given linear; k must be a multiple of 4."""
    if k % 4:
        raise ValueError("k must be a multiple of 4")
    bits = code_bits(seed, tensor_id(linear, SLOT_CODE_BITS), n * k // 4)
    return codes_from_bits(bits, n, k)


def scales(seed: int, n: int, nblocks: int, linear: int = 0,
           lo: float = 0.005, hi: float = 0.05) -> np.ndarray:
    """Block scales [n, nblocks] as fp16, fp16(U[lo, hi])."""
    u = uniform(seed, tensor_id(linear, SLOT_SCALES), n * nblocks)
    return (lo + (hi - lo) * u).astype(np.float16).reshape(n, nblocks)


def activations(seed: int, m: int, k: int, linear: int = 0,
                heavy: bool = False) -> np.ndarray:
    """Activations x [m, k] fp16 ~ N(0,1); heavy: 1% of entries are 50*z."""
    z = normal(seed, tensor_id(linear, SLOT_X), m * k)
    if heavy:
        sel = uniform(seed, tensor_id(linear, SLOT_HEAVY_SEL), m * k) < 0.01
        big = 50.0 * normal(seed, tensor_id(linear, SLOT_HEAVY_Z), m * k)
        z = np.where(sel, big, z)
    return z.astype(np.float16).reshape(m, k)


def act_scale(seed: int, linear: int = 0) -> float:
    """Static per-linear activation scale s = fp32(U[0.01, 0.1])."""
    u = uniform(seed, tensor_id(linear, SLOT_ACT_SCALE), 1)[0]
    return float(np.float32(0.01 + 0.09 * u))


def out_scale(seed: int, linear: int = 0) -> float:
    """Static per-linear output scale s_o = fp32(U[0.01, 0.1])."""
    u = uniform(seed, tensor_id(linear, SLOT_OUT_SCALE), 1)[0]
    return float(np.float32(0.01 + 0.09 * u))


def dense_normal(seed: int, n: int, k: int, linear: int = 0,
                 sigma: float = 0.02) -> np.ndarray:
    """A generic (not ternary) dense weight [n, k] fp32 ~ N(0, sigma^2)."""
    z = normal(seed, tensor_id(linear, SLOT_DENSE), n * k)
    return (sigma * z).astype(np.float32).reshape(n, k)


# ---------------------------------------------------------------- exact-sum inputs
def small_int_activations(seed: int, m: int, k: int, linear: int = 0,
                          amax: int = 2, exp: int = -2) -> np.ndarray:
    """x [m, k] fp16 with every entry an integer in [-amax, amax] times 2^exp
    (uniform on the integers).  With power-of-two scales every partial sum of
    the matvec is then an exact fp32 value at the sizes used here."""
    u = uniform(seed, tensor_id(linear, SLOT_EXACT_X), m * k)
    a = np.floor(u * (2 * amax + 1)) - amax
    return (a * 2.0 ** exp).astype(np.float16).reshape(m, k)


def pow2_scales(seed: int, n: int, nblocks: int, linear: int = 0,
                emin: int = -4, emax: int = 0) -> np.ndarray:
    """Block scales [n, nblocks] fp16, each 2^e with e uniform on [emin, emax]."""
    u = uniform(seed, tensor_id(linear, SLOT_EXACT_D), n * nblocks)
    e = emin + np.floor(u * (emax - emin + 1))
    return np.exp2(e).astype(np.float16).reshape(n, nblocks)


# ---------------------------------------------------------------- affine int4
def affine4_weights(seed: int, n: int, k: int, g: int, linear: int = 0):
    """Affine-int4 weights for one linear: (qs [n, k/2] uint8, s [n, k/g] fp16,
    z [n, k/g] fp16).  Every byte is random, so the 4-bit codes are i.i.d.
    uniform on 0..15; s = fp16(U[0.005, 0.05]) as the ternary block scales;
    z = fp16(U[0, 15]), a real zero point anywhere in the code range."""
    qs = code_bits(seed, tensor_id(linear, SLOT_CODE_BITS), n * k // 2).reshape(n, k // 2)
    sc = scales(seed, n, k // g, linear=linear)
    u = uniform(seed, tensor_id(linear, SLOT_ZERO_POINT), n * (k // g))
    z = (15.0 * u).astype(np.float16).reshape(n, k // g)
    return qs, sc, z
