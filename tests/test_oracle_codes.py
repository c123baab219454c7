"""Pins of the oracle's computed codes (3INST, 1MAD) and its binary16 rounding.

Source: "Trellis Quantization" (Lecture 1b) Part nine.  The pages describe the
codes' structure in words and print no constants and no decoded values, so
these tests check every one of the 2**16 states against properties the
structure fixes: the bit fields of the two 3INST halves, the byte-sum of 1MAD,
ranges, monotonicity, and first/second moments against closed forms.  Binary16
conversions are checked against CPython's own IEEE half packing (``struct``
format 'e'), an implementation independent of numpy's.
"""
import math
import struct
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np

from oracle import exl3_oracle as O

ALL = np.arange(1 << 16, dtype=np.uint32)


def _half_bits_to_float(b):
    return struct.unpack("<e", struct.pack("<H", int(b)))[0]


def _round_to_half(v):
    return struct.unpack("<H", struct.pack("<e", float(v)))[0]


def test_binary16_rounding_matches_cpython():
    rng = np.random.default_rng(11)
    v = np.concatenate([
        rng.normal(0, 2, 50000),
        rng.uniform(-8, 8, 50000),
        # exact ties between neighbouring halves in [1, 4)
        (np.arange(1024, 4096, dtype=np.float64) + 0.5) / 1024.0,
    ])
    ours = v.astype(np.float16).view(np.uint16)
    ref = np.array([_round_to_half(x) for x in v], dtype=np.uint16)
    np.testing.assert_array_equal(ours, ref)


def test_lcg_low_half_is_bijection():
    """A is odd, so s -> (A s + B) mod 2**16 permutes the 16-bit states."""
    x = O.lcg(ALL)
    assert O.LCG_A % 2 == 1
    assert len(np.unique(x & 0xFFFF)) == 1 << 16


def test_lcg_is_one_multiply_add_mod_2_32():
    """Spot values of one 32-bit multiply-add, computed with Python integers."""
    for s in (0, 1, 2, 0x1234, 0xFFFF):
        assert int(O.lcg(np.array([s], dtype=np.uint32))[0]) == (O.LCG_A * s + O.LCG_B) % (1 << 32)


def test_3inst_half_fields():
    """Step two: each half keeps its sign bit, the two low exponent bits and the
    ten mantissa bits of the LCG output; its biased exponent lands in 12..15,
    i.e. |half| in [1/8, 2).  Checked field by field on all 2**16 states."""
    x = O.lcg(ALL).astype(np.int64)
    h = (x & O.MASK_3INST) ^ O.MAGIC_3INST
    for half, src in ((h & 0xFFFF, x & 0xFFFF), (h >> 16, x >> 16)):
        assert np.all((half >> 15) == (src >> 15))            # sign kept
        assert np.all((half & 0x3FF) == (src & 0x3FF))        # mantissa kept
        exp = (half >> 10) & 0x1F
        assert exp.min() >= 12 and exp.max() <= 15
        assert np.all((exp & 3) == ((src >> 10) & 3))         # two low exponent bits kept
        mags = np.abs(np.array([_half_bits_to_float(b) for b in half[:4096]]))
        assert mags.min() >= 0.125 and mags.max() < 2.0


def test_3inst_sum_is_one_rounded_half_add():
    """Step three: w = round_half(lo + hi), with lo/hi read and the sum rounded by
    CPython's binary16 routines."""
    w = O.code_3inst(ALL).view(np.uint16)
    x = O.lcg(ALL).astype(np.int64)
    h = (x & O.MASK_3INST) ^ O.MAGIC_3INST
    for i in range(0, 1 << 16, 7):
        lo = _half_bits_to_float(h[i] & 0xFFFF)
        hi = _half_bits_to_float(h[i] >> 16)
        assert w[i] == _round_to_half(lo + hi), i


def test_3inst_moments_closed_form():
    """Each half is sign * 2**e * (1 + f/1024) with e uniform on {-3..0} and f
    uniform on 0..1023 (the low half exactly so, since the low 16 LCG bits are a
    permutation of the states).  E[half^2] = 1/4 * sum 4**e * E[(1+f/1024)^2]."""
    Eu = Fraction(1023, 2048)
    Eu2 = Fraction(1023 * 2047, 6 * 1024 * 1024)
    Eh2 = Fraction(1, 4) * sum(Fraction(4) ** e for e in range(-3, 1)) * (1 + 2 * Eu + Eu2)
    x = O.lcg(ALL).astype(np.int64)
    h = (x & O.MASK_3INST) ^ O.MAGIC_3INST
    lo = (h & 0xFFFF).astype(np.uint16).view(np.float16).astype(np.float64)
    assert abs(np.mean(lo ** 2) - float(Eh2)) < 1e-12
    assert abs(np.mean(lo)) < 1e-12
    w = O.code_3inst(ALL).astype(np.float64)
    assert np.all(np.isfinite(w)) and np.abs(w).max() < 4.0
    assert abs(w.mean()) < 0.02
    assert abs(w.var() / (2 * float(Eh2)) - 1) < 0.03


def test_1mad_constant_is_binary32_nearest():
    getcontext().prec = 60
    exact = Decimal(1) / Decimal(21845).sqrt()
    c = O.ONE_MAD_SCALE_F32
    assert c.dtype == np.float32
    up = np.nextafter(c, np.float32(1))
    dn = np.nextafter(c, np.float32(0))
    ec = abs(Decimal(float(c)) - exact)
    assert ec <= abs(Decimal(float(up)) - exact) and ec <= abs(Decimal(float(dn)) - exact)


def test_1mad_closed_form_moments():
    """Four i.i.d. uniform bytes: mean 510, variance 4*(256^2-1)/12 = 21845."""
    assert O.ONE_MAD_CENTRE == 4 * Fraction(255, 2)
    assert O.ONE_MAD_VARIANCE == 4 * Fraction(256 ** 2 - 1, 12)


def test_1mad_is_centred_scaled_byte_sum():
    """w * sqrt(21845) + 510 recovers the byte sum of the LCG output to within the
    two roundings; |w| <= 510/sqrt(21845); w is monotone in the byte sum;
    the sample moments over all states are close to 0 and 1."""
    x = O.lcg(ALL)
    S = np.array([sum((int(v) >> (8 * k)) & 0xFF for k in range(4)) for v in x[::5]])
    w = O.code_1mad(ALL)[::5].astype(np.float64)
    approx = w * math.sqrt(21845) + 510
    # binary16 relative half-ulp 2**-11, plus binary32: bound on |S - approx|
    assert np.all(np.abs(approx - S) <= 510 * 2.0 ** -10 + 1e-6)
    assert np.abs(w).max() <= 510 / math.sqrt(21845) * (1 + 2 ** -10)
    order = np.argsort(S, kind="stable")
    assert np.all(np.diff(w[order]) >= 0)
    wall = O.code_1mad(ALL).astype(np.float64)
    assert abs(wall.mean()) < 0.02
    assert abs(wall.var() - 1.0) < 0.05


def test_1mad_rounding_steps():
    """(S-510) is exact in binary32; the binary32 product is rounded once, then
    once more to binary16 (checked with Python fractions + CPython packing)."""
    c = Fraction(float(O.ONE_MAD_SCALE_F32))
    x = O.lcg(ALL)
    w = O.code_1mad(ALL).view(np.uint16)
    for i in range(0, 1 << 16, 97):
        S = sum((int(x[i]) >> (8 * k)) & 0xFF for k in range(4))
        prod = float(np.float32(float((S - 510) * c)))  # one binary32 rounding of the exact product
        assert w[i] == _round_to_half(prod), i


def test_codebook_dispatch():
    st = np.array([0, 1, 0xFFFF], dtype=np.uint32)
    np.testing.assert_array_equal(O.decode_states(st, 0), O.code_3inst(st))
    np.testing.assert_array_equal(O.decode_states(st, 1), O.code_1mad(st))
    np.testing.assert_array_equal(O.decode_states(st, 2), O.code_mcg(st))
    np.testing.assert_array_equal(O.decode_states(st, 3), O.code_mul1(st))
    try:
        O.decode_states(st, 4)
    except ValueError:
        pass
    else:
        raise AssertionError("unknown codebook must raise")


def test_mcg_generator_is_the_lcg_without_its_constant():
    """x_MCG = A*s mod 2**32, so x_LCG - x_MCG = B (mod 2**32) for every state,
    and the state 0 maps to x = 0, i.e. the two halves 0x3000 = 1/8 each and the
    weight 1/4."""
    x_m = O.mcg(ALL).astype(np.uint64)
    x_l = O.lcg(ALL).astype(np.uint64)
    assert np.all(((x_l - x_m) & 0xFFFFFFFF) == O.LCG_B)
    assert float(O.code_mcg(np.array([0], dtype=np.uint32))[0]) == 0.25
    for s in (1, 2, 12345, 0xFFFF):
        x = (O.LCG_A * s) & 0xFFFFFFFF
        h = (x & O.MASK_3INST) ^ O.MAGIC_3INST
        lo = _half_bits_to_float(h & 0xFFFF)
        hi = _half_bits_to_float(h >> 16)
        assert O.code_mcg(np.array([s], dtype=np.uint32)).view(np.uint16)[0] == _round_to_half(lo + hi)


def test_mcg_moments_match_3inst():
    """Same mask/XOR/add as 3INST on another uniform generator: mean about 0,
    variance about that of 3INST (the closed form of the 3INST test)."""
    w = O.code_mcg(ALL).astype(np.float64)
    w3 = O.code_3inst(ALL).astype(np.float64)
    assert abs(w.mean()) < 0.02
    assert abs(w.var() - w3.var()) < 0.05 * w3.var()


def test_mul1_masked_byte_sum():
    """w = fp16(fp32(S - 126) * fp32(1/sqrt(1365))) with S the sum of the four
    bytes of A*s, each masked to six bits (checked with Python integers, exact
    fractions and CPython's binary16 packing); S spans [0, 252]."""
    c = Fraction(float(O.MUL1_SCALE_F32))
    assert O.MUL1_SCALE_F32 == np.float32(1.0 / math.sqrt(1365))
    w = O.code_mul1(ALL).view(np.uint16)
    sums = []
    for s in range(0, 1 << 16, 89):
        x = (O.LCG_A * s) & 0xFFFFFFFF
        S = sum((x >> (8 * k)) & 0x3F for k in range(4))
        sums.append(S)
        prod = float(np.float32(float((S - 126) * c)))
        assert w[s] == _round_to_half(prod), s
    assert min(sums) >= 0 and max(sums) <= 252


def test_mul1_closed_form_moments():
    """Four uniform 6-bit values: mean 126 and variance 4*(64**2-1)/12 = 1365,
    so the weights have mean about 0 and variance about 1 over all states."""
    assert 4 * 63 / 2 == O.MUL1_CENTRE and 4 * (64 ** 2 - 1) // 12 == O.MUL1_VARIANCE
    w = O.code_mul1(ALL).astype(np.float64)
    assert abs(w.mean()) < 0.02
    assert abs(w.var() - 1.0) < 0.05
    assert np.abs(w).max() <= 126 / math.sqrt(1365) * (1 + 2 ** -10)
