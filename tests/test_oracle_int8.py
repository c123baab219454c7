"""Pins of the oracle's int8-activation path ("Trellis Quantization" Part
eleven: quantized eight-bit activations, the weight affine in a byte sum, one
dp4a per four products).  The quantizer is checked against what symmetric
rounding fixes: the error bound of half a step, the extreme code at the block
maximum, ties to even on constructed halves, zero blocks; the layer against
the fp64 layer on the dequantized activations and the exact integer form of
the byte-sum codes."""
import math
from fractions import Fraction

import numpy as np
import pytest

from oracle import exl3_oracle as O
from trellis_decode_gemv_gb300 import synth


def test_quantizer_error_bound_and_extremes():
    x = synth.activations(4, 512, synth.seed_for(80, 0))
    q, s = O.quantize_act(x)
    assert q.dtype == np.int8 and s.dtype == np.float32 and s.shape == (4, 4)
    xb = x.astype(np.float64).reshape(4, 4, 128)
    qb = q.astype(np.float64).reshape(4, 4, 128)
    err = np.abs(xb - qb * s.astype(np.float64)[:, :, None])
    assert np.all(err <= s.astype(np.float64)[:, :, None] * (0.5 + 1e-6))
    assert np.abs(q).max() == 127
    for r in range(4):
        for b in range(4):
            k = int(np.argmax(np.abs(xb[r, b])))
            assert abs(int(qb[r, b, k])) == 127
            assert s[r, b] == np.float32(np.float32(np.abs(xb[r, b]).max()) / np.float32(127))


def test_quantizer_ties_to_even_and_zero_blocks():
    """With the block maximum 127 the scale is exactly 1, so halves are exact
    ties: 0.5 -> 0, 1.5 -> 2, 2.5 -> 2, -3.5 -> -4."""
    x = np.zeros((2, 256), dtype=np.float16)
    x[0, :6] = [127, 0.5, 1.5, 2.5, -3.5, -126.5]
    q, s = O.quantize_act(x)
    assert s[0, 0] == 1.0
    assert list(q[0, :6]) == [127, 0, 2, 2, -4, -126]
    assert s[0, 1] == 0 and s[1, 0] == 0 and s[1, 1] == 0
    assert np.all(q[1] == 0) and np.all(q[0, 128:] == 0)


def test_quantizer_matches_exact_rational_rounding():
    """Each q is the nearest integer to the binary32 quotient, checked with
    exact fractions on a sample."""
    x = synth.activations(1, 128, synth.seed_for(80, 1))
    q, s = O.quantize_act(x)
    sc = Fraction(float(s[0, 0]))
    for j in range(0, 128, 5):
        quot = float(np.float32(Fraction(float(x[0, j])) / sc))  # one binary32 rounding
        assert int(q[0, j]) == round(quot)  # Python rounds ties to even


@pytest.mark.parametrize("cb", [O.CB_1MAD, O.CB_MUL1])
def test_int8_layer_is_the_layer_on_dequantized_activations(cb):
    m, n, K, M = 256, 384, 2, 3
    inp = synth.layer_inputs(m, n, K, M, config=81, index=cb)
    xt = O.rht(inp["x"].astype(np.float64), inp["s_in"]).astype(np.float16)
    q, s = O.quantize_act(xt)
    y8 = O.layer_forward_int8(inp["codes"], K, cb, m, n, inp["s_out"], inp["scales"], q, s)
    xhat = (q.astype(np.float64).reshape(M, 3, 128) * s.astype(np.float64)[:, :, None]).reshape(M, n)
    y = O.layer_forward(inp["codes"], K, cb, m, n, None, inp["s_out"], inp["scales"], xhat)
    np.testing.assert_allclose(y8, y, rtol=1e-12, atol=1e-12)
    # and close to the unquantized layer: int8 steps of max/127 per block
    yf = O.layer_forward(inp["codes"], K, cb, m, n, inp["s_in"], inp["s_out"], inp["scales"], inp["x"])
    rel = np.linalg.norm(y8 - yf) / np.linalg.norm(yf)
    assert 1e-4 < rel < 2e-2, rel
    with pytest.raises(ValueError):
        O.layer_forward_int8(inp["codes"], K, O.CB_3INST, m, n, inp["s_out"], inp["scales"], q, s)


@pytest.mark.parametrize("cb,centre,var", [(O.CB_1MAD, 510, 21845), (O.CB_MUL1, 126, 1365)])
def test_byte_sum_weights_times_int8_are_integer_dot_products(cb, centre, var):
    """The identity the dp4a path rests on, per weight and exactly: the
    defined weight is binary16((S - centre) * C); (S - centre) * q is the
    integer dp4a(bytes, q q q q) - centre * q, and the defined weight times q
    differs from C * that integer by the binary16 rounding only."""
    states = np.arange(0, 1 << 16, 37, dtype=np.uint32)
    w = O.decode_states(states, cb).astype(np.float64)
    x = (O.mcg(states) if cb == O.CB_MUL1 else O.lcg(states)).astype(np.int64)
    mask = 0x3F if cb == O.CB_MUL1 else 0xFF
    S = sum((x >> (8 * k)) & mask for k in range(4))
    C = 1.0 / math.sqrt(var)
    q = np.int64(-93)
    dp4a = sum(((x >> (8 * k)) & mask) * q for k in range(4))
    assert np.all(dp4a == S * q)
    np.testing.assert_allclose(w * q, (dp4a - centre * q) * C, rtol=2.0 ** -10, atol=1e-12)
