"""Pins of the computed codes' quality: the oracle's Viterbi encoder and the
mean-squared errors the pages print for a Gaussian source at two bits per
weight ("Trellis Quantization: Trading Memory for Cheap Compute", Part nine:
rate-distortion bound 1/16 = 0.0625, Lloyd-Max 0.118, E8 0.089, the trellis
with the three-instruction code about 0.069, and "the computed codes do
essentially as well as a truly random lookup table would").

The encoder itself is checked first: its Viterbi search against brute force on
a tiny trellis, and its tail-biting streams against the oracle's own decoder.
"""
import itertools

import numpy as np
import pytest

from oracle import exl3_encoder as E
from oracle import exl3_oracle as O


def _brute_force(values, target, K, L, start=None, forced=None):
    """Cheapest path by enumerating every first state and every appended bit
    sequence."""
    T = len(target)
    best = np.inf
    starts = range(1 << L) if start is None else [start]
    for s0 in starts:
        for bs in itertools.product(range(1 << K), repeat=T - 1):
            if forced and any((bs[t - 1] & m) != v for t, (m, v) in forced.items()):
                continue
            s = s0
            c = (values[s] - target[0]) ** 2
            for t in range(1, T):
                s = ((s << K) | bs[t - 1]) & ((1 << L) - 1)
                c += (values[s] - target[t]) ** 2
            best = min(best, c)
    return best


@pytest.mark.parametrize("dtype,rel", [(np.float64, 1e-12), (np.float32, 1e-5)])
@pytest.mark.parametrize("K,L,T", [(1, 4, 9), (2, 4, 6), (1, 5, 8)])
def test_viterbi_matches_brute_force(K, L, T, dtype, rel):
    rng = np.random.default_rng(100 + 10 * K + L)
    values = rng.normal(size=1 << L)
    target = rng.normal(size=T)
    if dtype == np.float32:  # the brute force sees the same binary32 inputs
        values = values.astype(np.float32).astype(np.float64)
        target = target.astype(np.float32).astype(np.float64)
    states, cost = E.viterbi(values, target, K, L, dtype=dtype)
    assert cost == pytest.approx(_brute_force(values, target, K, L), rel=rel)
    # the returned path is a legal shift-register path with that cost
    for t in range(1, T):
        assert states[t] >> K == states[t - 1] & ((1 << (L - K)) - 1)
    assert np.sum((values[states] - target) ** 2) == pytest.approx(cost, rel=rel)
    # fixed start and forced appended bits
    forced = {T - 1: ((1 << K) - 1, 1), T - 2: (1, 0)}
    states, cost = E.viterbi(values, target, K, L, start=3, forced=forced, dtype=dtype)
    assert states[0] == 3
    assert cost == pytest.approx(_brute_force(values, target, K, L, 3, forced), rel=rel)


@pytest.mark.parametrize("K,cb", [(2, O.CB_3INST), (3, O.CB_1MAD), (1, O.CB_3INST)])
def test_encoded_streams_are_tail_biting_codewords(K, cb):
    """The words the encoder emits decode, through the oracle's circular window
    and computed code, to exactly the path the encoder chose."""
    rng = np.random.default_rng(7 + K)
    values = E.codebook_values(cb)
    target = rng.normal(size=O.STEPS)
    words, states, mse = E.encode_tile(target, values, K)
    assert words.dtype == np.uint32 and words.shape == (8 * K,)
    assert np.array_equal(O.tile_states(words, K).astype(np.int64), states)
    decoded = O.decode_states(O.tile_states(words, K), cb).astype(np.float64)
    scale = np.sqrt(np.mean(O.decode_states(np.arange(1 << 16, dtype=np.uint32), cb).astype(np.float64) ** 2))
    assert np.mean((decoded / scale - target) ** 2) == pytest.approx(mse, rel=1e-9)


def test_lloyd_max_two_bits_matches_the_pages():
    """The measurement itself: a 4-level Lloyd-Max quantizer on the same kind of
    Gaussian samples gives the pages' 0.118 (textbook value 0.1175)."""
    x = np.random.default_rng(3).normal(size=400_000)
    levels, mse = E.lloyd_max(x, 4)
    assert mse == pytest.approx(0.1175, abs=0.002)
    assert np.allclose(np.abs(levels), [1.510, 0.4528, 0.4528, 1.510], atol=0.02)


@pytest.fixture(scope="module")
def gaussian_tiles():
    # 24 tiles = 6144 samples of N(0, 1)
    return np.random.default_rng(2025).normal(size=24 * O.STEPS)


def test_3inst_two_bit_mse(gaussian_tiles):
    """The trellis with the oracle's 3INST code at K = 2: about 0.069, above the
    rate-distortion bound 0.0625 and well below E8's 0.089."""
    mse = E.trellis_mse(E.codebook_values(O.CB_3INST), gaussian_tiles, 2)
    assert 0.0625 < mse < 0.075, mse
    assert mse == pytest.approx(0.069, abs=0.004)


def test_computed_codes_match_a_random_table(gaussian_tiles):
    """Every computed code does about as well as a truly random Gaussian table
    of the same size on the same samples."""
    rng = np.random.default_rng(99)
    table = rng.normal(size=1 << O.L)
    table /= np.sqrt(np.mean(table ** 2))
    ref = E.trellis_mse(table, gaussian_tiles, 2)
    for cb in (O.CB_3INST, O.CB_1MAD, O.CB_MCG, O.CB_MUL1):
        mse = E.trellis_mse(E.codebook_values(cb), gaussian_tiles, 2)
        assert abs(mse - ref) < 0.1 * ref, (cb, mse, ref)


def test_binary32_costs_follow_the_stated_rounding():
    """In float32 mode every path cost is the binary32 evaluation, in order, of
    best + (v - x)^2: recomputed here along the returned path with explicit
    float32 scalars, it matches bit for bit."""
    rng = np.random.default_rng(31)
    K, L, T = 2, 6, 12
    values = rng.normal(size=1 << L).astype(np.float32)
    target = rng.normal(size=T).astype(np.float32)
    states, cost = E.viterbi(values, target, K, L, dtype=np.float32)
    acc = np.float32(0)
    for t in range(T):
        d = np.float32(values[states[t]] - target[t])
        acc = np.float32(acc + np.float32(d * d)) if t else np.float32(d * d)
    assert np.float32(cost) == acc


@pytest.mark.parametrize("K,cb", [(2, O.CB_3INST), (1, O.CB_1MAD)])
def test_binary32_encoding_is_a_tail_biting_codeword(K, cb):
    """The float32 two-pass encoder on raw code values and a target in code
    units: its words decode to its path, and the path's binary32 cost is the
    returned one."""
    rng = np.random.default_rng(41 + K)
    raw = O.decode_states(np.arange(1 << O.L, dtype=np.uint32), cb).astype(np.float32)
    sigma = np.sqrt(np.mean(raw.astype(np.float64) ** 2))
    target = (rng.normal(size=O.STEPS) * sigma).astype(np.float32)
    words, states, mse = E.encode_tile(target, raw, K, dtype=np.float32)
    assert np.array_equal(O.tile_states(words, K).astype(np.int64), states)
    d = raw[states] - target
    assert np.sum(d.astype(np.float64) ** 2) / O.STEPS == pytest.approx(mse, rel=1e-5)
    # same quality as the float64 encoder on the normalized problem
    _, _, mse64 = E.encode_tile(target / sigma, raw / sigma, K)
    assert mse / sigma ** 2 == pytest.approx(mse64, rel=0.05)
