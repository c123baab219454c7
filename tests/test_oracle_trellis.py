"""Pins of the oracle's bitstream / trellis-state layer against what the pages fix.

Sources: "Trellis Quantization" (Lecture 1b) Part eight (16-bit window at bit
K*t, random access, tail-biting circular stream of exactly 256*K bits) and
"ExLlamaV3 & EXL3 Deep Dive" Section 3 (the shift-register transition equation).
None of these tests re-types the oracle's formula: they use closed forms for
one-bit streams, a hand-derived worked example, and an independent big-integer
rotation of the circular stream.
"""
import os

import numpy as np
import pytest

from oracle import exl3_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


@pytest.mark.parametrize("K", range(1, 9))
def test_single_set_bit_closed_form(K):
    """Stream with only bit p set: s_t != 0 iff the offset d = (p - K t) mod 256K
    is < 16, and then s_t = 2**(15 - d).  Every p, every t."""
    nbits = 256 * K
    nw = 8 * K
    p = np.arange(nbits)
    words = np.zeros((nbits, nw), dtype=np.uint32)
    words[p, p // 32] = (np.uint32(1) << (31 - (p % 32)).astype(np.uint32))
    st = O.tile_states(words, K)                    # [nbits, 256]
    t = np.arange(256)
    d = (p[:, None] - K * t[None, :]) % nbits
    expect = np.where(d < 16, 1 << (15 - np.minimum(d, 15)), 0)
    np.testing.assert_array_equal(st, expect)


def test_worked_example_bit200():
    """Lecture 1b Part eight: the 100th weight at K=2 starts at bit 200."""
    spec = {}
    states = {}
    zero = []
    for line in open(os.path.join(GOLDEN, "bit200_k2.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *rest = line.split()
        if key == "state":
            states[int(rest[0])] = int(rest[1], 16)
        elif key == "zero_steps":
            for r in rest:
                a, b = r.split("-")
                zero.extend(range(int(a), int(b) + 1))
        else:
            spec[key] = rest[0]
    K = int(spec["K"])
    start = int(spec["set_bits_start"])
    pattern = int(spec["pattern"], 16)
    bits = np.zeros(256 * K, dtype=np.uint8)
    for i in range(16):
        bits[start + i] = (pattern >> (15 - i)) & 1
    words = np.zeros(8 * K, dtype=np.uint32)
    for j in range(256 * K):
        if bits[j]:
            words[j // 32] |= np.uint32(1 << (31 - j % 32))
    st = O.tile_states(words, K)
    for t, v in states.items():
        assert st[t] == v, (t, hex(int(st[t])), hex(v))
    assert np.all(st[zero] == 0)


def _stream_int(words):
    v = 0
    for w in words:
        v = (v << 32) | int(w)
    return v


@pytest.mark.parametrize("K", range(1, 9))
def test_circular_rotation_and_transition(K):
    """Independent formulation: treat the tile's stream as one 256K-bit integer,
    rotate it left by K*t (tail-biting = circular) and read the top 16 bits.
    Then check the Deep Dive transition s_{t+1} = ((s_t << K) & 0xFFFF) | u_t
    for every t, including the wrap 255 -> 0."""
    rng = _rng(100 + K)
    nbits = 256 * K
    for _ in range(4):
        words = rng.integers(0, 1 << 32, size=8 * K, dtype=np.uint64).astype(np.uint32)
        st = O.tile_states(words, K)
        v = _stream_int(words)
        full = (1 << nbits) - 1
        for t in range(256):
            r = K * t
            rot = ((v << r) | (v >> (nbits - r))) & full if r else v
            assert int(st[t]) == rot >> (nbits - 16)
        for t in range(256):
            nxt = int(st[(t + 1) % 256])
            # u_t: the K stream bits right after s_t's window, read circularly
            u = 0
            for i in range(K):
                j = (K * t + 16 + i) % nbits
                u = (u << 1) | ((v >> (nbits - 1 - j)) & 1)
            assert nxt == (((int(st[t]) << K) & 0xFFFF) | u)


def test_states_are_16_bit():
    rng = _rng(7)
    for K in range(1, 9):
        words = rng.integers(0, 1 << 32, size=(16, 8 * K), dtype=np.uint64).astype(np.uint32)
        st = O.tile_states(words, K)
        assert st.max() < (1 << 16)


def test_all_ones_and_all_zeros_streams():
    """Degenerate streams: all-zero bits give state 0 everywhere; all-one bits
    give 0xFFFF everywhere (every window is full of ones)."""
    for K in range(1, 9):
        z = np.zeros(8 * K, dtype=np.uint32)
        o = np.full(8 * K, 0xFFFFFFFF, dtype=np.uint32)
        assert np.all(O.tile_states(z, K) == 0)
        assert np.all(O.tile_states(o, K) == 0xFFFF)


def test_tile_placement_row_major():
    """Reading: step t of tile (I, J) is element (16I + t//16, 16J + t%16).
    Build codes where exactly one tile holds a non-trivial stream and check that
    only that 16x16 block of W-hat differs from the all-zero-state value, with
    step t landing at (t//16, t%16)."""
    K, m, n = 2, 128, 256
    nt = (m // 16) * (n // 16)
    codes = np.zeros((nt, 8 * K), dtype=np.uint32)
    I, J = 3, 11
    rng = _rng(3)
    codes[I * (n // 16) + J] = rng.integers(0, 1 << 32, size=8 * K, dtype=np.uint64).astype(np.uint32)
    for cb in (O.CB_3INST, O.CB_1MAD):
        W = O.decode_tiles(codes.ravel(), K, cb, m, n)
        w0 = O.decode_states(np.zeros(1, dtype=np.uint32), cb)[0]
        st = O.tile_states(codes[I * (n // 16) + J], K)
        vals = O.decode_states(st, cb)
        block = W[16 * I:16 * I + 16, 16 * J:16 * J + 16]
        np.testing.assert_array_equal(block.ravel(), vals)   # t = 16 r + c
        mask = np.ones_like(W, dtype=bool)
        mask[16 * I:16 * I + 16, 16 * J:16 * J + 16] = False
        assert np.all(W[mask] == w0)
