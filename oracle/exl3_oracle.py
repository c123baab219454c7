"""Plain CPU oracle for the bitshift-trellis (QTIP / EXL3) quantized linear layer.

TEST INFRASTRUCTURE ONLY.  The product path (the CUDA library and its Python
binding) never imports, calls or links anything in this module.  Only the test
suite, the smoke check in ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use it.  It shares no code, constant or helper with the CUDA side:
each side writes the definitions below on its own, and the parity tests compare
the two.

Everything is numpy, slow and literal.  Each function follows one passage of the
source pages, named in its docstring:

  [DD]  "ExLlamaV3 & EXL3 Deep Dive" (abrarakhunji.com): Section 2 (randomized
        Hadamard incoherence processing, the runtime identity y = W x) and
        Section 3 (the bitshift-trellis state-transition equation and the
        conceptual decoder).
  [TQ]  "Trellis Quantization: Trading Memory for Cheap Compute" (Lecture 1b):
        Part three (integer budget, the int-to-half splice), Part six (RHT),
        Part eight (the bitshift trellis: 16-bit window, random access, 16x16
        tiles, tail-biting), Part nine (the 3INST and 1MAD computed codes),
        Part eleven (EXL3: 128-wide blockwise rotation; QTIP's whole-vector
        rotation, ``rht_whole``).
  [FG]  "EXL3 field guide" (LLM Cal): per-output-channel scales ("out_scales
        always").

Where the pages leave a step open, the reading taken is stated next to the
constant or function that embodies it.  The codebook constants (LCG multiplier
and increment, 3INST mask and magic) are readings, not printed by the pages; the
codebook *structure* is pinned by the tests in ``tests/test_oracle_*.py``, and
the numerical *quality* of these particular constants by the Viterbi encoder in
``exl3_encoder`` against the mean-squared errors [TQ] Part nine prints for a
Gaussian source at two bits per weight (``tests/test_oracle_encoder.py``).
"""
from __future__ import annotations

import math

import numpy as np

# ----------------------------------------------------------------------------
# Format constants
# ----------------------------------------------------------------------------

#: State width L in bits.  [TQ] Part eight and Part eleven: a 16-bit window.
L = 16
#: A trellis sequence covers one 16x16 tile: 256 steps.  [TQ] Part eight.
TILE = 16
STEPS = TILE * TILE

#: LCG multiplier / increment.  Reading: [TQ] Part nine only says "carefully
#: chosen constants"; the only pair printed anywhere on the pages is the one in
#: the conceptual decoder of [DD] Section 3, so both codes use it.
LCG_A = 0x9E3779B9
LCG_B = 0x7F4A7C15

#: 3INST mask and magic.  Reading of [TQ] Part nine, step two: keep the sign bit
#: and the low bits of each 16-bit half (sign, the two low exponent bits and the
#: ten mantissa bits), then XOR in a constant that pins the biased exponent to
#: 12..15, so every half lies in +-[1/8, 2).
MASK_3INST = 0x8FFF8FFF
MAGIC_3INST = 0x30003000

#: 1MAD centring and scaling.  Reading of [TQ] Part nine ("centred and scaled"):
#: four i.i.d. uniform bytes have mean 4 * 127.5 = 510 and variance
#: 4 * (256**2 - 1) / 12 = 21845, so the weight is (S - 510) / sqrt(21845).
ONE_MAD_CENTRE = 510
ONE_MAD_VARIANCE = 21845
#: 1/sqrt(21845) rounded once to binary32.
ONE_MAD_SCALE_F32 = np.float32(1.0 / math.sqrt(ONE_MAD_VARIANCE))

CB_3INST = 0
CB_1MAD = 1
CB_MCG = 2
CB_MUL1 = 3

#: mul1 masking, centring and scaling.  [TQ] Part eleven and Part twelve: the
#: integer generator multiplies the state by a constant, masks each of the four
#: bytes of the product down to six bits, sums the four bytes (dp4a against a
#: vector of ones) and subtracts a fixed offset, giving an integer in about
#: [-126, 126]; EXL3's mul1 moved to the same masked byte sum, and its weight
#: is an affine function of it.  Reading: the offset is the mean of four
#: uniform 6-bit values, 4 * 31.5 = 126, and the scale makes the variance one:
#: 4 * (64**2 - 1) / 12 = 1365.
MUL1_MASK = 0x3F3F3F3F
MUL1_CENTRE = 126
MUL1_VARIANCE = 1365
#: 1/sqrt(1365) rounded once to binary32.
MUL1_SCALE_F32 = np.float32(1.0 / math.sqrt(MUL1_VARIANCE))

#: Blockwise Hadamard width.  [TQ] Part eleven: EXL3 rotates 128-blocks along
#: each axis.
RHT_BLOCK = 128


# ----------------------------------------------------------------------------
# Bitstream and trellis state  ([TQ] Part eight, [DD] Section 3)
# ----------------------------------------------------------------------------

def tile_bits(words: np.ndarray) -> np.ndarray:
    """Bits of each tile's stream, in stream order.

    ``words`` is uint32 ``[..., 8K]`` (one tile per row of the last axis).  Bit j
    of the stream is bit ``31 - j % 32`` of word ``j // 32`` (MSB-first).

    Reading: [DD] Section 3 shifts new bits in at the low end of the state and
    takes them from the top of the incoming word with a left funnel shift, and
    [TQ] Part eight lays the bits of a sequence "end to end in one long
    string"; most-significant-bit-first inside each 32-bit word is the plainest
    layout consistent with both.
    """
    words = np.asarray(words, dtype=np.uint32)
    shifts = np.arange(31, -1, -1, dtype=np.uint32)
    bits = (words[..., :, None] >> shifts) & np.uint32(1)
    return bits.reshape(*words.shape[:-1], words.shape[-1] * 32).astype(np.uint8)


def tile_states(words: np.ndarray, K: int) -> np.ndarray:
    """Trellis state for every step of every tile.

    [TQ] Part eight: the state at step t is the 16-bit window of the stream that
    starts at bit K*t ("to decode the hundredth weight ... jump straight to bit
    two hundred" at K = 2), and the stream is circular (tail-biting: exactly
    256*K bits per tile, no stored start state):

        s_t = sum_{i=0..15} bit((K*t + i) mod 256K) * 2**(15 - i).

    The first stream bit of the window is the state's most significant bit, so
    s_{t+1} = ((s_t << K) & 0xFFFF) | (next K bits), the transition equation of
    [DD] Section 3.  Returns uint32 ``[..., 256]``.
    """
    nbits = STEPS * K
    words = np.asarray(words, dtype=np.uint32)
    assert words.shape[-1] * 32 == nbits, "a tile holds exactly 8*K words"
    bits = tile_bits(words)
    t = np.arange(STEPS)[:, None]
    i = np.arange(L)[None, :]
    idx = (K * t + i) % nbits                          # [256, 16]
    weights = (np.uint32(1) << (np.uint32(L - 1) - np.arange(L, dtype=np.uint32)))
    win = bits[..., idx].astype(np.uint32)             # [..., 256, 16]
    return (win * weights).sum(axis=-1, dtype=np.uint32)


# ----------------------------------------------------------------------------
# Computed codes  ([TQ] Part nine)
# ----------------------------------------------------------------------------

def lcg(states: np.ndarray) -> np.ndarray:
    """One linear-congruential step on the zero-extended 16-bit state:
    x = (A*s + B) mod 2**32.  [TQ] Part nine, step one (both codes)."""
    s = np.asarray(states, dtype=np.uint64)
    return ((np.uint64(LCG_A) * s + np.uint64(LCG_B)) & np.uint64(0xFFFFFFFF)).astype(np.uint32)


def mcg(states: np.ndarray) -> np.ndarray:
    """The multiplicative generator of MCG and mul1: x = A*s mod 2**32, the LCG
    without its additive constant.  [TQ] Part eleven ("drops the additive
    constant ... and keeps only the multiply").  Reading: the pages do not print
    the multiplier they adopt; the one LCG multiplier they print (A) is used."""
    s = np.asarray(states, dtype=np.uint64)
    return ((np.uint64(LCG_A) * s) & np.uint64(0xFFFFFFFF)).astype(np.uint32)


def _mask_xor_add(x: np.ndarray) -> np.ndarray:
    """Steps two and three of the three-instruction code on a 32-bit x: mask
    and XOR into two binary16 halves, one correctly rounded binary16 add."""
    h = (x & np.uint32(MASK_3INST)) ^ np.uint32(MAGIC_3INST)
    lo = (h & np.uint32(0xFFFF)).astype(np.uint16).view(np.float16)
    hi = (h >> np.uint32(16)).astype(np.uint16).view(np.float16)
    return (lo.astype(np.float64) + hi.astype(np.float64)).astype(np.float16)


def code_mcg(states: np.ndarray) -> np.ndarray:
    """MCG: the three-instruction code with the multiplicative generator.
    [TQ] Part eleven.  Returns float16."""
    return _mask_xor_add(mcg(states))


def code_mul1(states: np.ndarray) -> np.ndarray:
    """mul1: multiply, mask every byte of the product to six bits, sum the four
    bytes, subtract 126, scale by 1/sqrt(1365).  [TQ] Parts eleven and twelve.

    Precision reading as for 1MAD: (S - 126) is exact in binary32, multiplied by
    the binary32 constant with one rounding, then rounded once to binary16.
    Returns float16."""
    x = mcg(states) & np.uint32(MUL1_MASK)
    S = ((x & np.uint32(0xFF)) + ((x >> np.uint32(8)) & np.uint32(0xFF))
         + ((x >> np.uint32(16)) & np.uint32(0xFF)) + (x >> np.uint32(24)))
    centred = (S.astype(np.int64) - MUL1_CENTRE).astype(np.float32)
    return (centred * MUL1_SCALE_F32).astype(np.float32).astype(np.float16)


def code_3inst(states: np.ndarray) -> np.ndarray:
    """3INST: LCG, then mask-and-XOR into two binary16 halves, then one binary16
    add of the two halves.  [TQ] Part nine, steps one to three.

    The add is a single correctly rounded binary16 addition (round to nearest
    even): the exact sum is formed in float64, where it is exact, and rounded
    once.  Returns float16.
    """
    x = lcg(states)
    h = (x & np.uint32(MASK_3INST)) ^ np.uint32(MAGIC_3INST)
    lo = (h & np.uint32(0xFFFF)).astype(np.uint16).view(np.float16)
    hi = (h >> np.uint32(16)).astype(np.uint16).view(np.float16)
    return (lo.astype(np.float64) + hi.astype(np.float64)).astype(np.float16)


def code_1mad(states: np.ndarray) -> np.ndarray:
    """1MAD: LCG, sum of the four bytes of the result, centred and scaled.
    [TQ] Part nine ("runs the same generator, then sums the four bytes").

    Reading of the precision: (S - 510) is exact in binary32, it is multiplied by
    the binary32 constant 1/sqrt(21845) with one binary32 rounding, and the
    product is rounded once to binary16 (both round to nearest even).
    Returns float16.
    """
    x = lcg(states)
    S = ((x & np.uint32(0xFF)) + ((x >> np.uint32(8)) & np.uint32(0xFF))
         + ((x >> np.uint32(16)) & np.uint32(0xFF)) + (x >> np.uint32(24)))
    centred = (S.astype(np.int64) - ONE_MAD_CENTRE).astype(np.float32)
    return (centred * ONE_MAD_SCALE_F32).astype(np.float32).astype(np.float16)


def decode_states(states: np.ndarray, codebook: int) -> np.ndarray:
    if codebook == CB_3INST:
        return code_3inst(states)
    if codebook == CB_1MAD:
        return code_1mad(states)
    if codebook == CB_MCG:
        return code_mcg(states)
    if codebook == CB_MUL1:
        return code_mul1(states)
    raise ValueError(f"unknown codebook {codebook}")


# ----------------------------------------------------------------------------
# Tile layout
# ----------------------------------------------------------------------------

def check_shape(m: int, n: int, K: int) -> None:
    if m % RHT_BLOCK or n % RHT_BLOCK or m <= 0 or n <= 0:
        raise ValueError("m and n must be positive multiples of 128")
    if not 1 <= K <= 8:
        raise ValueError("K must be in 1..8 ([TQ] Part eleven)")


def decode_tiles(codes: np.ndarray, K: int, codebook: int, m: int, n: int,
                 tile_rows: np.ndarray | None = None) -> np.ndarray:
    """Decode the packed codes of an m x n weight matrix into binary16 W-hat.

    Layout (readings): tiles are stored row-major over (I, J), tile (I, J)
    covering rows 16I..16I+15 and columns 16J..16J+15, each holding 8K uint32
    words ([TQ] Part eight: one 256-step sequence per 16x16 tile).  Step t of a
    tile maps to element (r, c) = (t // 16, t % 16) of that tile: the pages name
    a 16x16 "tile permutation" without giving it, and row-major is the plainest.

    ``tile_rows`` optionally restricts the decode to those tile-row indices I
    (for sampled checks of large layers); the result then has 16*len(tile_rows)
    rows, in the order given.
    """
    check_shape(m, n, K)
    nw = 8 * K
    grid = np.asarray(codes, dtype=np.uint32).reshape(m // TILE, n // TILE, nw)
    if tile_rows is not None:
        grid = grid[np.asarray(tile_rows)]
    rows = grid.shape[0]
    out = np.empty((rows, TILE, n // TILE, TILE), dtype=np.float16)
    chunk = max(1, 8192 // (n // TILE))  # tile-rows per pass, bounds memory only
    for r0 in range(0, rows, chunk):
        st = tile_states(grid[r0:r0 + chunk], K)             # [c, n/16, 256]
        w = decode_states(st, codebook)                       # [c, n/16, 256]
        w = w.reshape(w.shape[0], n // TILE, TILE, TILE)      # [c, J, r, col]
        out[r0:r0 + chunk] = w.transpose(0, 2, 1, 3)          # [c, r, J, col]
    return out.reshape(rows * TILE, n)


# ----------------------------------------------------------------------------
# Randomized Hadamard transform  ([DD] Section 2, [TQ] Parts six and eleven)
# ----------------------------------------------------------------------------

def hadamard(d: int = RHT_BLOCK) -> np.ndarray:
    """Unnormalized Sylvester-ordered Hadamard matrix, H[i, j] =
    (-1)**popcount(i & j) (entries only +-1, [TQ] Part six).  float64."""
    i = np.arange(d)
    parity = np.bitwise_count(i[:, None] & i[None, :]) & 1
    return np.where(parity == 1, -1.0, 1.0)


def rht(v: np.ndarray, signs: np.ndarray | None) -> np.ndarray:
    """Blockwise randomized Hadamard transform along the last axis, in float64:

        out = Hb (s (.) v),  Hb = blockdiag over 128-blocks of H_128 / sqrt(128).

    [DD] Section 2 runtime identity (rotation of x as H diag(s) x), with the
    normalized, orthogonal H of that section, applied per 128-block as EXL3 does
    ([TQ] Part eleven).  ``signs is None`` means no rotation on that side.
    """
    v = np.asarray(v, dtype=np.float64)
    if signs is None:
        return v.copy()
    d = v.shape[-1]
    assert d % RHT_BLOCK == 0
    s = np.asarray(signs, dtype=np.float64)
    blocks = (v * s).reshape(*v.shape[:-1], d // RHT_BLOCK, RHT_BLOCK)
    out = blocks @ hadamard(RHT_BLOCK).T / math.sqrt(RHT_BLOCK)
    return out.reshape(v.shape)


def rht_whole(v: np.ndarray, signs: np.ndarray | None) -> np.ndarray:
    """QTIP's rotation over the whole last axis, in float64:

        out = H_d (s (.) v) / sqrt(d),  H_d the Sylvester Hadamard matrix of the
        full (power-of-two) length d.

    [TQ] Part eleven: QTIP rotates whole rows and columns, where EXL3 rotates
    128-blocks; Part six: the transform is only plus and minus ones, applied as
    a fast Walsh-Hadamard transform.  The butterflies below are the textbook
    iterative transform in Sylvester order: at span h, every pair (i, i + h)
    with bit h of i clear becomes (a + b, a - b).  ``signs is None`` means no
    rotation on that side.
    """
    v = np.asarray(v, dtype=np.float64)
    if signs is None:
        return v.copy()
    d = v.shape[-1]
    assert d > 0 and d & (d - 1) == 0, "whole-vector rotation needs a power-of-two length"
    u = (v * np.asarray(signs, dtype=np.float64)).reshape(-1, d).copy()
    h = 1
    while h < d:
        u = u.reshape(-1, d // (2 * h), 2, h)
        a = u[:, :, 0, :].copy()
        b = u[:, :, 1, :].copy()
        u[:, :, 0, :] = a + b
        u[:, :, 1, :] = a - b
        u = u.reshape(-1, d)
        h *= 2
    return (u / math.sqrt(d)).reshape(v.shape)


# ----------------------------------------------------------------------------
# The layer  ([DD] Section 2, [FG] out_scales)
# ----------------------------------------------------------------------------

def layer_forward(codes, K, codebook, m, n, s_in, s_out, scales, x) -> np.ndarray:
    """y = Hb(s_out (.) (scale (.) (W-hat Hb(s_in (.) x)))) in float64.

    [DD] Section 2: x is rotated on the way in and the product rotated back on
    the way out.  Reading of the sign/Hadamard order: the runtime identity of
    that section is taken (sign first, then Hadamard, on each side); since H_128
    is symmetric the output side H^T diag(s) is the same blockwise transform
    applied after the signs.  Reading of the scale placement ([FG]: per-output-
    channel scales): z = scale (.) (W-hat x-tilde), applied in the rotated domain
    before the output transform.  ``s_in``/``s_out`` None = no rotation on that
    side.  x is float16 [M, n]; returns float64 [M, m].
    """
    x = np.atleast_2d(np.asarray(x))
    W = decode_tiles(codes, K, codebook, m, n).astype(np.float64)
    xt = rht(x.astype(np.float64), s_in)
    z = (xt @ W.T) * np.asarray(scales, dtype=np.float64)
    return rht(z, s_out)


def layer_forward_rowblocks(codes, K, codebook, m, n, s_in, s_out, scales, x,
                            row_blocks) -> np.ndarray:
    """Rows of ``layer_forward`` for the listed 128-row output blocks only.

    The output transform mixes rows only within a 128-block, so each block of y
    depends on that block's 8 tile-rows alone.  Returns float64
    [M, 128*len(row_blocks)] in the order given.
    """
    x = np.atleast_2d(np.asarray(x))
    xt = rht(x.astype(np.float64), s_in)
    scales = np.asarray(scales, dtype=np.float64)
    s_out = None if s_out is None else np.asarray(s_out)
    outs = []
    for b in row_blocks:
        trows = np.arange(b * 8, b * 8 + 8)
        W = decode_tiles(codes, K, codebook, m, n, tile_rows=trows).astype(np.float64)
        z = (xt @ W.T) * scales[b * 128:(b + 1) * 128]
        sb = None if s_out is None else s_out[b * 128:(b + 1) * 128]
        outs.append(rht(z, sb))
    return np.concatenate(outs, axis=-1)


def layer_forward_whole(codes, K, codebook, m, n, s_in, s_out, scales, x) -> np.ndarray:
    """The layer with QTIP's whole-vector rotations instead of EXL3's 128-blocks
    ([TQ] Part eleven): y = H_m (s_out (.) (scale (.) (W-hat H_n (s_in (.) x))))
    with H_d / sqrt(d) over the full (power-of-two) n and m, in float64.  The
    same readings as ``layer_forward`` otherwise."""
    x = np.atleast_2d(np.asarray(x))
    W = decode_tiles(codes, K, codebook, m, n).astype(np.float64)
    xt = rht_whole(x.astype(np.float64), s_in)
    z = (xt @ W.T) * np.asarray(scales, dtype=np.float64)
    return rht_whole(z, s_out)


# ----------------------------------------------------------------------------
# The int8-activation path ([TQ] Part eleven)
# ----------------------------------------------------------------------------

#: int8 activations are quantized per 128-column block of each row.
INT8_BLOCK = 128
INT8_MAX = 127


def quantize_act(xt: np.ndarray):
    """Activations to int8 for the dp4a path.

    [TQ] Part eleven: with the weight an affine function of a byte sum (mul1)
    and the activations quantized to eight-bit integers, one dp4a computes
    code value times activation for four bytes at once.  The pages do not say
    how the activations are quantized.  Reading: symmetric, per 128-column
    block of each row of the rotated activations x-tilde (binary16), in
    binary32: scale = max|x| / 127 (one binary32 division), q = the nearest
    integer to x / scale (one binary32 division, ties to even); a block of
    zeros has scale 0 and q 0.  Returns (q int8 [M, n], scale float32
    [M, n/128]).
    """
    xt = np.atleast_2d(np.asarray(xt, dtype=np.float16)).astype(np.float32)
    M, n = xt.shape
    assert n % INT8_BLOCK == 0
    blocks = xt.reshape(M, n // INT8_BLOCK, INT8_BLOCK)
    amax = np.abs(blocks).max(axis=2)
    scale = (amax / np.float32(INT8_MAX)).astype(np.float32)
    safe = np.where(scale > 0, scale, np.float32(1))
    q = np.rint(blocks / safe[:, :, None]).astype(np.float32)
    q = np.where(scale[:, :, None] > 0, q, 0)
    return q.reshape(M, n).astype(np.int8), scale


def layer_forward_int8(codes, K, codebook, m, n, s_out, scales, q, qscale) -> np.ndarray:
    """The layer on int8 activations: y = Hb(s_out (.) (scale (.) (W-hat x-hat)))
    with x-hat = q * qscale per 128-column block (already rotated), in float64.
    Only the byte-sum codes (1MAD, mul1) have the affine form the dp4a path
    uses ([TQ] Part eleven)."""
    if codebook not in (CB_1MAD, CB_MUL1):
        raise ValueError("the int8-activation path needs a byte-sum code (1MAD or mul1)")
    q = np.atleast_2d(np.asarray(q, dtype=np.float64))
    M = q.shape[0]
    xhat = (q.reshape(M, n // INT8_BLOCK, INT8_BLOCK)
            * np.asarray(qscale, dtype=np.float64).reshape(M, n // INT8_BLOCK, 1)).reshape(M, n)
    W = decode_tiles(codes, K, codebook, m, n).astype(np.float64)
    z = (xhat @ W.T) * np.asarray(scales, dtype=np.float64)
    return rht(z, s_out)
