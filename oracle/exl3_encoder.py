"""Viterbi encoder for the bitshift trellis, used to pin the quality of the
computed codes.

TEST INFRASTRUCTURE ONLY, like ``exl3_oracle``: the product path never imports,
calls or links it, and it shares nothing with the CUDA side.  It exists so that
the codebook readings of the oracle (LCG constants, 3INST mask and magic, 1MAD
centring) can be checked against the one number the pages print for them: the
mean-squared error of the trellis with the three-instruction code on a
synthetic Gaussian source at two bits per weight, about 0.069 ("Trellis
Quantization: Trading Memory for Cheap Compute", Part nine), between the
rate-distortion bound 1/16 and the E8 lattice's 0.089.

What it follows:

* Part seven of the same lecture: the Viterbi algorithm walks the sequence one
  step at a time, keeps for every state the cheapest path that ends in it, and
  reads the best path back at the end.
* Part eight: the bitshift trellis (an L-bit window that moves K bits per step,
  so the successors of state s are ((s << K) | b) mod 2**L), and the
  tail-biting approximation: rotate the sequence by half its length, run
  Viterbi, read off the state in the middle, then run Viterbi again on the
  original sequence constrained to start with that state and to wrap around
  onto it.

Everything is numpy and literal; the cost of a path is the sum of squared
differences between the decoded values and the target sequence.  The path
costs run in float64 by default; a float32 mode takes every argmin decision on
binary32 costs evaluated in a stated order (``viterbi``), so that another
binary32 implementation of the same search can be compared with it bit for
bit (its chosen words and its final cost).
"""
from __future__ import annotations

import numpy as np

from . import exl3_oracle as O


def viterbi(values: np.ndarray, target: np.ndarray, K: int, L: int, start: int | None = None,
            forced: dict | None = None, dtype=np.float64):
    """Cheapest state path of the L-bit, K-bit-shift trellis for `target`.

    values  [2**L]: the decoded value of every state;
    target  [T]: the sequence to quantize;
    start   None (any first state) or the required first state;
    forced  {t: (mask, bits)}: at step t >= 1 the K appended bits b must
            satisfy b & mask == bits;
    dtype   the arithmetic of the path costs: float64, or float32, where every
            difference, square and sum is one binary32 rounding, in this
            order: cost_t(s) = best_{t-1}(s >> K) + (v(s) - x_t)^2.  Ties go to
            the smallest predecessor index h and, at the end, the smallest
            state.
    Returns (states int64 [T], cost).
    """
    values = np.asarray(values, dtype=dtype)
    target = np.asarray(target, dtype=dtype)
    T = len(target)
    nst = 1 << L
    nb = 1 << K
    low = nst >> K
    inf = dtype(np.inf)
    cost = (values - target[0]) ** 2
    if start is not None:
        keep = np.zeros(nst, dtype=bool)
        keep[start] = True
        cost = np.where(keep, cost, inf)
    back = np.empty((T, low), dtype=np.uint8)
    bvals = np.arange(nst) & (nb - 1)
    for t in range(1, T):
        # predecessors of s' = ((s << K) | b) mod 2**L are s = (s' >> K) | (h << (L - K))
        grouped = cost.reshape(nb, low)  # [h, s' >> K]
        h = np.argmin(grouped, axis=0)
        best = grouped[h, np.arange(low)]
        back[t] = h
        cost = np.repeat(best, nb) + (values - target[t]) ** 2
        if forced is not None and t in forced:
            mask, bits = forced[t]
            cost = np.where((bvals & mask) == bits, cost, inf)
    states = np.empty(T, dtype=np.int64)
    s = int(np.argmin(cost))
    total = float(cost[s])
    for t in range(T - 1, -1, -1):
        states[t] = s
        if t > 0:
            s = (s >> K) | (int(back[t][s >> K]) << (L - K))
    return states, total


def _stream_bit_of_start(start: int, j: int, L: int) -> int:
    """Bit j (j < L) of a stream whose first window is `start` (MSB first)."""
    return (start >> (L - 1 - j)) & 1


def encode_tile(target: np.ndarray, values: np.ndarray, K: int, L: int = O.L, dtype=np.float64):
    """Tail-biting encoding of one 256-step sequence (one 16x16 tile), by the
    two-pass approximation of Part eight, with path costs in `dtype` (see
    ``viterbi``).  Returns (words uint32 [8K], states int64 [256], mse)."""
    T = len(target)
    nbits = T * K
    # Pass 1: the sequence rotated by half its length, free start and end; the
    # state in the middle of that path is the window at the start (and, by
    # wrapping, at the end) of the original sequence.
    half = T // 2
    rotated = np.roll(target, -half)
    states1, _ = viterbi(values, rotated, K, L, dtype=dtype)
    s_star = int(states1[half])
    # Pass 2: the original sequence, starting with s_star; the bits appended at
    # steps whose new bits lie past the end of the circular stream must repeat
    # the stream's first bits, i.e. those of s_star.
    forced = {}
    for t in range(1, T):
        first = K * (t - 1) + L  # stream index of the first appended bit
        mask = bits = 0
        for i in range(K):
            j = first + i
            if j >= nbits:
                shift = K - 1 - i
                mask |= 1 << shift
                bits |= _stream_bit_of_start(s_star, j - nbits, L) << shift
        if mask:
            forced[t] = (mask, bits)
    states, cost = viterbi(values, target, K, L, start=s_star, forced=forced, dtype=dtype)
    # The stream: the first window, then the K bits appended at each step.
    stream = np.zeros(nbits, dtype=np.uint8)
    for j in range(min(L, nbits)):
        stream[j] = _stream_bit_of_start(s_star, j, L)
    for t in range(1, T):
        b = int(states[t]) & ((1 << K) - 1)
        for i in range(K):
            j = K * (t - 1) + L + i
            if j < nbits:
                stream[j] = (b >> (K - 1 - i)) & 1
    words = np.packbits(stream.reshape(-1, 32), axis=1, bitorder="big").view(">u4").astype(np.uint32).ravel()
    return words, states, cost / T


def codebook_values(codebook: int, unit_variance: bool = True) -> np.ndarray:
    """The decoded value of every 16-bit state, in float64; with unit_variance,
    divided by the codebook's standard deviation over all states (a Gaussian
    source of variance 1 is quantized; in a layer the per-channel scale plays
    this part)."""
    v = O.decode_states(np.arange(1 << O.L, dtype=np.uint32), codebook).astype(np.float64)
    if unit_variance:
        v = v / np.sqrt(np.mean(v * v))
    return v


def trellis_mse(values: np.ndarray, samples: np.ndarray, K: int) -> float:
    """Mean-squared error of the tail-biting trellis code with state values
    `values` on `samples` (a multiple of 256 long), tile by tile."""
    tiles = samples.reshape(-1, O.STEPS)
    return float(np.mean([encode_tile(t, values, K)[2] for t in tiles]))


def lloyd_max(samples: np.ndarray, levels: int, iters: int = 200) -> tuple[np.ndarray, float]:
    """Lloyd-Max scalar quantizer fitted to `samples` (the classical
    alternating nearest-level / centroid iteration).  Returns (levels, mse)."""
    q = np.quantile(samples, (np.arange(levels) + 0.5) / levels)
    for _ in range(iters):
        edges = (q[1:] + q[:-1]) / 2
        idx = np.searchsorted(edges, samples)
        q = np.array([samples[idx == k].mean() for k in range(levels)])
    edges = (q[1:] + q[:-1]) / 2
    idx = np.searchsorted(edges, samples)
    return q, float(np.mean((samples - q[idx]) ** 2))
