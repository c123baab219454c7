"""Seeded synthetic inputs and the workload shapes.

This module holds no decode, transform or product arithmetic: it only draws
random numbers and lists shapes, so both the CUDA path and the CPU oracle can be
fed the same inputs.  All arrays are numpy, on the host.

Recipe (the pages measure on real Llama checkpoints, which are not available;
these synthetic tensors of the same shapes stand in for them):

* packed codes: i.i.d. uniform uint32 words.  Every bit pattern is a valid
  tail-biting trellis codeword, so a uniform bitstream is a legal stream.
* per-output-channel scales: fp16(0.02 * N(1, 0.1)).
* sign vectors: Rademacher +-1 as fp16.
* activations x: fp16(N(0, 1)), one row per batch element.

Seeds: ``seed_for(config, tensor)`` = splitmix64(0xE3E30000 + 1000*config +
tensor), fed to numpy's PCG64.
"""
from __future__ import annotations

import numpy as np

_MASK64 = (1 << 64) - 1


def splitmix64(x: int) -> int:
    """The splitmix64 output function (Steele, Lea, Flood 2014), used to spread
    small integer seeds over 64 bits."""
    x = (x + 0x9E3779B97F4A7C15) & _MASK64
    z = x
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def seed_for(config: int, tensor: int) -> int:
    return splitmix64(0xE3E30000 + 1000 * config + tensor)


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def packed_codes(m: int, n: int, K: int, seed: int) -> np.ndarray:
    """Uniform random packed stream for an m x n layer: (m/16)*(n/16)*8K uint32."""
    count = (m // 16) * (n // 16) * 8 * K
    return _rng(seed).integers(0, 1 << 32, size=count, dtype=np.uint64).astype(np.uint32)


def sign_vector(d: int, seed: int) -> np.ndarray:
    """Rademacher +-1 vector of length d as float16."""
    bits = _rng(seed).integers(0, 2, size=d)
    return np.where(bits == 1, 1.0, -1.0).astype(np.float16)


def channel_scales(m: int, seed: int) -> np.ndarray:
    """Per-output-channel scales fp16(0.02 * N(1, 0.1))."""
    return (0.02 * _rng(seed).normal(1.0, 0.1, size=m)).astype(np.float16)


def activations(M: int, n: int, seed: int) -> np.ndarray:
    """x ~ fp16(N(0, 1)), shape [M, n]."""
    return _rng(seed).standard_normal(size=(M, n)).astype(np.float16)


def outlier_activations(M: int, n: int, seed: int, channels: int = 4, magnitude: float = 1000.0) -> np.ndarray:
    """Heavy-tailed activations: fp16(N(0, 1)) with `channels` channels (the
    same columns in every row) set to +-magnitude with random signs -- the
    outlier features that the input rotation exists to spread out."""
    rng = _rng(seed)
    x = rng.standard_normal(size=(M, n))
    cols = rng.choice(n, size=channels, replace=False)
    signs = np.where(rng.integers(0, 2, size=(M, channels)) == 1, 1.0, -1.0)
    x[:, cols] = magnitude * signs
    return x.astype(np.float16)


def layer_inputs(m: int, n: int, K: int, M: int, config: int, index: int) -> dict:
    """All inputs of one layer with the standard seeds (tensor ids 10*index+0..4)."""
    b = 10 * index
    return dict(
        codes=packed_codes(m, n, K, seed_for(config, b + 0)),
        s_in=sign_vector(n, seed_for(config, b + 1)),
        s_out=sign_vector(m, seed_for(config, b + 2)),
        scales=channel_scales(m, seed_for(config, b + 3)),
        x=activations(M, n, seed_for(config, b + 4)),
    )


# ----------------------------------------------------------------------------
# Workloads (shapes are (out m, in n))
# ----------------------------------------------------------------------------

CB_3INST, CB_1MAD = 0, 1

#: Single 4096x4096 layer, K=2, 1MAD, batch 1.
SINGLE_4096 = [("w", 4096, 4096, 2, CB_1MAD)]

LLAMA8B_SHAPES = [("q", 4096, 4096), ("k", 1024, 4096), ("v", 1024, 4096),
                  ("o", 4096, 4096), ("gate", 14336, 4096), ("up", 14336, 4096),
                  ("down", 4096, 14336)]

LLAMA70B_SHAPES = [("q", 8192, 8192), ("k", 1024, 8192), ("v", 1024, 8192),
                   ("o", 8192, 8192), ("gate", 28672, 8192), ("up", 28672, 8192),
                   ("down", 8192, 28672)]


CB_MCG = 2
CB_MUL1 = 3
CODE_NAMES = {CB_3INST: "3inst", CB_1MAD: "1mad", CB_MCG: "mcg", CB_MUL1: "mul1"}


def llama8b_layer_set(codes=(CB_1MAD, CB_3INST)):
    """Llama-3-8B-shaped decoder layer set: every projection at K = 2, 3, 4 with
    each code (42 GEMVs, 1.309 G weights for two codes)."""
    out = []
    for cb in codes:
        for K in (2, 3, 4):
            for name, m, n in LLAMA8B_SHAPES:
                out.append((f"{name}.K{K}.{CODE_NAMES[cb]}", m, n, K, cb))
    return out


def llama70b_stack(layers: int = 32):
    """Llama-3-70B-shaped layers, K = 2, 3INST, all resident."""
    return [(f"L{l}.{name}", m, n, 2, CB_3INST)
            for l in range(layers) for name, m, n in LLAMA70B_SHAPES]


def whole_attention_stack(layers: int = 8):
    """Llama-3-70B attention projections (power-of-two shapes, as QTIP's
    whole-vector rotations need), K = 2, 3INST, all resident."""
    return [(f"L{l}.{name}", m, n, 2, CB_3INST)
            for l in range(layers) for name, m, n in LLAMA70B_SHAPES if name in ("q", "k", "v", "o")]


BATCH_SWEEP = [1, 2, 4, 8, 16, 32]
BATCH_SWEEP_SHAPES = [("gate", 14336, 4096, 3, CB_1MAD), ("down", 4096, 14336, 3, CB_1MAD)]


def mixed_stack_widths(seed: int = seed_for(4, 999)) -> np.ndarray:
    """Per-tensor K of the 240 MLP tensors of the 80-layer mixed stack: a seeded
    shuffle of 84 x K2 + 146 x K3 + 10 x K4, which with the attention tensors at
    K4 gives a decoder-body average of 2.9010 bits per weight."""
    ks = np.array([2] * 84 + [3] * 146 + [4] * 10)
    _rng(seed).shuffle(ks)
    return ks


def mixed_stack(layers: int = 80, codebook: int = CB_3INST):
    """80 layers of {q, o 8192x8192 at K4; gate, up 28672x8192; down 8192x28672
    at the shuffled widths} plus the 128256x8192 lm_head at K6."""
    ks = mixed_stack_widths()
    out, i = [], 0
    for l in range(layers):
        out.append((f"L{l}.q", 8192, 8192, 4, codebook))
        out.append((f"L{l}.o", 8192, 8192, 4, codebook))
        for name, m, n in (("gate", 28672, 8192), ("up", 28672, 8192), ("down", 8192, 28672)):
            out.append((f"L{l}.{name}", m, n, int(ks[i]), codebook))
            i += 1
    out.append(("lm_head", 128256, 8192, 6, codebook))
    return out
