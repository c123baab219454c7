"""Parity with heavy-tailed activations and large channel scales.

Outlier features are the reason the input rotation exists ("ExLlamaV3 & EXL3
Deep Dive" Section 2), and 16-bit arithmetic is where they hurt ("Trellis
Quantization" Part eleven reports overflow in half-precision decoding on some
models).  These tests feed x with four channels at +-1000 (before the input
RHT; everything else N(0, 1)) and scales 50x the standard 0.02 scale, on the
Llama-3-70B and mixed-stack layer shapes at full size, through every kernel
family: the decode-MMA kernel (default, batch 1 and 16), the warp-shuffle
kernel (binary16 products, 16-column binary16 partial sums), and both prefill
strategies.  Checked on sampled 128-row output blocks against the oracle's
float64 layer, at the same tolerance as every layer test.
"""
import numpy as np
import pytest
import torch

from oracle import exl3_oracle as O
from trellis_decode_gemv_gb300 import binding as B
from trellis_decode_gemv_gb300 import synth
from tests.gpu_helpers import assert_layer_close, upload

pytestmark = pytest.mark.gpu

SHAPES = [
    (8192, 8192, 2, 0),      # Llama-3-70B q/o, K2 3INST
    (28672, 8192, 2, 0),     # gate/up
    (8192, 28672, 2, 0),     # down
    (8192, 8192, 4, 0),      # mixed stack attention, K4
    (28672, 8192, 3, 1),     # mixed stack MLP width, 1MAD
    (128256, 8192, 6, 0),    # mixed stack lm_head, K6
]


def _inputs(m, n, K, M, index):
    inp = synth.layer_inputs(m, n, K, M, config=95, index=index)
    inp["x"] = synth.outlier_activations(M, n, synth.seed_for(95, 10 * index + 5))
    inp["scales"] = (inp["scales"].astype(np.float32) * 50.0).astype(np.float16)
    return inp


def _check(inp, K, cb, m, n, M, path=None, prefill=None, what=""):
    d = upload(inp)
    ws = torch.zeros(B.exl3_gemm_workspace_bytes(m, n, M), dtype=torch.uint8, device="cuda")
    y = torch.full((M, m), float("nan"), dtype=torch.float16, device="cuda")
    if path is not None:
        B.exl3_set_path(path)
    if prefill is not None:
        B.exl3_set_prefill(prefill)
    try:
        B.exl3_gemm(d["codes"], K, cb, m, n, d["s_in"], d["s_out"], d["scales"], d["x"], y=y, workspace=ws)
        torch.cuda.synchronize()
    finally:
        B.exl3_set_path(B.PATH_AUTO)
        B.exl3_set_prefill(B.PREFILL_AUTO)
    nb = m // 128
    rbs = sorted({0, nb // 2, nb - 1})
    ref = O.layer_forward_rowblocks(inp["codes"], K, cb, m, n, inp["s_in"], inp["s_out"], inp["scales"],
                                    inp["x"], rbs)
    cols = torch.cat([torch.arange(b * 128, b * 128 + 128) for b in rbs]).cuda()
    assert np.abs(ref).max() > 10.0  # the outliers reach the output
    assert_layer_close(y[:, cols], ref, what)


@pytest.mark.parametrize("m,n,K,cb", SHAPES)
@pytest.mark.parametrize("M", [1, 16])
def test_outliers_decode_mma(m, n, K, cb, M):
    _check(_inputs(m, n, K, M, index=m // 128 + n // 128 + K + M), K, cb, m, n, M, what=f"{m}x{n} M={M}")


@pytest.mark.parametrize("m,n,K,cb", SHAPES)
def test_outliers_warp_shuffle(m, n, K, cb):
    M = 1
    _check(_inputs(m, n, K, M, index=m // 128 + n // 128 + K), K, cb, m, n, M, path=B.PATH_SHUFFLE,
           what=f"shuffle {m}x{n}")


@pytest.mark.parametrize("m,n,K,cb", [SHAPES[0], SHAPES[2], SHAPES[4]])
@pytest.mark.parametrize("M,prefill", [(48, "fused"), (300, "decode_once")])
def test_outliers_prefill(m, n, K, cb, M, prefill):
    pf = B.PREFILL_FUSED if prefill == "fused" else B.PREFILL_DECODE_ONCE
    _check(_inputs(m, n, K, M, index=m // 128 + n // 128 + K + M), K, cb, m, n, M, prefill=pf,
           what=f"{prefill} {m}x{n} M={M}")
