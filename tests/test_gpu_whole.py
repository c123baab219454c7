"""GPU parity of QTIP's whole-vector rotation ("Trellis Quantization" Part
eleven: QTIP rotates whole rows and columns): the standalone transform
exl3_rht_whole against the oracle's float64 rht_whole (one binary16 rounding
of an fp32 computation), and the layer exl3_gemm_whole against the oracle's
layer_forward_whole (relative L2 <= 5e-3, |err| <= 1e-2 * max|y_ref|) on every
kernel family: warp-shuffle (M <= 2), tensor-core (3..32) and dense prefill
(M > 32)."""
import numpy as np
import pytest
import torch

from oracle import exl3_oracle as O
from trellis_decode_gemv_gb300 import binding as B
from trellis_decode_gemv_gb300 import synth
from tests.gpu_helpers import assert_layer_close, to_dev, upload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows,d", [(1, 128), (3, 1024), (2, 4096), (5, 16384), (1, 32768)])
def test_rht_whole_matches_oracle(rows, d):
    x = synth.activations(rows, d, synth.seed_for(60, d))
    s = synth.sign_vector(d, synth.seed_for(60, d + 1))
    ref = O.rht_whole(x.astype(np.float64), s)
    got = B.exl3_rht_whole(to_dev(x), to_dev(s))
    torch.cuda.synchronize()
    g = got.float().cpu().numpy().astype(np.float64)
    # one rounding to binary16 of an fp32 evaluation
    assert np.all(np.abs(g - ref) <= np.abs(ref) * 2.0 ** -11 * 1.001 + 1e-5), np.max(np.abs(g - ref))


def test_rht_whole_round_trip():
    """H_d / sqrt(d) is an orthogonal involution: s (.) H(H(s (.) x)) = x up to
    two binary16 roundings."""
    d = 8192
    x = synth.activations(2, d, synth.seed_for(61, 0))
    s = synth.sign_vector(d, synth.seed_for(61, 1))
    ones = torch.ones(d, dtype=torch.float16, device="cuda")
    back = B.exl3_rht_whole(B.exl3_rht_whole(to_dev(x), to_dev(s)), ones) * to_dev(s)
    torch.cuda.synchronize()
    err = back.float().cpu().numpy() - x.astype(np.float32)
    assert np.abs(err).max() < 4 * 2.0 ** -10 * np.abs(x).max()


def _layer(inp, K, cb, m, n, s_in=True, s_out=True):
    d = upload(inp)
    M = inp["x"].shape[0]
    y = torch.full((M, m), float("nan"), dtype=torch.float16, device="cuda")
    ws = torch.zeros(B.exl3_gemm_whole_workspace_bytes(m, n, M), dtype=torch.uint8, device="cuda")
    B.exl3_gemm_whole(d["codes"], K, cb, m, n, d["s_in"] if s_in else None, d["s_out"] if s_out else None,
                      d["scales"], d["x"], y=y, workspace=ws)
    torch.cuda.synchronize()
    assert B.workspace_status(ws, m) == 0
    ref = O.layer_forward_whole(inp["codes"], K, cb, m, n, inp["s_in"] if s_in else None,
                                inp["s_out"] if s_out else None, inp["scales"], inp["x"])
    return y, ref


@pytest.mark.parametrize("m,n,M,K,cb", [
    (128, 128, 1, 2, 0), (256, 512, 1, 3, 1), (1024, 4096, 1, 2, 1), (4096, 1024, 2, 4, 0),
    (512, 256, 8, 2, 2), (1024, 1024, 17, 3, 3), (256, 1024, 40, 2, 1), (2048, 512, 300, 3, 0),
])
def test_gemm_whole_matches_oracle(m, n, M, K, cb):
    inp = synth.layer_inputs(m, n, K, M, config=62, index=m + n + M)
    y, ref = _layer(inp, K, cb, m, n)
    assert_layer_close(y, ref, f"{m}x{n} M={M}")


@pytest.mark.parametrize("s_in,s_out", [(False, True), (True, False), (False, False)])
def test_gemm_whole_one_side(s_in, s_out):
    m, n, K, cb, M = 512, 2048, 2, 1, 3
    inp = synth.layer_inputs(m, n, K, M, config=63, index=int(s_in) + 2 * int(s_out))
    y, ref = _layer(inp, K, cb, m, n, s_in, s_out)
    assert_layer_close(y, ref, f"s_in={s_in} s_out={s_out}")


def test_gemm_whole_4096_square_batch1():
    """A Llama attention projection shape, every output checked."""
    m = n = 4096
    K, cb, M = 2, 1, 1
    inp = synth.layer_inputs(m, n, K, M, config=64, index=0)
    y, ref = _layer(inp, K, cb, m, n)
    assert_layer_close(y, ref, "4096x4096 whole")


def test_gemm_whole_extreme_lengths():
    """The longest input (32768: 256 blocks across) into the shortest output
    (128: nothing across), every output checked."""
    m, n, K, cb, M = 128, 32768, 2, 0, 2
    inp = synth.layer_inputs(m, n, K, M, config=65, index=0)
    y, ref = _layer(inp, K, cb, m, n)
    assert_layer_close(y, ref, "128 x 32768")


def _whole_group(shapes, K, M, config, rot=None):
    out = []
    for i, (m, n) in enumerate(shapes):
        inp = synth.layer_inputs(m, n, K, M, config=config, index=i)
        use_in, use_out = rot[i] if rot else (True, True)
        if not use_in:
            inp["s_in"] = None
        if not use_out:
            inp["s_out"] = None
        d = upload({k: v for k, v in inp.items() if v is not None})
        d.setdefault("s_in", None)
        d.setdefault("s_out", None)
        d.update(m=m, n=n, y=torch.full((M, m), float("nan"), dtype=torch.float16, device="cuda"))
        out.append((inp, d))
    return out


@pytest.mark.parametrize("M", [1, 2, 5, 32])
@pytest.mark.parametrize("K,cb", [(2, 0), (3, 1)])
def test_gemm_whole_grouped_matches_oracle(M, K, cb):
    """q/k/v-like group (one wide, two narrow outputs) and lengths that differ
    per layer: one chain of launches, every layer against the oracle's
    whole-vector layer, the status word (byte 0) left at zero."""
    shapes = [(1024, 1024), (256, 1024), (256, 1024)] if M != 5 else [(512, 2048), (2048, 512), (128, 128)]
    layers = _whole_group(shapes, K, M, config=66 + M)
    ws = torch.zeros(B.exl3_gemm_whole_grouped_workspace_bytes(shapes, M), dtype=torch.uint8, device="cuda")
    B.exl3_gemm_whole_grouped([d for _, d in layers], K, cb, workspace=ws)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32)[0]) == 0
    for inp, d in layers:
        ref = O.layer_forward_whole(inp["codes"], K, cb, d["m"], d["n"], inp["s_in"], inp["s_out"], inp["scales"],
                                    inp["x"])
        assert_layer_close(d["y"], ref, f"grouped {d['m']}x{d['n']} M={M}")


def test_gemm_whole_grouped_one_sided_and_reuse():
    """Layers without an input or an output rotation in the same group, and
    a second call on the same workspace."""
    shapes = [(512, 1024), (1024, 512), (256, 256), (128, 2048)]
    rot = [(False, True), (True, False), (False, False), (True, True)]
    K, cb, M = 2, 1, 3
    layers = _whole_group(shapes, K, M, config=69, rot=rot)
    ws = torch.zeros(B.exl3_gemm_whole_grouped_workspace_bytes(shapes, M), dtype=torch.uint8, device="cuda")
    for _ in range(2):
        for _, d in layers:
            d["y"].fill_(float("nan"))
        B.exl3_gemm_whole_grouped([d for _, d in layers], K, cb, workspace=ws)
        torch.cuda.synchronize()
        for inp, d in layers:
            ref = O.layer_forward_whole(inp["codes"], K, cb, d["m"], d["n"], inp["s_in"], inp["s_out"],
                                        inp["scales"], inp["x"])
            assert_layer_close(d["y"], ref, f"one-sided {d['m']}x{d['n']}")
