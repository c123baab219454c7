"""GPU parity of the int8-activation path ("Trellis Quantization" Part eleven:
eight-bit activations, byte-sum codes, one dp4a per four products):

* the quantizer, bit-exact against the oracle's binary32 quantizer on seeded
  binary16 activations (q and the block scales);
* exl3_gemm_i8 on given int8 activations against the oracle's float64 layer on
  the same dequantized activations (relative L2 <= 5e-3, |err| <= 1e-2 *
  max|y_ref|), for 1MAD and mul1, K = 1..8, batch chunks of 1, 2, 4, 8;
* exl3_gemm_int8act from binary16 activations against the oracle's
  quantize-then-layer, and its distance from the unquantized layer;
* the grouped calls (one K and code; and layers of their own K and code in one
  chain) against the same per layer."""
import numpy as np
import pytest
import torch

from oracle import exl3_oracle as O
from trellis_decode_gemv_gb300 import binding as B
from trellis_decode_gemv_gb300 import synth
from tests.gpu_helpers import assert_layer_close, layer_error, to_dev, upload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,n", [(1, 128), (3, 4096), (8, 14336)])
def test_quantizer_bit_exact(M, n):
    x = synth.activations(M, n, synth.seed_for(82, n))
    x[0, :128] = 0  # a zero block
    q, qs = B.exl3_quantize_act(to_dev(x))
    torch.cuda.synchronize()
    q_ref, qs_ref = O.quantize_act(x)
    np.testing.assert_array_equal(q.cpu().numpy(), q_ref)
    np.testing.assert_array_equal(qs.cpu().numpy().view(np.uint32), qs_ref.view(np.uint32))


def _int8_inputs(m, n, K, M, cfg, idx):
    inp = synth.layer_inputs(m, n, K, M, config=cfg, index=idx)
    xt = O.rht(inp["x"].astype(np.float64), inp["s_in"]).astype(np.float16)  # a rotated activation
    q, qs = O.quantize_act(xt)
    return inp, q, qs


@pytest.mark.parametrize("cb", [1, 3])
@pytest.mark.parametrize("K", [1, 2, 3, 4, 5, 6, 7, 8])
def test_gemm_i8_codes_and_widths(K, cb):
    m, n, M = 256, 512, 1
    inp, q, qs = _int8_inputs(m, n, K, M, 83, 10 * K + cb)
    d = upload(inp)
    y = B.exl3_gemm_i8(d["codes"], K, cb, m, n, d["s_out"], d["scales"], to_dev(q), to_dev(qs))
    torch.cuda.synchronize()
    ref = O.layer_forward_int8(inp["codes"], K, cb, m, n, inp["s_out"], inp["scales"], q, qs)
    assert_layer_close(y, ref, f"K={K} cb={cb}")


@pytest.mark.parametrize("M", [1, 2, 3, 5, 8, 15, 32])
def test_gemm_i8_batches(M):
    m, n, K, cb = 1024, 1024, 3, 3
    inp, q, qs = _int8_inputs(m, n, K, M, 84, M)
    d = upload(inp)
    ws = torch.zeros(B.exl3_gemm_i8_workspace_bytes(m, n, M), dtype=torch.uint8, device="cuda")
    y = B.exl3_gemm_i8(d["codes"], K, cb, m, n, d["s_out"], d["scales"], to_dev(q), to_dev(qs), workspace=ws)
    torch.cuda.synchronize()
    assert B.workspace_status(ws, m) == 0
    assert float(ws[256:256 + 4 * M * m].view(torch.float32).abs().sum()) == 0.0  # row sums left at zero
    ref = O.layer_forward_int8(inp["codes"], K, cb, m, n, inp["s_out"], inp["scales"], q, qs)
    assert_layer_close(y, ref, f"M={M}")


@pytest.mark.parametrize("m,n,K,cb", [(14336, 4096, 2, 1), (4096, 14336, 4, 3)])
def test_gemm_int8act_llama_shapes(m, n, K, cb):
    """From binary16 activations: against the oracle's quantize-then-layer on
    sampled row blocks, and about 1% from the unquantized layer."""
    M = 1
    inp = synth.layer_inputs(m, n, K, M, config=85, index=K)
    d = upload(inp)
    y = B.exl3_gemm_int8act(d["codes"], K, cb, m, n, d["s_in"], d["s_out"], d["scales"], d["x"])
    torch.cuda.synchronize()
    rbs = [0, 13, m // 128 - 1]
    xt = O.rht(inp["x"].astype(np.float64), inp["s_in"]).astype(np.float16)
    q, qs = O.quantize_act(xt)
    xhat = (q.astype(np.float64).reshape(M, n // 128, 128) * qs.astype(np.float64)[:, :, None]).reshape(M, n)
    ref8 = O.layer_forward_rowblocks(inp["codes"], K, cb, m, n, None, inp["s_out"], inp["scales"], xhat, rbs)
    cols = torch.cat([torch.arange(b * 128, b * 128 + 128) for b in rbs]).cuda()
    got = y.view(M, m)[:, cols]
    assert_layer_close(got, ref8, "int8act vs quantized oracle")
    reff = O.layer_forward_rowblocks(inp["codes"], K, cb, m, n, inp["s_in"], inp["s_out"], inp["scales"],
                                     inp["x"], rbs)
    rel, _ = layer_error(got, reff)
    assert 1e-3 < rel < 2.5e-2, rel


@pytest.mark.parametrize("M", [1, 3])
def test_int8act_grouped_matches_the_oracle_per_layer(M):
    """q/k/v-like layers with different shapes and their own x in one grouped
    call: each layer within tolerance of the oracle's quantize-then-layer."""
    K, cb = 2, 3
    shapes = [(512, 1024), (256, 1024), (256, 1024), (128, 2048)]
    layers, refs = [], []
    for i, (m, n) in enumerate(shapes):
        inp = synth.layer_inputs(m, n, K, M, config=86, index=10 * M + i)
        d = upload(inp)
        layers.append(dict(codes=d["codes"], m=m, n=n, s_in=d["s_in"], s_out=d["s_out"], scales=d["scales"],
                           x=d["x"], y=torch.full((M, m), float("nan"), dtype=torch.float16, device="cuda")))
        xt = O.rht(inp["x"].astype(np.float64), inp["s_in"]).astype(np.float16)
        q, qs = O.quantize_act(xt)
        refs.append(O.layer_forward_int8(inp["codes"], K, cb, m, n, inp["s_out"], inp["scales"], q, qs))
    ws = torch.zeros(B.exl3_group_i8_workspace_bytes(shapes, M), dtype=torch.uint8, device="cuda")
    B.exl3_gemm_int8act_grouped(layers, K, cb, workspace=ws)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0
    for L, ref in zip(layers, refs):
        assert_layer_close(L["y"], ref, f"grouped {L['m']}x{L['n']} M={M}")
    # the same layers one call at a time agree within one binary16 rounding
    for L in layers:
        y1 = B.exl3_gemm_int8act(L["codes"], K, cb, L["m"], L["n"], L["s_in"], L["s_out"], L["scales"], L["x"])
        torch.cuda.synchronize()
        assert float((y1.float() - L["y"].float()).abs().max()) <= 2.0 ** -9 * float(y1.float().abs().max())


def test_int8act_without_rotations():
    """s_in and s_out absent: x itself is quantized, no output transform."""
    m, n, K, cb, M = 512, 1024, 3, 1, 2
    inp = synth.layer_inputs(m, n, K, M, config=88, index=0)
    d = upload(inp)
    y = B.exl3_gemm_int8act(d["codes"], K, cb, m, n, None, None, d["scales"], d["x"])
    torch.cuda.synchronize()
    q, qs = O.quantize_act(inp["x"])
    ref = O.layer_forward_int8(inp["codes"], K, cb, m, n, None, inp["scales"], q, qs)
    assert_layer_close(y, ref, "no rotation")


def test_int8act_grouped_batch_32():
    """32 rows: four batch chunks of eight through the grouped call."""
    K, cb, M = 2, 1, 32
    shapes = [(256, 512), (128, 512)]
    layers, refs = [], []
    for i, (m, n) in enumerate(shapes):
        inp = synth.layer_inputs(m, n, K, M, config=89, index=i)
        d = upload(inp)
        layers.append(dict(codes=d["codes"], m=m, n=n, s_in=d["s_in"], s_out=d["s_out"], scales=d["scales"],
                           x=d["x"], y=torch.empty((M, m), dtype=torch.float16, device="cuda")))
        xt = O.rht(inp["x"].astype(np.float64), inp["s_in"]).astype(np.float16)
        q, qs = O.quantize_act(xt)
        refs.append(O.layer_forward_int8(inp["codes"], K, cb, m, n, inp["s_out"], inp["scales"], q, qs))
    B.exl3_gemm_int8act_grouped(layers, K, cb)
    torch.cuda.synchronize()
    for L, ref in zip(layers, refs):
        assert_layer_close(L["y"], ref, f"grouped M=32 {L['m']}x{L['n']}")


@pytest.mark.parametrize("M", [1, 2, 3])
def test_int8act_multi_code_group(M):
    """Layers of every K and both byte-sum codes, classes interleaved, in one
    exl3_gemm_int8act_multi call: each layer within tolerance of the oracle's
    quantize-then-layer, and within one binary16 rounding of its own
    exl3_gemm_int8act call; the marshalled-once object gives the same."""
    kcs = [(2, 1), (3, 3), (2, 1), (1, 3), (4, 1), (5, 3), (6, 1), (7, 3), (8, 1), (3, 3), (2, 3)]
    shapes = [(256, 512), (128, 1024), (384, 256), (128, 128), (256, 384), (128, 256), (128, 512),
              (256, 128), (128, 256), (512, 256), (128, 640)]
    layers, refs = [], []
    for i, ((K, cb), (m, n)) in enumerate(zip(kcs, shapes)):
        inp = synth.layer_inputs(m, n, K, M, config=91, index=100 * M + i)
        d = upload(inp)
        layers.append(dict(codes=d["codes"], m=m, n=n, K=K, cb=cb, s_in=d["s_in"], s_out=d["s_out"],
                           scales=d["scales"], x=d["x"],
                           y=torch.full((M, m), float("nan"), dtype=torch.float16, device="cuda")))
        xt = O.rht(inp["x"].astype(np.float64), inp["s_in"]).astype(np.float16)
        q, qs = O.quantize_act(xt)
        refs.append(O.layer_forward_int8(inp["codes"], K, cb, m, n, inp["s_out"], inp["scales"], q, qs))
    ws = torch.zeros(B.exl3_multi_i8_workspace_bytes(shapes, M), dtype=torch.uint8, device="cuda")
    B.exl3_gemm_int8act_multi(layers, workspace=ws)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0
    for L, ref in zip(layers, refs):
        assert_layer_close(L["y"], ref, f"multi K{L['K']} cb{L['cb']} {L['m']}x{L['n']} M={M}")
    for L in layers:
        y1 = B.exl3_gemm_int8act(L["codes"], L["K"], L["cb"], L["m"], L["n"], L["s_in"], L["s_out"], L["scales"],
                                 L["x"])
        torch.cuda.synchronize()
        assert float((y1.float() - L["y"].float()).abs().max()) <= 2.0 ** -9 * float(y1.float().abs().max())
    first = [L["y"].clone() for L in layers]
    obj = B.Exl3LinearMulti(layers, int8=True)
    for L in layers:
        L["y"].fill_(float("nan"))
    obj()
    obj()  # the workspace is left clean for the next call
    torch.cuda.synchronize()
    for L, y0 in zip(layers, first):
        assert float((y0.float() - L["y"].float()).abs().max()) <= 2.0 ** -9 * float(y0.float().abs().max())


@pytest.mark.parametrize("M", [1, 3])
def test_int8act_multi_repeated_calls_see_new_x(M):
    """As the binary16 multi-code test: a second call of the same object after
    new activations are written into the same x tensors follows the new x."""
    kcs = [(2, 1), (3, 3), (2, 3), (4, 1)]
    shapes = [(1024, 2048), (512, 1024), (768, 1024), (256, 512)]
    layers, inps = [], []
    for i, ((m, n), (K, cb)) in enumerate(zip(shapes, kcs)):
        inp = synth.layer_inputs(m, n, K, M, config=151 + M, index=i)
        d = upload(inp)
        d.update(m=m, n=n, K=K, cb=cb, y=torch.full((M, m), float("nan"), dtype=torch.float16, device="cuda"))
        layers.append(d)
        inps.append(inp)
    obj = B.Exl3LinearMulti(layers, int8=True)
    for call in range(2):
        if call:
            for i, (d, inp) in enumerate(zip(layers, inps)):
                inp["x"] = synth.activations(M, d["n"], synth.seed_for(161 + M, i))
                d["x"].copy_(torch.from_numpy(inp["x"]).to("cuda"))
        obj()
        torch.cuda.synchronize()
        for i, (d, inp) in enumerate(zip(layers, inps)):
            xt = O.rht(inp["x"].astype(np.float64), inp["s_in"]).astype(np.float16)
            q, qs = O.quantize_act(xt)
            ref = O.layer_forward_int8(inp["codes"], d["K"], d["cb"], d["m"], d["n"], inp["s_out"], inp["scales"],
                                       q, qs)
            assert_layer_close(d["y"], ref, f"call {call} layer {i} K{d['K']} cb{d['cb']}")


def test_int8act_multi_one_k_launch():
    """Batch 1, the 1MAD and mul1 layers of K = 2 large enough for 32-tile
    sub-units share one launch (one loop per code), with a ragged row (72 tile
    columns) and a K = 3 layer on its own kernel: every output within one
    binary16 rounding of its own exl3_gemm_int8act call (parity-tested against
    the oracle above), the small layers also against the oracle."""
    spec = [(14336, 4096, 2, 1), (4096, 4096, 2, 3), (1024, 1152, 2, 3), (1024, 4096, 3, 1),
            (1024, 4096, 2, 1)]
    layers, inps = [], []
    for i, (m, n, K, cb) in enumerate(spec):
        inp = synth.layer_inputs(m, n, K, 1, config=181, index=i)
        d = upload(inp)
        d.update(m=m, n=n, K=K, cb=cb, y=torch.full((1, m), float("nan"), dtype=torch.float16, device="cuda"))
        layers.append(d)
        inps.append(inp)
    B.exl3_gemm_int8act_multi(layers)
    torch.cuda.synchronize()
    for i, (d, inp) in enumerate(zip(layers, inps)):
        y1 = B.exl3_gemm_int8act(d["codes"], d["K"], d["cb"], d["m"], d["n"], d["s_in"], d["s_out"], d["scales"],
                                 d["x"])
        torch.cuda.synchronize()
        assert float((y1.float() - d["y"].float()).abs().max()) <= 2.0 ** -9 * float(y1.float().abs().max())
        if d["m"] * d["n"] <= 1024 * 4096:
            xt = O.rht(inp["x"].astype(np.float64), inp["s_in"]).astype(np.float16)
            q, qs = O.quantize_act(xt)
            ref = O.layer_forward_int8(inp["codes"], d["K"], d["cb"], d["m"], d["n"], inp["s_out"], inp["scales"],
                                       q, qs)
            assert_layer_close(d["y"], ref, f"layer {i} K{d['K']} cb{d['cb']}")
