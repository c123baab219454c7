"""GPU parity of exl3_gemm_grouped: several independent layers in one call.

Each layer's output is checked against the oracle's float64 layer (relative L2
<= 5e-3, |err| <= 1e-2 * max|y_ref|) and against a separate exl3_gemm_small
call on the same inputs (equal up to one binary16 rounding: the fp32 row sums
are added in a different order)."""
import numpy as np
import pytest
import torch

from oracle import exl3_oracle as O
from trellis_decode_gemv_gb300 import binding as B
from trellis_decode_gemv_gb300 import synth
from tests.gpu_helpers import assert_layer_close, upload

pytestmark = pytest.mark.gpu


def _layers(shapes, K, cb, M, config, rot=None):
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


def _check(layers, K, cb, M):
    for inp, d in layers:
        m, n = d["m"], d["n"]
        ref = O.layer_forward(inp["codes"], K, cb, m, n, inp["s_in"], inp["s_out"], inp["scales"], inp["x"])
        assert_layer_close(d["y"], ref, f"{m}x{n}")
        single = B.exl3_gemm_small(d["codes"], K, cb, m, n, d["s_in"], d["s_out"], d["scales"], d["x"])
        torch.cuda.synchronize()
        diff = (single.float() - d["y"].float()).abs().max()
        assert float(diff) <= 2.0 ** -9 * float(single.float().abs().max()) + 1e-6


@pytest.mark.parametrize("M", [1, 2, 5])
@pytest.mark.parametrize("K,cb", [(3, 1), (2, 0), (2, 2), (3, 3)])
def test_grouped_mixed_shapes(M, K, cb):
    shapes = [(256, 384), (384, 1280), (128, 640)]
    layers = _layers(shapes, K, cb, M, config=70 + M)
    B.exl3_gemm_grouped([d for _, d in layers], K, cb)
    torch.cuda.synchronize()
    _check(layers, K, cb, M)


@pytest.mark.parametrize("M", [3, 8])
def test_grouped_forced_warp_shuffle_chunks(M):
    shapes = [(256, 512), (512, 256)]
    layers = _layers(shapes, 4, 1, M, config=75 + M)
    B.exl3_set_path(B.PATH_SHUFFLE)
    try:
        B.exl3_gemm_grouped([d for _, d in layers], 4, 1)
        torch.cuda.synchronize()
    finally:
        B.exl3_set_path(B.PATH_AUTO)
    _check(layers, 4, 1, M)


def test_grouped_rotations_off_and_single_layer():
    shapes = [(256, 256), (384, 512), (128, 128)]
    layers = _layers(shapes, 2, 1, 1, config=79, rot=[(False, True), (True, False), (False, False)])
    B.exl3_gemm_grouped([d for _, d in layers], 2, 1)
    torch.cuda.synchronize()
    _check(layers, 2, 1, 1)
    one = _layers([(640, 384)], 3, 0, 1, config=80)
    B.exl3_gemm_grouped([d for _, d in one], 3, 0)
    torch.cuda.synchronize()
    _check(one, 3, 0, 1)


def test_grouped_attention_projections_sampled():
    """q, k, v of the 8B shapes (4096x4096, 1024x4096, 1024x4096) in one call,
    K = 2, 1MAD, checked on sampled 128-row blocks of every layer; the group
    workspace is reused for a second call."""
    K, cb = 2, 1
    shapes = [(4096, 4096), (1024, 4096), (1024, 4096)]
    layers = _layers(shapes, K, cb, 1, config=81)
    ws = B.alloc_group_workspace(shapes, 1, "cuda")
    for _ in range(2):
        B.exl3_gemm_grouped([d for _, d in layers], K, cb, workspace=ws)
        torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0
    for inp, d in layers:
        m, n = d["m"], d["n"]
        rbs = sorted({0, m // 128 - 1, m // 256})
        ref = O.layer_forward_rowblocks(inp["codes"], K, cb, m, n, inp["s_in"], inp["s_out"],
                                        inp["scales"], inp["x"], rbs)
        cols = torch.cat([torch.arange(b * 128, b * 128 + 128) for b in rbs]).cuda()
        assert_layer_close(d["y"][:, cols], ref, f"{m}x{n}")


def test_group_object_matches_oracle():
    """binding.Exl3LinearGroup: bound x/y tensors, called twice with new x."""
    shapes = [(256, 384), (384, 384)]
    layers = _layers(shapes, 2, 0, 1, config=82)
    grp = B.Exl3LinearGroup([d for _, d in layers], 2, 0)
    grp()
    for inp, d in layers:  # new inputs written into the bound x
        x2 = synth.activations(1, d["n"], seed=synth.seed_for(83, d["m"]))
        d["x"].copy_(torch.from_numpy(x2).cuda())
        inp["x"] = x2
    grp()
    torch.cuda.synchronize()
    _check(layers, 2, 0, 1)


@pytest.mark.parametrize("M", [1, 4])
def test_grouped_many_layers(M):
    """A full group of EXL3_MAX_GROUP layers of mixed shapes (the layers are
    found by binary search over their first units), each checked against a
    separate call; a sample against the oracle."""
    rng = np.random.default_rng(90 + M)
    dims = [128, 256, 384, 640]
    shapes = [(int(rng.choice(dims)), int(rng.choice(dims))) for _ in range(B.MAX_GROUP)]
    layers = _layers(shapes, 2, 1, M, config=90 + M)
    B.exl3_gemm_grouped([d for _, d in layers], 2, 1)
    torch.cuda.synchronize()
    for i, (inp, d) in enumerate(layers):
        m, n = d["m"], d["n"]
        single = B.exl3_gemm_small(d["codes"], 2, 1, m, n, d["s_in"], d["s_out"], d["scales"], d["x"])
        torch.cuda.synchronize()
        diff = (single.float() - d["y"].float()).abs().max()
        assert float(diff) <= 2.0 ** -9 * float(single.float().abs().max()) + 1e-6, f"layer {i} {m}x{n}"
    _check([layers[0], layers[len(layers) // 2], layers[-1]], 2, 1, M)
    with pytest.raises((ValueError, B.Exl3Error)):
        B.exl3_gemm_grouped([d for _, d in layers] + [layers[0][1]], 2, 1)


@pytest.mark.parametrize("M", [1, 2, 3])
def test_multi_code_group(M):
    """Layers of different K and code (every code, K = 1..8) in one
    exl3_gemm_multi call: one chain with a layer kernel per (K, code) class
    at M <= 2, the decode-MMA path per class above; each layer equals a
    separate call, a sample equals the oracle."""
    kcs = [(2, 0), (3, 1), (4, 0), (5, 0), (6, 0), (2, 1), (4, 1), (3, 0), (1, 0), (8, 1), (2, 2), (3, 3)]
    shapes = [(256, 384), (384, 256), (128, 640), (256, 256), (128, 384), (384, 512), (256, 128), (512, 256),
              (128, 256), (256, 256), (384, 128), (128, 512)]
    layers = []
    for i, ((m, n), (K, cb)) in enumerate(zip(shapes, kcs)):
        inp = synth.layer_inputs(m, n, K, M, config=95 + M, index=i)
        d = upload(inp)
        d.update(m=m, n=n, K=K, cb=cb, y=torch.full((M, m), float("nan"), dtype=torch.float16, device="cuda"))
        layers.append((inp, d))
    B.exl3_gemm_multi([d for _, d in layers])
    torch.cuda.synchronize()
    for i, (inp, d) in enumerate(layers):
        m, n, K, cb = d["m"], d["n"], d["K"], d["cb"]
        single = B.exl3_gemm_small(d["codes"], K, cb, m, n, d["s_in"], d["s_out"], d["scales"], d["x"])
        torch.cuda.synchronize()
        diff = (single.float() - d["y"].float()).abs().max()
        assert float(diff) <= 2.0 ** -9 * float(single.float().abs().max()) + 1e-6, f"layer {i} K{K} cb{cb}"
        if i % 4 == 0:
            ref = O.layer_forward(inp["codes"], K, cb, m, n, inp["s_in"], inp["s_out"], inp["scales"], inp["x"])
            assert_layer_close(d["y"], ref, f"layer {i} K{K} cb{cb}")
    # the marshalled-once object: same outputs, written into the bound y
    first = [d["y"].clone() for _, d in layers]
    for _, d in layers:
        d["y"].fill_(float("nan"))
    obj = B.Exl3LinearMulti([d for _, d in layers])
    obj()
    torch.cuda.synchronize()
    for (_, d), y0 in zip(layers, first):
        diff = (y0.float() - d["y"].float()).abs().max()
        assert float(diff) <= 2.0 ** -9 * float(y0.float().abs().max()) + 1e-6


@pytest.mark.parametrize("M", [1, 3])
def test_multi_repeated_calls_see_new_x(M):
    """One marshalled multi-code object called twice with new activations
    written into the same x tensors (the same workspace, so the same x-pair
    scratch): the second call's outputs follow the new x.  The sub-unit
    kernels after a chain's first one do not wait for it before they read x
    pairs, so this checks that they never read the previous call's."""
    kcs = [(2, 0), (3, 1), (2, 1), (4, 0), (2, 0)]
    shapes = [(1024, 2048), (512, 1024), (768, 1024), (256, 512), (1024, 1024)]
    layers, inps = [], []
    for i, ((m, n), (K, cb)) in enumerate(zip(shapes, kcs)):
        inp = synth.layer_inputs(m, n, K, M, config=131 + M, index=i)
        d = upload(inp)
        d.update(m=m, n=n, K=K, cb=cb, y=torch.full((M, m), float("nan"), dtype=torch.float16, device="cuda"))
        layers.append(d)
        inps.append(inp)
    obj = B.Exl3LinearMulti(layers)
    for call in range(2):
        if call:
            for i, (d, inp) in enumerate(zip(layers, inps)):
                inp["x"] = synth.activations(M, d["n"], synth.seed_for(141 + M, i))
                d["x"].copy_(torch.from_numpy(inp["x"]).to("cuda"))
        obj()
        torch.cuda.synchronize()
        for i, (d, inp) in enumerate(zip(layers, inps)):
            ref = O.layer_forward(inp["codes"], d["K"], d["cb"], d["m"], d["n"], inp["s_in"], inp["s_out"],
                                  inp["scales"], inp["x"])
            assert_layer_close(d["y"], ref, f"call {call} layer {i} K{d['K']} cb{d['cb']}")


@pytest.mark.parametrize("case", ["K2 codes in one launch", "K6 codes in one launch",
                                  "K2 codes, 3 rows on the warp-shuffle path"])
def test_multi_class_launches_sampled(case):
    """Batch 1: the classes of one K whose tiles are enough for 32-tile
    sub-units share one launch (one loop per code), the other classes run
    one launch each.  Layers interleave K and codes and include a ragged row
    (72 tile columns); sampled 128-row blocks of each output against the
    oracle, and every output against separate calls.  With 3 rows on the
    warp-shuffle kernels the one-row chunk after the two-row one takes the
    shared launch."""
    M = 3 if "3 rows" in case else 1
    if case.startswith("K2"):
        spec = [(14336, 4096, 2, 0), (1024, 4096, 2, 3), (4096, 4096, 4, 1), (1024, 4096, 3, 1),
                (4096, 4096, 2, 2), (1024, 1152, 3, 0), (1024, 4096, 2, 1), (4096, 4096, 6, 0)]
    else:
        spec = [(14336, 4096, 6, 0), (4096, 4096, 6, 1), (1024, 4096, 6, 0), (1024, 1152, 6, 3),
                (1024, 4096, 2, 1)]
    layers = []
    for i, (m, n, K, cb) in enumerate(spec):
        inp = synth.layer_inputs(m, n, K, M, config=171 + len(spec) + M, index=i)
        d = upload(inp)
        d.update(m=m, n=n, K=K, cb=cb, y=torch.full((M, m), float("nan"), dtype=torch.float16, device="cuda"))
        layers.append((inp, d))
    if M > 2:
        B.exl3_set_path(B.PATH_SHUFFLE)
    try:
        B.exl3_gemm_multi([d for _, d in layers])
        singles = [B.exl3_gemm_small(d["codes"], d["K"], d["cb"], d["m"], d["n"], d["s_in"], d["s_out"],
                                     d["scales"], d["x"]) for _, d in layers]
        torch.cuda.synchronize()
    finally:
        B.exl3_set_path(B.PATH_AUTO)
    rng = np.random.default_rng(171)
    for i, ((inp, d), single) in enumerate(zip(layers, singles)):
        m, n, K, cb = d["m"], d["n"], d["K"], d["cb"]
        diff = (single.float() - d["y"].float()).abs().max()
        assert float(diff) <= 2.0 ** -9 * float(single.float().abs().max()) + 1e-6, f"layer {i} K{K} cb{cb}"
        nb = m // 128
        rbs = sorted(set([0, nb - 1] + list(rng.integers(0, nb, 2))))
        ref = O.layer_forward_rowblocks(inp["codes"], K, cb, m, n, inp["s_in"], inp["s_out"], inp["scales"],
                                        inp["x"], rbs)
        cols = torch.cat([torch.arange(b * 128, b * 128 + 128) for b in rbs]).cuda()
        assert_layer_close(d["y"][:, cols], ref, f"layer {i} K{K} cb{cb}")
