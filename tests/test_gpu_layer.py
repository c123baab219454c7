"""GPU parity of the fused layer (exl3_gemv / exl3_gemm_small) against the CPU
oracle's float64 layer_forward, through the C ABI.

Criteria: relative L2 error <= 5e-3 and every |err| <= 1e-2 * max|y_ref|.
Small shapes are checked in full (several 128-row blocks, several K-splits,
ragged split sizes); the full-size layer shapes of the benchmark workloads are
checked on sampled 128-row output blocks, in the same launch configuration the
benchmark times.
"""
import numpy as np
import pytest
import torch

from oracle import exl3_oracle as O
from trellis_decode_gemv_gb300 import binding as B
from trellis_decode_gemv_gb300 import synth
from tests.gpu_helpers import assert_layer_close, upload

pytestmark = pytest.mark.gpu


def _run(inp_d, K, cb, m, n, M, use_in=True, use_out=True, ws=None, gemv=False):
    x = inp_d["x"]
    y = torch.full((M, m), float("nan"), dtype=torch.float16, device="cuda")
    s_in = inp_d["s_in"] if use_in else None
    s_out = inp_d["s_out"] if use_out else None
    if gemv:
        B.exl3_gemv(inp_d["codes"], K, cb, m, n, s_in, s_out, inp_d["scales"], x.view(-1),
                    y=y.view(-1), workspace=ws)
    else:
        B.exl3_gemm_small(inp_d["codes"], K, cb, m, n, s_in, s_out, inp_d["scales"], x,
                          y=y, workspace=ws)
    torch.cuda.synchronize()
    return y


@pytest.mark.parametrize("K", range(1, 9))
@pytest.mark.parametrize("cb", [0, 1, 2, 3])
def test_gemv_all_widths(K, cb):
    m, n = 256, 384
    inp = synth.layer_inputs(m, n, K, 1, config=60, index=10 * K + cb)
    y = _run(upload(inp), K, cb, m, n, 1, gemv=True)
    ref = O.layer_forward(inp["codes"], K, cb, m, n, inp["s_in"], inp["s_out"], inp["scales"], inp["x"])
    assert_layer_close(y, ref, f"K={K} cb={cb}")


@pytest.mark.parametrize("m,n", [(128, 128), (128, 4096), (384, 1280), (1024, 640), (640, 2944)])
@pytest.mark.parametrize("K,cb", [(2, 1), (3, 0), (4, 1)])
def test_gemv_shapes(m, n, K, cb):
    inp = synth.layer_inputs(m, n, K, 1, config=61, index=m + n + K)
    y = _run(upload(inp), K, cb, m, n, 1, gemv=True)
    ref = O.layer_forward(inp["codes"], K, cb, m, n, inp["s_in"], inp["s_out"], inp["scales"], inp["x"])
    assert_layer_close(y, ref, f"{m}x{n}")


@pytest.mark.parametrize("use_in,use_out", [(False, False), (True, False), (False, True)])
def test_gemv_without_rotations(use_in, use_out):
    m, n, K, cb = 384, 512, 3, 1
    inp = synth.layer_inputs(m, n, K, 1, config=62, index=int(use_in) * 2 + int(use_out))
    y = _run(upload(inp), K, cb, m, n, 1, use_in, use_out)
    ref = O.layer_forward(inp["codes"], K, cb, m, n, inp["s_in"] if use_in else None,
                          inp["s_out"] if use_out else None, inp["scales"], inp["x"])
    assert_layer_close(y, ref)


def test_unrotated_core_composes_with_standalone_transforms():
    """exl3_rht_in -> core (no rotations, unit scales) -> scale -> exl3_rht_out
    agrees with the fused call within the layer tolerance."""
    m, n, K, cb = 512, 768, 2, 0
    inp = synth.layer_inputs(m, n, K, 1, config=63, index=0)
    d = upload(inp)
    fused = _run(d, K, cb, m, n, 1)
    xr = B.exl3_rht_in(d["x"], d["s_in"])
    ones = torch.ones(m, dtype=torch.float16, device="cuda")
    z = B.exl3_gemm_small(d["codes"], K, cb, m, n, None, None, ones, xr)
    z = (z.float() * d["scales"].float()).half()
    y = B.exl3_rht_out(z, d["s_out"])
    torch.cuda.synchronize()
    ref = O.layer_forward(inp["codes"], K, cb, m, n, inp["s_in"], inp["s_out"], inp["scales"], inp["x"])
    assert_layer_close(fused, ref)
    assert_layer_close(y, ref)


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8, 13, 32])
def test_gemm_small_batches(M):
    m, n, K, cb = 384, 640, 3, 1
    inp = synth.layer_inputs(m, n, K, M, config=64, index=M)
    y = _run(upload(inp), K, cb, m, n, M)
    ref = O.layer_forward(inp["codes"], K, cb, m, n, inp["s_in"], inp["s_out"], inp["scales"], inp["x"])
    assert_layer_close(y, ref, f"M={M}")


@pytest.mark.parametrize("M", [3, 5, 8, 13, 32])
def test_gemm_small_batches_warp_shuffle(M):
    """The warp-shuffle kernel (batch chunks of 8, 4, 2, 1) forced for batches
    that the automatic choice sends to the tensor-core kernel."""
    m, n, K, cb = 384, 640, 2, 0
    inp = synth.layer_inputs(m, n, K, M, config=66, index=M)
    B.exl3_set_path(B.PATH_SHUFFLE)
    try:
        y = _run(upload(inp), K, cb, m, n, M)
    finally:
        B.exl3_set_path(B.PATH_AUTO)
    ref = O.layer_forward(inp["codes"], K, cb, m, n, inp["s_in"], inp["s_out"], inp["scales"], inp["x"])
    assert_layer_close(y, ref, f"M={M}")


@pytest.mark.parametrize("M,cb", [(1, 0), (1, 1), (2, 1), (1, 2), (2, 3)])
def test_large_layer_kernel_full(M, cb):
    """4096 x 10112: at least 1024 tiles per SM, so batch chunks of 1 and 2 run
    the one-CTA-per-SM sub-unit kernel; n/128 = 79 is odd, so the last
    sub-unit of every tile row is the ragged 8-tile one.  Checked in full."""
    m, n, K = 4096, 10112, 2
    inp = synth.layer_inputs(m, n, K, M, config=67, index=M + 10 * cb)
    y = _run(upload(inp), K, cb, m, n, M)
    ref = O.layer_forward(inp["codes"], K, cb, m, n, inp["s_in"], inp["s_out"], inp["scales"], inp["x"])
    assert_layer_close(y, ref, f"M={M} cb={cb}")


def test_workspace_reuse_and_special_inputs():
    """Two calls on one workspace agree (the arrival counters and the fp32 row
    sums are left at zero); x = 0 gives y = 0 exactly; zero scales give 0."""
    m, n, K, cb = 1024, 2048, 2, 0
    inp = synth.layer_inputs(m, n, K, 1, config=65, index=0)
    d = upload(inp)
    ws = B.alloc_workspace(m, n, 1, "cuda")
    y1 = _run(d, K, cb, m, n, 1, ws=ws)
    y2 = _run(d, K, cb, m, n, 1, ws=ws)
    # fp32 atomic accumulation order varies: equal up to one binary16 rounding
    diff = (y1.float() - y2.float()).abs()
    assert float(diff.max()) <= 2.0 ** -9 * float(y1.float().abs().max())
    cnt = ws[:(m // 128) * 4].view(torch.int32)
    assert int(cnt.abs().sum()) == 0
    zacc = ws[256:256 + 4 * m].view(torch.float32)
    assert float(zacc.abs().sum()) == 0.0
    d0 = dict(d, x=torch.zeros_like(d["x"]))
    assert int(_run(d0, K, cb, m, n, 1, ws=ws).float().abs().sum()) == 0
    dz = dict(d, scales=torch.zeros_like(d["scales"]))
    assert int(_run(dz, K, cb, m, n, 1, ws=ws).float().abs().sum()) == 0


def _sampled(name, m, n, K, cb, M, config, index, blocks=3):
    inp = synth.layer_inputs(m, n, K, M, config=config, index=index)
    y = _run(upload(inp), K, cb, m, n, M)
    rng = np.random.default_rng(index + 7)
    nb = m // 128
    rbs = sorted(set([0, nb - 1] + list(rng.integers(0, nb, blocks))))
    ref = O.layer_forward_rowblocks(inp["codes"], K, cb, m, n, inp["s_in"], inp["s_out"],
                                    inp["scales"], inp["x"], rbs)
    cols = torch.cat([torch.arange(b * 128, b * 128 + 128) for b in rbs]).cuda()
    assert_layer_close(y[:, cols], ref, name)


def test_single_4096_layer_full():
    """4096x4096, K=2, 1MAD, batch 1 -- checked on every output."""
    m = n = 4096
    inp = synth.layer_inputs(m, n, 2, 1, config=0, index=0)
    y = _run(upload(inp), 2, 1, m, n, 1, gemv=True)
    ref = O.layer_forward(inp["codes"], 2, 1, m, n, inp["s_in"], inp["s_out"], inp["scales"], inp["x"])
    assert_layer_close(y, ref, "4096x4096")


@pytest.mark.parametrize("case", list(enumerate(synth.llama8b_layer_set())), ids=lambda c: c[1][0])
def test_llama8b_layer_set_sampled(case):
    i, (name, m, n, K, cb) = case
    _sampled(name, m, n, K, cb, 1, config=1, index=i, blocks=2)


@pytest.mark.parametrize("name,m,n", synth.LLAMA70B_SHAPES)
def test_llama70b_shapes_sampled(name, m, n):
    _sampled(name, m, n, 2, 0, 1, config=2, index=m // 128 + n // 128, blocks=2)


@pytest.mark.parametrize("M", synth.BATCH_SWEEP)
@pytest.mark.parametrize("shape", synth.BATCH_SWEEP_SHAPES, ids=lambda s: s[0])
def test_batch_sweep_sampled(M, shape):
    name, m, n, K, cb = shape
    _sampled(f"{name} M={M}", m, n, K, cb, M, config=3, index=M * 10 + (m > n), blocks=2)


@pytest.mark.parametrize("name,m,n,K", [
    ("attn", 8192, 8192, 4), ("gate.K2", 28672, 8192, 2), ("up.K3", 28672, 8192, 3),
    ("down.K4", 8192, 28672, 4), ("down.K3", 8192, 28672, 3), ("lm_head", 128256, 8192, 6),
])
def test_mixed_stack_shapes_sampled(name, m, n, K):
    _sampled(name, m, n, K, 0, 1, config=4, index=K * 1000 + m // 128, blocks=2)


@pytest.mark.parametrize("M", [1, 2])
def test_ragged_units_sampled(M):
    """A long layer with n/16 = 72 tile columns: the batch-1/2 kernel cuts tile
    rows into 16-tile units, so every row ends in a partial unit of 8 tiles."""
    _sampled(f"34688x1152 M={M}", 34688, 1152, 2, 1, M, config=69, index=M, blocks=3)


def test_layer_object_matches_functional_call():
    """binding.Exl3Linear (the layer marshalled once) gives the functional
    call's result, for batch 1 and a smaller batch than it was built for."""
    m, n, K, cb = 512, 768, 3, 1
    inp = synth.layer_inputs(m, n, K, 2, config=68, index=0)
    d = upload(inp)
    lin = B.Exl3Linear(d["codes"], K, cb, m, n, d["s_in"], d["s_out"], d["scales"], max_batch=2)
    y2 = lin(d["x"])
    y1 = lin(d["x"][0])
    torch.cuda.synchronize()
    ref = O.layer_forward(inp["codes"], K, cb, m, n, inp["s_in"], inp["s_out"], inp["scales"], inp["x"])
    assert_layer_close(y2, ref, "batch 2")
    assert_layer_close(y1.view(1, -1), ref[:1], "batch 1")
    with pytest.raises(ValueError):
        lin(torch.zeros(3, n, dtype=torch.float16, device="cuda"))
