"""GPU parity of the tensor-core (tcgen05) layer kernel against the CPU oracle.

The kernel family is forced with exl3_set_path(EXL3_PATH_TENSOR) so every
batch size, including 1, runs on decoded tiles in TMEM feeding tcgen05 MMAs.
Criteria as for the other layer tests: relative L2 error <= 5e-3 and every
|err| <= 1e-2 * max|y_ref| against the oracle's float64 layer.
"""
import numpy as np
import pytest
import torch

from oracle import exl3_oracle as O
from trellis_decode_gemv_gb300 import binding as B
from trellis_decode_gemv_gb300 import synth
from tests.gpu_helpers import assert_layer_close, upload

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def tensor_path():
    B.exl3_set_path(B.PATH_TENSOR)
    yield
    B.exl3_set_path(B.PATH_AUTO)


def _run(inp, K, cb, m, n, M, use_in=True, use_out=True):
    d = upload(inp)
    ws = B.alloc_workspace(m, n, M, "cuda")
    y = torch.full((M, m), float("nan"), dtype=torch.float16, device="cuda")
    B.exl3_gemm_small(d["codes"], K, cb, m, n, d["s_in"] if use_in else None,
                      d["s_out"] if use_out else None, d["scales"], d["x"], y=y, workspace=ws)
    torch.cuda.synchronize()
    assert B.workspace_status(ws, m) == 0, "device-side wait timed out"
    return y


def _ref(inp, K, cb, m, n, use_in=True, use_out=True):
    return O.layer_forward(inp["codes"], K, cb, m, n, inp["s_in"] if use_in else None,
                           inp["s_out"] if use_out else None, inp["scales"], inp["x"])


@pytest.mark.parametrize("K", range(1, 9))
@pytest.mark.parametrize("cb", [0, 1, 2, 3])
def test_tc_all_widths_batch1(K, cb):
    m, n = 256, 384
    inp = synth.layer_inputs(m, n, K, 1, config=80, index=10 * K + cb)
    assert_layer_close(_run(inp, K, cb, m, n, 1), _ref(inp, K, cb, m, n), f"K={K} cb={cb}")


@pytest.mark.parametrize("M", [1, 2, 3, 8, 13, 16, 17, 32])
@pytest.mark.parametrize("cb", [0, 1, 2, 3])
def test_tc_batches(M, cb):
    m, n, K = 384, 1280, 3
    inp = synth.layer_inputs(m, n, K, M, config=81, index=M + 100 * cb)
    assert_layer_close(_run(inp, K, cb, m, n, M), _ref(inp, K, cb, m, n), f"M={M}")


@pytest.mark.parametrize("use_in,use_out", [(False, False), (True, False), (False, True)])
def test_tc_without_rotations(use_in, use_out):
    m, n, K, cb = 256, 512, 2, 1
    inp = synth.layer_inputs(m, n, K, 2, config=82, index=2 * use_in + use_out)
    y = _run(inp, K, cb, m, n, 2, use_in, use_out)
    assert_layer_close(y, _ref(inp, K, cb, m, n, use_in, use_out))


@pytest.mark.parametrize("m,n,K,cb,M", [
    (4096, 4096, 2, 1, 1), (1024, 4096, 4, 0, 1), (14336, 4096, 3, 1, 8),
    (4096, 14336, 3, 1, 32), (8192, 8192, 2, 0, 1),
])
def test_tc_large_sampled(m, n, K, cb, M):
    inp = synth.layer_inputs(m, n, K, M, config=83, index=m // 128 + K)
    y = _run(inp, K, cb, m, n, M)
    nb = m // 128
    rbs = sorted({0, nb - 1, nb // 2})
    ref = O.layer_forward_rowblocks(inp["codes"], K, cb, m, n, inp["s_in"], inp["s_out"],
                                    inp["scales"], inp["x"], rbs)
    cols = torch.cat([torch.arange(b * 128, b * 128 + 128) for b in rbs]).cuda()
    assert_layer_close(y[:, cols], ref, f"{m}x{n} M={M}")


def test_tc_matches_shuffle_path():
    """Both kernel families agree with each other within the tolerance."""
    m, n, K, cb = 2048, 3072, 4, 0
    inp = synth.layer_inputs(m, n, K, 1, config=84, index=0)
    y_tc = _run(inp, K, cb, m, n, 1)
    B.exl3_set_path(B.PATH_SHUFFLE)
    y_sh = _run(inp, K, cb, m, n, 1)
    assert_layer_close(y_tc, y_sh.double().cpu().numpy())


def test_tc_workspace_reuse_and_row_sums_cleared():
    """Two calls in a row on one workspace agree within one binary16 rounding
    (fp32 reductions land in any order) and leave the row sums at zero; the
    1024 x 4096 layer has 256 chunks, so the work ranges of the 152-CTA grid
    straddle row blocks."""
    m, n, K, cb, M = 1024, 4096, 3, 1, 5
    inp = synth.layer_inputs(m, n, K, M, config=85, index=0)
    d = upload(inp)
    ws = B.alloc_workspace(m, n, M, "cuda")
    ys = []
    for _ in range(2):
        y = torch.full((M, m), float("nan"), dtype=torch.float16, device="cuda")
        B.exl3_gemm_small(d["codes"], K, cb, m, n, d["s_in"], d["s_out"], d["scales"], d["x"],
                          y=y, workspace=ws)
        torch.cuda.synchronize()
        ys.append(y)
    assert B.workspace_status(ws, m) == 0
    diff = (ys[0].float() - ys[1].float()).abs()
    assert float(diff.max()) <= 2.0 ** -9 * float(ys[0].float().abs().max())
    zacc = ws[256:256 + 4 * M * m].view(torch.float32)
    assert float(zacc.abs().sum()) == 0.0
    assert_layer_close(ys[1], _ref(inp, K, cb, m, n), "second call")
