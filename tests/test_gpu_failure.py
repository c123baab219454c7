"""Failure detection of the tensor-core kernels, tested without a GPU fault.

The test hook exl3_debug_stall_tensor_wait leaves the kernel's wait for
operand B unsatisfied (the producer posts nothing).  The bounded wait runs out,
every role stops, tensor memory is freed, and the kernel sets the workspace
status word, which the host reads.  The next call, with the hook off, must be
correct: the context stays usable.
"""
import time

import pytest
import torch

from oracle import exl3_oracle as O
from trellis_decode_gemv_gb300 import binding as B
from trellis_decode_gemv_gb300 import synth
from tests.gpu_helpers import assert_layer_close, upload

pytestmark = pytest.mark.gpu


def _call(d, K, cb, m, n, M, ws):
    y = torch.full((M, m), float("nan"), dtype=torch.float16, device="cuda")
    B.exl3_gemm_small(d["codes"], K, cb, m, n, d["s_in"], d["s_out"], d["scales"], d["x"], y=y,
                      workspace=ws)
    torch.cuda.synchronize()
    return y


@pytest.mark.parametrize("M", [1, 4])
def test_tensor_wait_timeout_sets_status_and_context_survives(M):
    """The decode-MMA kernel with its MMAs never issued (the hook): at M = 1
    the kernel rotates x itself, at M = 4 an image kernel runs first."""
    m, n, K, cb = 384, 1280, 3, 1
    inp = synth.layer_inputs(m, n, K, M, config=90, index=0)
    d = upload(inp)
    ws = B.alloc_workspace(m, n, M, "cuda")
    B.exl3_set_path(B.PATH_TENSOR)
    try:
        B.exl3_debug_stall_tensor_wait(True)
        try:
            t0 = time.perf_counter()
            _call(d, K, cb, m, n, M, ws)
            elapsed = time.perf_counter() - t0
        finally:
            B.exl3_debug_stall_tensor_wait(False)
        print(f"stalled call returned after {elapsed:.3f} s")
        assert B.workspace_status(ws, m) == 1
        assert B.exl3_device_status(ws, 4 * (m // 128)) == 9  # EXL3_ERR_DEVICE_CHECK
        assert elapsed < 60.0
        # no partial sum reached the row sums, no block counter moved
        zacc = ws[256:256 + 4 * M * m].view(torch.float32)
        assert float(zacc.abs().sum()) == 0.0
        assert int(ws[:4 * (m // 128)].view(torch.int32).abs().sum()) == 0
        # clear the status word; the next call is correct
        off = 4 * (m // 128)
        ws[off:off + 4].zero_()
        y = _call(d, K, cb, m, n, M, ws)
        assert B.workspace_status(ws, m) == 0
        assert B.exl3_device_status(ws, 4 * (m // 128)) == 0
        ref = O.layer_forward(inp["codes"], K, cb, m, n, inp["s_in"], inp["s_out"], inp["scales"], inp["x"])
        assert_layer_close(y, ref, "after a timed-out call")
    finally:
        B.exl3_set_path(B.PATH_AUTO)


@pytest.mark.parametrize("prefill", ["fused", "decode_once"])
@pytest.mark.parametrize("m,n,M", [(256, 3200, 90), (384, 512, 300)])
def test_dense_prefill_wait_timeout_sets_status_and_context_survives(m, n, M, prefill):
    """The dense prefill kernel (fused, or from decoded images) with its
    producer stalled: with K split (first shape) the row sums stay zero;
    without (second) nothing is written.  The next call is correct."""
    K, cb = 2, 0
    B.exl3_set_prefill(B.PREFILL_FUSED if prefill == "fused" else B.PREFILL_DECODE_ONCE)
    try:
        _dense_stall(m, n, M, K, cb)
    finally:
        B.exl3_set_prefill(B.PREFILL_AUTO)


def _dense_stall(m, n, M, K, cb):
    inp = synth.layer_inputs(m, n, K, M, config=98, index=0)
    d = upload(inp)
    ws = torch.zeros(B.exl3_gemm_workspace_bytes(m, n, M), dtype=torch.uint8, device="cuda")

    def call():
        y = torch.full((M, m), float("nan"), dtype=torch.float16, device="cuda")
        B.exl3_gemm(d["codes"], K, cb, m, n, d["s_in"], d["s_out"], d["scales"], d["x"], y=y, workspace=ws)
        torch.cuda.synchronize()
        return y

    B.exl3_debug_stall_tensor_wait(True)
    try:
        t0 = time.perf_counter()
        call()
        elapsed = time.perf_counter() - t0
    finally:
        B.exl3_debug_stall_tensor_wait(False)
    print(f"stalled dense call returned after {elapsed:.3f} s")
    assert B.workspace_status(ws, m) == 1
    assert elapsed < 60.0
    zacc = ws[256:256 + 4 * M * m].view(torch.float32)
    assert float(zacc.abs().sum()) == 0.0
    off = 4 * (m // 128)
    ws[off:off + 4].zero_()
    y = call()
    assert B.workspace_status(ws, m) == 0
    ref = O.layer_forward(inp["codes"], K, cb, m, n, inp["s_in"], inp["s_out"], inp["scales"], inp["x"])
    assert_layer_close(y, ref, "dense after a timed-out call")
