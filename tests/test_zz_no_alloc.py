"""exl3_gemv_noalloc: the batch-1 layer for callers that cannot allocate device
memory (host callbacks, allocator hooks, plugins whose host framework owns
every allocation, loops that must never allocate).  Instead of a workspace it
uses the library's own fixed device scratch array.

Its output must agree with exl3_gemv's (same inputs, caller-provided
workspace) within the layer tolerance of the other GPU tests, on two calls in
a row (the second call runs on the scratch the first one left behind).  This
file is collected last so that a run stopping at its first failure has already
run every other test.
"""
import numpy as np
import pytest
import torch

from oracle import exl3_oracle as O
from trellis_decode_gemv_gb300 import binding as B
from trellis_decode_gemv_gb300 import synth
from tests.gpu_helpers import assert_layer_close, upload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("m,n,K,cb", [
    (4096, 4096, 2, 1),      # x pairs, many K-splits into the row sums
    (1024, 14336, 3, 0),
    (81920, 256, 4, 1),      # 320 KB of row sums, one tile column per row block
    (256, 384, 8, 0),
])
def test_noalloc_matches_gemv_twice(m, n, K, cb):
    inp = synth.layer_inputs(m, n, K, 1, config=70, index=K + 10 * cb)
    d = upload(inp)
    x = d["x"].view(-1)
    ref = B.exl3_gemv(d["codes"], K, cb, m, n, d["s_in"], d["s_out"], d["scales"], x)
    torch.cuda.synchronize()
    ref64 = ref.double().cpu().numpy()[None, :]
    # the oracle's float64 layer on three 128-row blocks (first, middle, last)
    nb = m // 128
    rbs = sorted({0, nb // 2, nb - 1})
    oref = O.layer_forward_rowblocks(inp["codes"], K, cb, m, n, inp["s_in"], inp["s_out"], inp["scales"],
                                     inp["x"], rbs)
    cols = torch.cat([torch.arange(b * 128, b * 128 + 128) for b in rbs]).cuda()
    for call in range(2):
        y = torch.full((m,), float("nan"), dtype=torch.float16, device="cuda")
        B.exl3_gemv_noalloc(d["codes"], K, cb, m, n, d["s_in"], d["s_out"], d["scales"], x, y=y)
        torch.cuda.synchronize()
        assert_layer_close(y.view(1, -1), ref64, f"noalloc call {call + 1} against exl3_gemv")
        assert_layer_close(y.view(1, -1)[:, cols], oref, f"noalloc call {call + 1} against the oracle")


def test_noalloc_rejects_layers_beyond_its_scratch():
    """Layers whose scratch exceeds the fixed array are refused before anything
    is launched (fake, never-dereferenced device addresses): one through its
    row sums and counters, one through its x pairs alone."""
    lib = B.load_library()
    A = 0x10000
    m = (1 << 20) + 128           # 4 * m bytes of row sums > 4 MiB
    st = lib.exl3_gemv_noalloc(A, 2, 0, m, 128, A, A, A, A, A, None)
    assert st == 10, B.exl3_status_string(st)
    assert "scratch" in B.exl3_status_string(10)
    # 128 rows fit easily; 2^20 columns need 4 MiB of x pairs on top
    st = lib.exl3_gemv_noalloc(A, 2, 0, 128, 1 << 20, A, A, A, A, A, None)
    assert st == 10, B.exl3_status_string(st)
    # an ordinary argument error is still reported as before
    assert lib.exl3_gemv_noalloc(A, 2, 0, 100, 128, A, A, A, A, A, None) == 2
