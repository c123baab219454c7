"""GPU parity of exl3_gemm at prefill batches (M > 32) against the oracle's
float64 layer (relative L2 <= 5e-3, |err| <= 1e-2 * max|y_ref|), for both
prefill strategies:

* fused (the default up to 256 rows): the dense tcgen05 kernel with eight
  decode warps that turn each stage's codes into the binary16 operand-A image
  in shared memory, over batch tiles of 64 rows (M <= 64), 128 (M <= 128) or
  256;
* decode-once (the default above 256 rows): the matrix decoded once into
  binary16 operand images, then the dense tcgen05 kernel over batch tiles
  (one tile of 64 rows up to M = 64, one of 128 up to M = 128, tiles of 256
  above).  Both dense variants finish the
  layer from tensor memory when every unit covers all of K (n < 1024 here) or
  adding partial sums of K splits, the last split finishing the block
  (n >= 1024 with few row blocks);
* passes (EXL3_PATH_TENSOR): passes of 128 rows through the tensor-core kernel
  with 128 batch columns per MMA, decoding into tensor memory per pass.

Batches cover full tiles, partial tiles (33..255 rows), several tiles, and
(for the passes) last passes small enough for the skinny kernel."""
import numpy as np
import pytest
import torch

from oracle import exl3_oracle as O
from trellis_decode_gemv_gb300 import binding as B
from trellis_decode_gemv_gb300 import synth
from tests.gpu_helpers import assert_layer_close, upload

pytestmark = pytest.mark.gpu


_PREFILL = {"fused": B.PREFILL_FUSED, "decode_once": B.PREFILL_DECODE_ONCE}


def _select(strategy):
    B.exl3_set_path(B.PATH_TENSOR if strategy == "passes" else B.PATH_AUTO)
    B.exl3_set_prefill(_PREFILL.get(strategy, B.PREFILL_AUTO))


def _reset():
    B.exl3_set_path(B.PATH_AUTO)
    B.exl3_set_prefill(B.PREFILL_AUTO)


@pytest.fixture(params=["fused", "decode_once", "passes"])
def strategy(request):
    _select(request.param)
    yield request.param
    _reset()


@pytest.fixture(params=["fused", "decode_once"])
def dense_strategy(request):
    _select(request.param)
    yield request.param
    _reset()


def _run(inp, K, cb, m, n, M, ws=None):
    d = upload(inp)
    if ws is None:
        ws = torch.zeros(B.exl3_gemm_workspace_bytes(m, n, M), dtype=torch.uint8, device="cuda")
    y = torch.full((M, m), float("nan"), dtype=torch.float16, device="cuda")
    B.exl3_gemm(d["codes"], K, cb, m, n, d["s_in"], d["s_out"], d["scales"], d["x"], y=y, workspace=ws)
    torch.cuda.synchronize()
    assert B.workspace_status(ws, m) == 0
    return y, ws


def _dense_scratch_left_zero(ws, m, n, M):
    """fp32 row sums and the K-split arrival counters of the dense path are
    zero after a call (workspace layout of exl3_gemm_workspace_bytes)."""
    a256 = lambda b: (b + 255) // 256 * 256  # noqa: E731
    tiles = (M + 255) // 256
    zacc = a256(4 * (m // 128 + 1))
    cnt = zacc + a256(4 * M * m) + a256(2 * tiles * 256 * n) + a256(2 * m * n)
    assert float(ws[zacc:zacc + 4 * M * m].view(torch.float32).abs().sum()) == 0.0
    assert int(ws[cnt:cnt + 4 * (m // 128) * tiles].view(torch.int32).abs().sum()) == 0


def _ref(inp, K, cb, m, n):
    return O.layer_forward(inp["codes"], K, cb, m, n, inp["s_in"], inp["s_out"], inp["scales"], inp["x"])


@pytest.mark.parametrize("M", [33, 64, 65, 100, 128, 129, 160, 256, 300, 513])
def test_prefill_batches(strategy, M):
    m, n, K, cb = 256, 384, 3, 1
    inp = synth.layer_inputs(m, n, K, M, config=90, index=M)
    y, _ = _run(inp, K, cb, m, n, M)
    assert_layer_close(y, _ref(inp, K, cb, m, n), f"{strategy} M={M}")


@pytest.mark.parametrize("cb", [0, 1, 2, 3])
@pytest.mark.parametrize("K", [1, 2, 4, 8])
def test_prefill_codes_and_widths(strategy, K, cb):
    m, n, M = 384, 512, 64
    inp = synth.layer_inputs(m, n, K, M, config=91, index=10 * K + cb)
    y, _ = _run(inp, K, cb, m, n, M)
    assert_layer_close(y, _ref(inp, K, cb, m, n), f"{strategy} K={K} cb={cb}")


@pytest.mark.parametrize("K,cb", [(3, 0), (5, 2), (6, 3), (7, 1)])
def test_prefill_split_k(strategy, K, cb):
    """Few row blocks and long rows: the dense kernel splits K (50 stages of
    64 columns: three splits of 16, 17 and 17 from decoded images, ten of five
    fused) and the last split of each block finishes it."""
    m, n, M = 256, 3200, 90
    inp = synth.layer_inputs(m, n, K, M, config=95, index=K)
    y, ws = _run(inp, K, cb, m, n, M)
    assert_layer_close(y, _ref(inp, K, cb, m, n), f"{strategy} split K={K}")
    if strategy != "passes":
        _dense_scratch_left_zero(ws, m, n, M)


def test_prefill_split_k_several_tiles(dense_strategy):
    """K split with three batch tiles (the last ragged) and repeated calls on
    one workspace: every (block, tile) counter is reset for the next call."""
    m, n, K, cb, M = 384, 2048, 2, 1, 600
    inp = synth.layer_inputs(m, n, K, M, config=99, index=0)
    ref = _ref(inp, K, cb, m, n)
    y, ws = _run(inp, K, cb, m, n, M)
    assert_layer_close(y, ref, "split, 3 tiles")
    for _ in range(2):
        y, _ = _run(inp, K, cb, m, n, M, ws)
        assert_layer_close(y, ref, "split, 3 tiles, workspace reused")
    _dense_scratch_left_zero(ws, m, n, M)


def test_prefill_no_rotation(strategy):
    """s_in and s_out absent: y = binary16(scale (.) (W-hat x))."""
    m, n, K, cb, M = 384, 1024, 2, 0, 70
    inp = synth.layer_inputs(m, n, K, M, config=96, index=0)
    d = upload(inp)
    ws = torch.zeros(B.exl3_gemm_workspace_bytes(m, n, M), dtype=torch.uint8, device="cuda")
    y = B.exl3_gemm(d["codes"], K, cb, m, n, None, None, d["scales"], d["x"], workspace=ws)
    torch.cuda.synchronize()
    ref = O.layer_forward(inp["codes"], K, cb, m, n, None, None, inp["scales"], inp["x"])
    assert_layer_close(y, ref, f"{strategy} no rotation")


def test_prefill_ragged_chunks_and_workspace_reuse(strategy):
    """n/128 odd, two calls on one workspace, row sums left at zero."""
    m, n, K, cb, M = 640, 1152, 2, 0, 150
    inp = synth.layer_inputs(m, n, K, M, config=92, index=0)
    y1, ws = _run(inp, K, cb, m, n, M)
    y2, _ = _run(inp, K, cb, m, n, M, ws)
    assert float((y1.float() - y2.float()).abs().max()) <= 2.0 ** -9 * float(y1.float().abs().max())
    if strategy != "passes":
        _dense_scratch_left_zero(ws, m, n, M)
    else:  # fp32 row sums [128][m] after the counters
        assert float(ws[256:256 + 4 * 128 * m].view(torch.float32).abs().sum()) == 0.0
    assert_layer_close(y2, _ref(inp, K, cb, m, n))


def test_prefill_large_sampled(strategy):
    """4096 x 4096, K = 2, 1MAD, 512 rows (two dense tiles, four passes),
    sampled blocks and rows."""
    m = n = 4096
    K, cb, M = 2, 1, 512
    inp = synth.layer_inputs(m, n, K, M, config=93, index=0)
    y, _ = _run(inp, K, cb, m, n, M)
    rbs = [0, 17, 31]
    rows = [0, 200, 255, 256, 511]
    x = inp["x"][rows]
    ref = O.layer_forward_rowblocks(inp["codes"], K, cb, m, n, inp["s_in"], inp["s_out"], inp["scales"], x, rbs)
    cols = torch.cat([torch.arange(b * 128, b * 128 + 128) for b in rbs]).cuda()
    assert_layer_close(y[rows][:, cols], ref, f"{strategy} 4096x4096 M=512")


def test_prefill_full_width_single_pass_dense(dense_strategy):
    """Enough row blocks for one unit per CTA without a K split: 9728 x 512,
    300 rows (152 units of 128 rows x 256 batch rows), every output checked."""
    m, n, K, cb, M = 9728, 512, 2, 3, 300
    inp = synth.layer_inputs(m, n, K, M, config=97, index=0)
    y, _ = _run(inp, K, cb, m, n, M)
    assert_layer_close(y, _ref(inp, K, cb, m, n), "9728x512 M=300")


def test_small_batches_go_through_gemm_small():
    m, n, K, cb, M = 256, 256, 2, 1, 7
    inp = synth.layer_inputs(m, n, K, M, config=94, index=0)
    y, _ = _run(inp, K, cb, m, n, M)
    assert_layer_close(y, _ref(inp, K, cb, m, n))


def test_prefill_passes_repeated_1mad_block_sums():
    """Back-to-back 128-row passes with the 1MAD correction: each pass's MMA
    kernel reads the block sums the operand-image kernel before it writes, so
    every call, repeated, must match on every row."""
    m, n, K, cb, M = 256, 384, 3, 1, 513
    inp = synth.layer_inputs(m, n, K, M, config=90, index=M)
    ref = _ref(inp, K, cb, m, n)
    B.exl3_set_path(B.PATH_TENSOR)
    try:
        d = upload(inp)
        ws = torch.zeros(B.exl3_gemm_workspace_bytes(m, n, M), dtype=torch.uint8, device="cuda")
        ys = [torch.empty((M, m), dtype=torch.float16, device="cuda") for _ in range(6)]
        for y in ys:
            B.exl3_gemm(d["codes"], K, cb, m, n, d["s_in"], d["s_out"], d["scales"], d["x"], y=y, workspace=ws)
        torch.cuda.synchronize()
        for i, y in enumerate(ys):
            got = y.float().cpu().numpy()
            row_err = np.linalg.norm(got - ref, axis=1) / np.linalg.norm(ref, axis=1)
            assert np.all(row_err <= 5e-3), (i, np.nonzero(row_err > 5e-3)[0][:8])
    finally:
        B.exl3_set_path(B.PATH_AUTO)


def test_prefill_two_rounds_of_units(dense_strategy):
    """228 units (76 row blocks x 3 tiles) over 152 CTAs: two rounds, the
    second partial; every output checked, scratch left at zero, workspace
    reused."""
    m, n, K, cb, M = 9728, 2048, 2, 1, 600
    inp = synth.layer_inputs(m, n, K, M, config=87, index=0)
    ref = _ref(inp, K, cb, m, n)
    y, ws = _run(inp, K, cb, m, n, M)
    assert_layer_close(y, ref, "tail split")
    y2, _ = _run(inp, K, cb, m, n, M, ws)
    assert_layer_close(y2, ref, "tail split, workspace reused")
    _dense_scratch_left_zero(ws, m, n, M)


@pytest.mark.parametrize("M", [40, 120])
def test_prefill_narrow_tiles_two_rounds_and_split(dense_strategy, M):
    """The 64- and 128-row tiles: 160 row blocks over 152 CTAs (a second,
    partial round), then a layer of two row blocks split in K; every output
    checked, scratch left at zero."""
    for m, n, cfg in [(20480, 256, 0), (256, 3200, 1)]:
        K, cb = 2, 1
        inp = synth.layer_inputs(m, n, K, M, config=86, index=2 * M + cfg)
        ref = _ref(inp, K, cb, m, n)
        y, ws = _run(inp, K, cb, m, n, M)
        assert_layer_close(y, ref, f"{m}x{n} M={M}")
        _dense_scratch_left_zero(ws, m, n, M)


@pytest.mark.parametrize("M", [100, 200])
@pytest.mark.parametrize("K,cb", [(2, 0), (3, 2), (4, 3), (5, 1)])
def test_prefill_fused_codes_on_wide_tiles(K, cb, M):
    """The fused kernel's 128- and 256-row tiles with every code: the
    three-instruction codes as defined binary16 weights, the byte-sum codes as
    exact centred sums with the scale applied to z."""
    _select("fused")
    try:
        m, n = 384, 640
        inp = synth.layer_inputs(m, n, K, M, config=85, index=10 * K + cb + M)
        y, ws = _run(inp, K, cb, m, n, M)
        assert_layer_close(y, _ref(inp, K, cb, m, n), f"fused K={K} cb={cb} M={M}")
        _dense_scratch_left_zero(ws, m, n, M)
    finally:
        _reset()
