"""GPU parity: tile decode (bit-exact) and the standalone randomized Hadamard
transforms, against the CPU oracle, through the C ABI.

Decode must match the oracle's binary16 W-hat bit for bit ("Trellis
Quantization" Parts eight and nine: one defined value per state).  The
transforms are compared with the oracle's float64 result; the GPU output is
rounded once to binary16, so each element may differ by at most half a
binary16 ulp plus fp32 accumulation noise.
"""
import numpy as np
import pytest
import torch

from oracle import exl3_oracle as O
from trellis_decode_gemv_gb300 import binding as B
from trellis_decode_gemv_gb300 import synth
from tests.gpu_helpers import to_dev

pytestmark = pytest.mark.gpu


def _decode_gpu(codes, K, cb, m, n):
    d = to_dev(codes)
    w = torch.full((m, n), float("nan"), dtype=torch.float16, device="cuda")
    B.exl3_decode_tiles(d, K, cb, m, n, out=w)
    torch.cuda.synchronize()
    return w


@pytest.mark.parametrize("K", range(1, 9))
@pytest.mark.parametrize("cb", [0, 1, 2, 3])
@pytest.mark.parametrize("m,n", [(128, 128), (256, 384)])
def test_decode_bit_exact_small(K, cb, m, n):
    codes = synth.packed_codes(m, n, K, synth.seed_for(50, 10 * K + cb))
    w = _decode_gpu(codes, K, cb, m, n).cpu().numpy().view(np.uint16)
    ref = O.decode_tiles(codes, K, cb, m, n).view(np.uint16)
    np.testing.assert_array_equal(w, ref)


def _every_state_codes():
    """K = 8 streams whose windows take every 16-bit value: the state of step t
    is stream bytes t and t+1, so tile j of the first 256 repeats the bytes
    (j, k) for k = 0..127 and tile j of the next 256 the bytes (j, 128 + k).
    512 tiles: a 128 x 1024 layer."""
    K = 8
    tiles = []
    for half in (0, 128):
        for j in range(256):
            b = np.empty(256, dtype=np.uint8)
            b[0::2] = j
            b[1::2] = half + np.arange(128)
            tiles.append(np.frombuffer(b.tobytes(), dtype=">u4").astype(np.uint32))
    return np.concatenate(tiles), K, 128, 1024


@pytest.mark.parametrize("cb", [0, 1, 2, 3])
def test_decode_every_state_exhaustive(cb):
    """Every one of the 2**16 states decoded on the GPU, bit-exact against the
    oracle."""
    codes, K, m, n = _every_state_codes()
    states = O.tile_states(codes.reshape(-1, 8 * K), K)
    assert len(np.unique(states)) == 1 << 16
    w = _decode_gpu(codes, K, cb, m, n).cpu().numpy().view(np.uint16)
    ref = O.decode_tiles(codes, K, cb, m, n).view(np.uint16)
    np.testing.assert_array_equal(w, ref)


def test_decode_degenerate_streams():
    """All-zero and all-one streams: every state is 0x0000 / 0xFFFF."""
    m = n = 128
    for K in (1, 4, 8):
        for fill in (0, 0xFFFFFFFF):
            codes = np.full((m // 16) * (n // 16) * 8 * K, fill, dtype=np.uint32)
            for cb in (0, 1, 2, 3):
                w = _decode_gpu(codes, K, cb, m, n).cpu().numpy().view(np.uint16)
                np.testing.assert_array_equal(w, O.decode_tiles(codes, K, cb, m, n).view(np.uint16))


@pytest.mark.parametrize("m,n,K,cb", [
    (4096, 4096, 2, 1),       # single 4096x4096 layer
    (1024, 4096, 3, 0),
    (14336, 4096, 4, 1),
    (4096, 14336, 3, 0),
    (28672, 8192, 2, 0),
    (128256, 8192, 6, 0),     # lm_head width
])
def test_decode_bit_exact_sampled_large(m, n, K, cb):
    codes = synth.packed_codes(m, n, K, synth.seed_for(51, m // 128 + K))
    w = _decode_gpu(codes, K, cb, m, n)
    rng = np.random.default_rng(m + n + K)
    trows = np.unique(np.concatenate([[0, m // 16 - 1], rng.integers(0, m // 16, 6)]))
    ref = O.decode_tiles(codes, K, cb, m, n, tile_rows=trows).view(np.uint16)
    rows = (trows[:, None] * 16 + np.arange(16)[None, :]).ravel()
    got = w[torch.from_numpy(rows).cuda()].cpu().numpy().view(np.uint16)
    np.testing.assert_array_equal(got, ref)
    del w
    torch.cuda.empty_cache()


def _assert_half_rounded(got_t, ref):
    got = got_t.float().cpu().numpy().astype(np.float64)
    bound = np.abs(ref) * 2.0 ** -11 * 1.001 + 1e-6
    assert np.all(np.abs(got - ref) <= bound), np.max(np.abs(got - ref) - bound)


@pytest.mark.parametrize("M,d", [(1, 128), (3, 384), (2, 4096), (1, 28672), (32, 14336)])
def test_rht_in_and_out(M, d):
    x = synth.activations(M, d, synth.seed_for(52, d))
    s = synth.sign_vector(d, synth.seed_for(52, d + 1))
    ref = O.rht(x.astype(np.float64), s)
    got = B.exl3_rht_in(to_dev(x), to_dev(s))
    torch.cuda.synchronize()
    _assert_half_rounded(got, ref)
    got2 = B.exl3_rht_out(to_dev(x), to_dev(s))
    torch.cuda.synchronize()
    _assert_half_rounded(got2, ref)


def test_rht_round_trip():
    """Hb is an involution: s (.) Hb(Hb(s (.) x)) returns x up to two binary16
    roundings."""
    d = 1024
    x = synth.activations(4, d, synth.seed_for(53, 0))
    s = synth.sign_vector(d, synth.seed_for(53, 1))
    ones = torch.ones(d, dtype=torch.float16, device="cuda")
    xr = B.exl3_rht_in(to_dev(x), to_dev(s))
    back = B.exl3_rht_in(xr, ones) * to_dev(s)
    torch.cuda.synchronize()
    err = (back.float().cpu().numpy() - x.astype(np.float32))
    assert np.abs(err).max() < 4 * 2.0 ** -10 * np.abs(x).max()
