"""GPU parity of the tail-biting Viterbi encoder (exl3_encode_tiles) against
the oracle's encoder in its binary32 mode ("Trellis Quantization" Parts seven
and eight): the same words and the same binary32 cost, bit for bit, on
seeded Gaussian sequences; the two-bit mean-squared error the pages print for
the three-instruction code (about 0.069); and the words decoding, through the
library's own tile decoder, to values whose squared error is the cost."""
import numpy as np
import pytest
import torch

from oracle import exl3_encoder as E
from oracle import exl3_oracle as O
from trellis_decode_gemv_gb300 import binding as B
from trellis_decode_gemv_gb300 import synth

pytestmark = pytest.mark.gpu


def _raw_values(cb):
    return O.decode_states(np.arange(1 << O.L, dtype=np.uint32), cb).astype(np.float32)


def _targets(tiles, cb, seed):
    """N(0, 1) samples scaled by the code's rms value, in binary32 (code units)."""
    raw = _raw_values(cb).astype(np.float64)
    sigma = np.sqrt(np.mean(raw ** 2))
    g = synth.activations(tiles, O.STEPS, synth.seed_for(70, seed)).astype(np.float64)
    return (g * sigma).astype(np.float32), sigma


@pytest.mark.parametrize("K,cb", [(1, 0), (2, 0), (2, 1), (3, 2), (4, 3), (6, 1), (8, 0)])
def test_encoder_matches_oracle_bit_for_bit(K, cb):
    tiles = 2
    target, _ = _targets(tiles, cb, 10 * K + cb)
    words, cost = B.exl3_encode_tiles(torch.from_numpy(target).cuda(), K, cb)
    torch.cuda.synchronize()
    words = words.cpu().numpy().view(np.uint32)
    cost = cost.cpu().numpy()
    raw = _raw_values(cb)
    for i in range(tiles):
        w_ref, _, mse = E.encode_tile(target[i], raw, K, dtype=np.float32)
        np.testing.assert_array_equal(words[i], w_ref, err_msg=f"tile {i}")
        assert cost[i] == np.float32(mse * O.STEPS), (i, cost[i], mse * O.STEPS)


def test_two_bit_mse_of_the_three_instruction_code():
    """24 tiles (6144 samples) of a unit Gaussian at K = 2 with 3INST: the
    pages' 0.069, between the rate-distortion bound 1/16 and E8's 0.089."""
    tiles = 24
    target, sigma = _targets(tiles, 0, 99)
    _, cost = B.exl3_encode_tiles(torch.from_numpy(target).cuda(), 2, 0)
    torch.cuda.synchronize()
    mse = float(cost.double().sum()) / (tiles * O.STEPS) / sigma ** 2
    assert 0.0625 < mse < 0.075, mse
    assert mse == pytest.approx(0.069, abs=0.004)


def test_words_decode_to_the_encoded_values():
    """64 tiles as one 128 x 128 matrix (tile (I, J) = tile 8I + J): the
    library's decoder turns the words into values whose squared error against
    the target is the returned cost; one workspace slot (tiles in series)
    gives the same words."""
    K, cb, tiles = 3, 1, 64
    target, _ = _targets(tiles, cb, 5)
    t = torch.from_numpy(target).cuda()
    words, cost = B.exl3_encode_tiles(t, K, cb)
    one = torch.empty(B.exl3_encode_workspace_bytes(K, 1), dtype=torch.uint8, device="cuda")
    words1, cost1 = B.exl3_encode_tiles(t, K, cb, workspace=one)
    w = B.exl3_decode_tiles(words.view(-1), K, cb, 128, 128)
    torch.cuda.synchronize()
    assert torch.equal(words, words1) and torch.equal(cost, cost1)
    W = w.float().cpu().numpy().astype(np.float64)
    tiles_vals = W.reshape(8, 16, 8, 16).transpose(0, 2, 1, 3).reshape(tiles, O.STEPS)
    err = ((tiles_vals - target.astype(np.float64)) ** 2).sum(axis=1)
    np.testing.assert_allclose(err, cost.cpu().numpy().astype(np.float64), rtol=1e-5)
