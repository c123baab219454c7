"""Pins of the oracle's randomized Hadamard transform and layer forward.

Sources: "ExLlamaV3 & EXL3 Deep Dive" Section 2 (normalized Walsh-Hadamard
matrix with H H^T = I, Rademacher signs, and the runtime identity
y = W x = H^T diag(s_left) (W~ (H diag(s_right) x))); "Trellis Quantization"
Part six (Hadamard entries are only +-1) and Part eleven (128-wide blockwise
rotation).  Pins: scipy's textbook Sylvester construction, exact integer
orthogonality, the inverse transform, the y = W x identity on a dense W, and a
brute-force dense evaluation of the whole layer with a separately written
sequential trellis walker.  The whole-vector variant (QTIP rotates full rows
and columns, Part eleven) is pinned against scipy's full Sylvester matrices,
the Kronecker factorization H_{128B} = H_B (x) H_128, orthogonality, and the
same brute-force layer with full-size matrices.
"""
import numpy as np
import pytest
import scipy.linalg

from oracle import exl3_oracle as O
from trellis_decode_gemv_gb300 import synth


def test_hadamard_is_sylvester_and_orthogonal():
    H = O.hadamard(128)
    np.testing.assert_array_equal(H, scipy.linalg.hadamard(128))
    HHt = (H.astype(np.int64) @ H.T.astype(np.int64))
    np.testing.assert_array_equal(HHt, 128 * np.eye(128, dtype=np.int64))
    assert set(np.unique(H)) == {-1.0, 1.0}


def _dense_blockwise(d, signs=None):
    Hn = scipy.linalg.hadamard(128) / np.sqrt(128)
    B = np.kron(np.eye(d // 128), Hn)
    if signs is not None:
        B = B @ np.diag(np.asarray(signs, dtype=np.float64))
    return B


def test_rht_matches_dense_matrix_and_inverts():
    rng = np.random.default_rng(5)
    for d in (128, 384, 1024):
        v = rng.standard_normal((3, d))
        s = np.where(rng.integers(0, 2, d) == 1, 1.0, -1.0)
        out = O.rht(v, s)
        np.testing.assert_allclose(out, v @ _dense_blockwise(d, s).T, rtol=0, atol=1e-12)
        # Hb is an involution and the signs square to one: s (.) Hb(Hb(s (.) v)) = v
        back = O.rht(out, np.ones(d)) * s
        np.testing.assert_allclose(back, v, rtol=0, atol=1e-12)
        np.testing.assert_array_equal(O.rht(v, None), v)


def test_runtime_identity_recovers_dense_W():
    """Deep Dive Section 2: if W~ = diag(s_l) H_m W diag(s_r) H_n^T (the offline
    form consistent with the runtime identity taken), the runtime computation
    Hb(s_l (.) (W~ Hb(s_r (.) x))) returns W x exactly (to fp64 rounding)."""
    rng = np.random.default_rng(9)
    m, n = 256, 384
    W = rng.standard_normal((m, n))
    sl = np.where(rng.integers(0, 2, m) == 1, 1.0, -1.0)
    sr = np.where(rng.integers(0, 2, n) == 1, 1.0, -1.0)
    Hm = _dense_blockwise(m)
    Hn = _dense_blockwise(n)
    Wt = np.diag(sl) @ Hm @ W @ np.diag(sr) @ Hn.T
    x = rng.standard_normal((2, n))
    y = O.rht(O.rht(x, sr) @ Wt.T, sl)
    np.testing.assert_allclose(y, x @ W.T, rtol=0, atol=1e-10)


def _walk_decode(codes, K, cb, m, n):
    """Brute-force decoder written independently of the oracle's window
    extraction: per tile, turn the words into one big integer, take s_0 as the
    first 16 stream bits, then walk the shift-register recurrence
    s_{t+1} = ((s_t << K) & 0xFFFF) | u_t, where u_t are the K bits that follow
    the current window (wrapping around the end of the circular stream)."""
    nw = 8 * K
    nbits = 256 * K
    tiles = np.asarray(codes).reshape(m // 16, n // 16, nw)
    states = np.zeros((m // 16, n // 16, 256), dtype=np.uint32)
    for I in range(m // 16):
        for J in range(n // 16):
            v = 0
            for w in tiles[I, J]:
                v = (v << 32) | int(w)
            bit = lambda j: (v >> (nbits - 1 - (j % nbits))) & 1  # noqa: E731
            s = 0
            for i in range(16):
                s = (s << 1) | bit(i)
            for t in range(256):
                states[I, J, t] = s
                u = 0
                for i in range(K):
                    u = (u << 1) | bit(K * t + 16 + i)
                s = ((s << K) & 0xFFFF) | u
    vals = O.decode_states(states, cb).astype(np.float64)       # [I, J, 256]
    W = np.zeros((m, n))
    for t in range(256):
        W[(t // 16)::16, (t % 16)::16] = vals[:, :, t]
    return W


@pytest.mark.parametrize("K,cb,m,n,M", [
    (1, 0, 128, 128, 1), (2, 1, 128, 256, 2), (3, 0, 256, 128, 1),
    (4, 1, 128, 128, 3), (5, 0, 128, 128, 1), (6, 1, 128, 128, 1),
    (7, 0, 128, 128, 2), (8, 1, 128, 128, 1),
])
def test_layer_brute_force(K, cb, m, n, M):
    inp = synth.layer_inputs(m, n, K, M, config=90, index=K)
    W = _walk_decode(inp["codes"], K, cb, m, n)
    np.testing.assert_array_equal(
        W, O.decode_tiles(inp["codes"], K, cb, m, n).astype(np.float64))
    A = (_dense_blockwise(m, None) @ np.diag(inp["s_out"].astype(np.float64))
         @ np.diag(inp["scales"].astype(np.float64)) @ W
         @ _dense_blockwise(n, inp["s_in"]))
    y_bf = inp["x"].astype(np.float64) @ A.T
    y = O.layer_forward(inp["codes"], K, cb, m, n, inp["s_in"], inp["s_out"],
                        inp["scales"], inp["x"])
    np.testing.assert_allclose(y, y_bf, rtol=1e-12, atol=1e-12 * np.abs(y_bf).max())


def test_layer_special_cases():
    m, n, K, cb = 256, 384, 3, 1
    inp = synth.layer_inputs(m, n, K, 2, config=91, index=0)
    f = lambda x, **kw: O.layer_forward(inp["codes"], K, cb, m, n,  # noqa: E731
                                        kw.get("s_in", inp["s_in"]), kw.get("s_out", inp["s_out"]),
                                        kw.get("scales", inp["scales"]), x)
    x = inp["x"]
    assert np.all(f(np.zeros_like(x)) == 0)
    assert np.all(f(x, scales=np.zeros(m, dtype=np.float16)) == 0)
    # linear in x (fp64 evaluation of fp16 inputs)
    x1 = x[0:1].astype(np.float64)
    x2 = x[1:2].astype(np.float64)
    np.testing.assert_allclose(f(2 * x1 - 3 * x2), 2 * f(x1) - 3 * f(x2), atol=1e-9)
    # one-hot x with no rotation picks a scaled column of W-hat
    W = O.decode_tiles(inp["codes"], K, cb, m, n).astype(np.float64)
    e = np.zeros((1, n))
    e[0, 77] = 1.0
    col = f(e, s_in=None, s_out=None)
    np.testing.assert_array_equal(col[0], W[:, 77] * inp["scales"].astype(np.float64))


def test_rowblock_sampling_matches_full():
    m, n, K, cb = 512, 256, 2, 0
    inp = synth.layer_inputs(m, n, K, 1, config=92, index=0)
    args = (inp["codes"], K, cb, m, n, inp["s_in"], inp["s_out"], inp["scales"], inp["x"])
    full = O.layer_forward(*args)
    part = O.layer_forward_rowblocks(*args, row_blocks=[3, 1])
    np.testing.assert_allclose(part, np.concatenate([full[:, 384:512], full[:, 128:256]], 1),
                               rtol=1e-13, atol=1e-13)


# ---- QTIP's whole-vector rotation ("Trellis Quantization" Part eleven) -------

@pytest.mark.parametrize("d", [1, 2, 8, 128, 256, 1024])
def test_rht_whole_matches_scipy_sylvester(d):
    """H_d (s (.) v) / sqrt(d) against scipy's Sylvester matrix, row for row."""
    rng = np.random.default_rng(100 + d)
    v = rng.standard_normal((3, d))
    s = np.where(rng.integers(0, 2, d) == 1, 1.0, -1.0)
    ref = (v * s) @ scipy.linalg.hadamard(d).T / np.sqrt(d)
    np.testing.assert_allclose(O.rht_whole(v, s), ref, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(O.rht_whole(v, None), v)


def test_rht_whole_kronecker_and_blockwise():
    """Sylvester order makes H_{128 B} = H_B (x) H_128, so the whole-vector
    transform is the blockwise one followed by a transform across the blocks;
    at d = 128 the two rotations coincide."""
    for B in (2, 4, 8):
        np.testing.assert_array_equal(scipy.linalg.hadamard(128 * B),
                                      np.kron(scipy.linalg.hadamard(B), scipy.linalg.hadamard(128)))
    rng = np.random.default_rng(7)
    d = 1024
    v = rng.standard_normal((2, d))
    s = np.where(rng.integers(0, 2, d) == 1, 1.0, -1.0)
    blockwise = O.rht(v, s)  # (I (x) H_128) diag(s) v / sqrt(128)
    across = blockwise.reshape(2, d // 128, 128).transpose(0, 2, 1) @ scipy.linalg.hadamard(d // 128).T
    across = across.transpose(0, 2, 1).reshape(2, d) / np.sqrt(d // 128)
    np.testing.assert_allclose(O.rht_whole(v, s), across, rtol=0, atol=1e-12)
    v128 = rng.standard_normal((2, 128))
    s128 = np.where(rng.integers(0, 2, 128) == 1, 1.0, -1.0)
    np.testing.assert_allclose(O.rht_whole(v128, s128), O.rht(v128, s128), rtol=0, atol=1e-13)


def test_rht_whole_is_orthogonal_involution():
    rng = np.random.default_rng(8)
    d = 4096
    v = rng.standard_normal((2, d))
    s = np.where(rng.integers(0, 2, d) == 1, 1.0, -1.0)
    out = O.rht_whole(v, s)
    np.testing.assert_allclose(np.linalg.norm(out, axis=1), np.linalg.norm(v, axis=1), rtol=1e-12)
    np.testing.assert_allclose(O.rht_whole(out, np.ones(d)) * s, v, rtol=0, atol=1e-11)
    with pytest.raises(AssertionError):
        O.rht_whole(np.ones((1, 384)), np.ones(384))


def test_layer_whole_brute_force():
    """The whole-vector layer against a dense evaluation with scipy's full
    Hadamard matrices and the separately written trellis walker."""
    m, n, K, cb, M = 256, 512, 2, 1, 3
    inp = synth.layer_inputs(m, n, K, M, config=93, index=0)
    W = _walk_decode(inp["codes"], K, cb, m, n)
    Hm = scipy.linalg.hadamard(m) / np.sqrt(m)
    Hn = scipy.linalg.hadamard(n) / np.sqrt(n)
    A = (Hm @ np.diag(inp["s_out"].astype(np.float64)) @ np.diag(inp["scales"].astype(np.float64)) @ W
         @ Hn @ np.diag(inp["s_in"].astype(np.float64)))
    y_bf = inp["x"].astype(np.float64) @ A.T
    y = O.layer_forward_whole(inp["codes"], K, cb, m, n, inp["s_in"], inp["s_out"], inp["scales"], inp["x"])
    np.testing.assert_allclose(y, y_bf, rtol=1e-12, atol=1e-12 * np.abs(y_bf).max())
    # differs from the blockwise layer (the rotations are not the same map)
    yb = O.layer_forward(inp["codes"], K, cb, m, n, inp["s_in"], inp["s_out"], inp["scales"], inp["x"])
    assert np.abs(y - yb).max() > 0.1 * np.abs(yb).max()
