"""The C ABI library loads, exports every entry point the header declares, and
rejects bad arguments on the host before anything reaches a GPU.

These run without a GPU: every call below fails validation, which happens
before the library touches the CUDA runtime.  The fake pointers are never
dereferenced.
"""
import ctypes

import pytest

from trellis_decode_gemv_gb300 import binding as B

A = 0x10000  # a 16-byte aligned fake device address (never dereferenced)


@pytest.fixture(scope="module")
def lib():
    return B.load_library()


def test_exports_every_declared_entry_point(lib):
    names = B.header_entry_points()
    assert {"exl3_rht_in", "exl3_rht_out", "exl3_decode_tiles", "exl3_gemv",
            "exl3_gemm_small", "exl3_workspace_bytes"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_version(lib):
    for s in range(10):
        assert len(B.exl3_status_string(s)) > 0
    assert "sm_103a" in B.exl3_version()


def _ws(m, n, M):
    a256 = lambda b: (b + 255) // 256 * 256  # noqa: E731
    counters = a256(4 * (m // 128 + 1))
    zacc = a256(4 * M * m)
    nb = 16 if M <= 16 else 32
    bimg = a256(2 * nb * n)
    bsum = a256(4 * M * (n // 128))
    return counters + zacc + bimg + bsum


def test_debug_hook_and_path_setter(lib):
    assert lib.exl3_debug_stall_tensor_wait(1) == 0
    assert lib.exl3_debug_stall_tensor_wait(0) == 0
    assert lib.exl3_set_path(3) == 5  # unknown path: rejected
    assert lib.exl3_set_path(0) == 0
    assert lib.exl3_set_prefill(3) == 5  # unknown prefill strategy: rejected
    assert lib.exl3_set_prefill(-1) == 5
    for s in (1, 2, 0):
        assert lib.exl3_set_prefill(s) == 0


def test_prefill_strategy_launch_counts(lib):
    """exl3_gemm above 32 rows: two launches fused (operand B, fused GEMM),
    three decode-once (decode to images, operand B, GEMM); AUTO takes the
    fused kernel up to 256 rows."""
    try:
        assert lib.exl3_set_prefill(1) == 0
        assert lib.exl3_gemm_launches(256, 512, 64) == 2 and lib.exl3_gemm_launches(256, 512, 1000) == 2
        assert lib.exl3_set_prefill(2) == 0
        assert lib.exl3_gemm_launches(256, 512, 64) == 3
        assert lib.exl3_set_prefill(0) == 0
        assert lib.exl3_gemm_launches(256, 512, 256) == 2 and lib.exl3_gemm_launches(256, 512, 257) == 3
    finally:
        lib.exl3_set_prefill(0)


def test_workspace_bytes(lib):
    assert B.exl3_workspace_bytes(100, 128, 1) == 0
    assert B.exl3_workspace_bytes(128, 128, 0) == 0
    assert B.exl3_workspace_bytes(128, 128, 33) == 0
    for m, n, M in [(4096, 4096, 1), (4096, 4096, 8), (1024, 28672, 1), (128256, 8192, 32)]:
        assert B.exl3_workspace_bytes(m, n, M) == _ws(m, n, M)


def _gemm(lib, m=256, n=256, K=2, cb=0, M=1, codes=A, scales=A, x=A, y=A, s_in=A, s_out=A,
          ws=A, ws_bytes=1 << 30):
    return lib.exl3_gemm_small(codes, K, cb, m, n, s_in, s_out, scales, M, x, y, ws, ws_bytes, None)


@pytest.mark.parametrize("kw,status", [
    (dict(m=100), 2), (dict(n=130), 2), (dict(m=0), 2), (dict(n=-128), 2),
    (dict(K=0), 3), (dict(K=9), 3), (dict(cb=4), 4), (dict(cb=-1), 4),
    (dict(M=0), 5), (dict(M=33), 5),
    (dict(codes=None), 1), (dict(scales=None), 1), (dict(x=None), 1), (dict(y=None), 1),
    (dict(codes=A + 4), 6), (dict(x=A + 2), 6), (dict(y=A + 8), 6), (dict(s_in=A + 2), 6),
    (dict(s_out=A + 2), 6), (dict(scales=A + 2), 6),
    (dict(ws=None), 7), (dict(ws_bytes=16), 7), (dict(ws=A + 4), 6),
])
def test_gemm_small_validation(lib, kw, status):
    assert _gemm(lib, **kw) == status


def test_gemv_validation(lib):
    assert lib.exl3_gemv(A, 2, 0, 100, 128, A, A, A, A, A, A, 1 << 20, None) == 2
    assert lib.exl3_gemv(A, 2, 0, 128, 128, A, A, A, A, A, A, 8, None) == 7


def test_decode_and_rht_validation(lib):
    assert lib.exl3_decode_tiles(A, 2, 0, 128, 96, A, None) == 2
    assert lib.exl3_decode_tiles(A, 10, 0, 128, 128, A, None) == 3
    assert lib.exl3_decode_tiles(A, 2, 4, 128, 128, A, None) == 4
    assert lib.exl3_decode_tiles(None, 2, 0, 128, 128, A, None) == 1
    assert lib.exl3_decode_tiles(A + 4, 2, 0, 128, 128, A, None) == 6
    assert lib.exl3_rht_in(A, A, A, 0, 128, None) == 5
    assert lib.exl3_rht_in(A, A, A, 1, 100, None) == 2
    assert lib.exl3_rht_in(A, None, A, 1, 128, None) == 1
    assert lib.exl3_rht_out(A, A, A + 2, 1, 128, None) == 6


def test_missing_library_raises(monkeypatch, tmp_path):
    monkeypatch.setattr(B, "_LIB", None)
    monkeypatch.setenv("EXL3_LIBRARY", str(tmp_path / "nope.so"))
    with pytest.raises(B.Exl3Error):
        B.load_library()
    monkeypatch.setattr(B, "_LIB", None)
    monkeypatch.delenv("EXL3_LIBRARY")
    assert isinstance(B.load_library(), ctypes.CDLL)


def _group(shapes, codes=A, x=A, y=A, scales=A):
    arr = (B.Exl3Layer * len(shapes))()
    for i, (m, n) in enumerate(shapes):
        arr[i].codes, arr[i].m, arr[i].n = codes, m, n
        arr[i].s_in = arr[i].s_out = A
        arr[i].scales, arr[i].x, arr[i].y = scales, x, y
    return arr


def test_group_workspace_bytes(lib):
    a256 = lambda b: (b + 255) // 256 * 256  # noqa: E731
    shapes = [(4096, 4096), (1024, 4096), (1024, 4096)]
    for M in (1, 2, 5, 32):
        mb = min(M, 8)
        nb = 16 if M <= 16 else 32
        # status word; per layer block counters and row sums; per layer the x
        # pairs or (M > 2) the decode-MMA kernel's operand images
        fixed = 256 + sum(a256(4 * (m // 128)) + a256(4 * M * m) for m, n in shapes)
        scratch = sum(a256(max(4 * mb * n, a256(2 * nb * n) + 4 * M * (n // 128) if M > 2 else 0))
                      for m, n in shapes)
        assert lib.exl3_group_workspace_bytes(_group(shapes), 3, M) == fixed + scratch
    assert lib.exl3_group_workspace_bytes(_group([(100, 128)]), 1, 1) == 0
    assert lib.exl3_group_workspace_bytes(_group(shapes), 0, 1) == 0
    assert lib.exl3_group_workspace_bytes(_group(shapes), B.MAX_GROUP + 1, 1) == 0


def test_grouped_validation(lib):
    g = _group([(256, 256), (128, 384)])
    ok = dict(K=2, cb=0, M=1, ws=A, wsb=1 << 30)

    def call(arr=g, count=2, K=2, cb=0, M=1, ws=A, wsb=1 << 30):
        return lib.exl3_gemm_grouped(arr, count, K, cb, M, ws, wsb, None)

    assert call(arr=None) == 1
    assert call(count=0) == 5 and call(count=B.MAX_GROUP + 1) == 5
    assert call(K=0) == 3 and call(cb=4) == 4 and call(M=33) == 5
    assert call(arr=_group([(256, 256), (130, 384)])) == 2
    assert call(arr=_group([(256, 256)], codes=None), count=1) == 1
    assert call(arr=_group([(256, 256)], x=A + 2), count=1) == 6
    assert call(wsb=64) == 7 and call(ws=None) == 7
    assert ok  # the remaining arguments are valid


def test_gemm_prefill_workspace_and_validation(lib):
    a256 = lambda b: (b + 255) // 256 * 256  # noqa: E731
    assert B.exl3_gemm_workspace_bytes(4096, 4096, 32) == B.exl3_workspace_bytes(4096, 4096, 32)
    m, n = 4096, 14336
    passes = (a256(4 * (m // 128 + 1)) + a256(4 * 128 * m) + a256(2 * 128 * n) + a256(4 * 128 * (n // 128)))

    def dense(M):  # counters | fp32 row sums [M][m] | operand-B tiles of 256 rows | decoded matrix | arrivals
        tiles = (M + 255) // 256
        return (a256(4 * (m // 128 + 1)) + a256(4 * M * m) + a256(2 * tiles * 256 * n)
                + a256(2 * m * n) + a256(4 * (m // 128) * tiles))
    for M in (33, 256, 257, 5000):
        assert B.exl3_gemm_workspace_bytes(m, n, M) == max(passes, dense(M))
    assert B.exl3_gemm_workspace_bytes(m, n, 0) == 0
    assert lib.exl3_gemm_launches(100, 256, 64) == 0 and lib.exl3_gemm_launches(256, 256, 0) == 0
    call = lambda **kw: lib.exl3_gemm(kw.get("codes", A), 2, kw.get("cb", 0), kw.get("m", 256), 256, A, A, A,
                                      kw.get("M", 64), A, A, kw.get("ws", A), kw.get("wsb", 1 << 30), None)  # noqa: E731
    assert call(M=0) == 5
    assert call(m=100) == 2
    assert call(cb=4) == 4
    assert call(codes=None) == 1
    assert call(wsb=16) == 7


def test_whole_vector_workspace_and_validation(lib):
    a256 = lambda b: (b + 255) // 256 * 256  # noqa: E731
    for m, n, M in ((4096, 1024, 1), (1024, 4096, 40), (128, 32768, 3)):
        inner = a256(B.exl3_gemm_workspace_bytes(m, n, M))
        want = inner + a256(2 * max(m, n)) + a256(2 * M * n) + a256(2 * M * m)
        assert B.exl3_gemm_whole_workspace_bytes(m, n, M) == want
    for m, n, M in ((384, 1024, 1), (1024, 14336, 1), (65536, 1024, 1), (64, 1024, 1), (1024, 1024, 0)):
        assert B.exl3_gemm_whole_workspace_bytes(m, n, M) == 0
    call = lambda **kw: lib.exl3_gemm_whole(kw.get("codes", A), kw.get("K", 2), 0, kw.get("m", 256),  # noqa: E731
                                            kw.get("n", 512), A, A, A, kw.get("M", 1), A, A, kw.get("ws", A),
                                            kw.get("wsb", 1 << 30), None)
    assert call(M=0) == 5
    assert call(m=384) == 2 and call(n=14336) == 2 and call(n=65536) == 2
    assert call(K=9) == 3
    assert call(codes=None) == 1
    assert call(wsb=16) == 7 and call(ws=None) == 7
    assert lib.exl3_rht_whole(A, A, A, 0, 1024, None) == 5
    assert lib.exl3_rht_whole(A, A, A, 2, 1536, None) == 2
    assert lib.exl3_rht_whole(A, A, A, 2, 65536, None) == 2
    assert lib.exl3_rht_whole(A, None, A, 2, 1024, None) == 1
    assert lib.exl3_rht_whole(A + 8, A, A, 2, 1024, None) == 6


def test_whole_grouped_workspace_and_validation(lib):
    a256 = lambda b: (b + 255) // 256 * 256  # noqa: E731
    shapes = [(4096, 4096), (1024, 4096), (1024, 4096)]
    for M in (1, 3, 32):
        inner = a256(lib.exl3_group_workspace_bytes(_group(shapes), 3, M))
        want = inner + a256(2 * 4096) + sum(a256(2 * M * n) + a256(2 * M * m) for m, n in shapes)
        assert lib.exl3_gemm_whole_grouped_workspace_bytes(_group(shapes), 3, M) == want
        assert B.exl3_gemm_whole_grouped_workspace_bytes(shapes, M) == want
    assert lib.exl3_gemm_whole_grouped_workspace_bytes(_group([(384, 1024)]), 1, 1) == 0
    assert lib.exl3_gemm_whole_grouped_workspace_bytes(_group(shapes), 3, 33) == 0
    assert lib.exl3_gemm_whole_grouped_workspace_bytes(_group(shapes), 0, 1) == 0
    assert lib.exl3_gemm_whole_grouped_workspace_bytes(_group(shapes), B.MAX_GROUP + 1, 1) == 0
    assert lib.exl3_gemm_whole_grouped_workspace_bytes(None, 1, 1) == 0
    g = _group([(256, 512), (1024, 512)])

    def call(arr=g, count=2, K=2, cb=0, M=1, ws=A, wsb=1 << 30):
        return lib.exl3_gemm_whole_grouped(arr, count, K, cb, M, ws, wsb, None)

    assert call(arr=None) == 1
    assert call(count=0) == 5 and call(count=B.MAX_GROUP + 1) == 5  # as exl3_gemm_grouped
    assert call(M=0) == 5 and call(M=33) == 5
    assert call(arr=_group([(256, 512), (384, 512)])) == 2
    assert call(K=9) == 3 and call(cb=4) == 4
    assert call(arr=_group([(256, 512)], scales=None), count=1) == 1
    assert call(arr=_group([(256, 512)], y=A + 2), count=1) == 6
    assert call(wsb=64) == 7 and call(ws=None) == 7 and call(ws=A + 8) == 6


def test_encoder_workspace_and_validation(lib):
    for K in range(1, 9):
        assert B.exl3_encode_workspace_bytes(K, 3) == 3 * 256 * (1 << (16 - K))
    assert B.exl3_encode_workspace_bytes(0, 1) == 0 and B.exl3_encode_workspace_bytes(9, 1) == 0
    assert B.exl3_encode_workspace_bytes(2, 0) == 0
    slot = B.exl3_encode_workspace_bytes(2, 1)
    call = lambda **kw: lib.exl3_encode_tiles(kw.get("t", A), kw.get("tiles", 4), kw.get("K", 2),  # noqa: E731
                                              kw.get("cb", 0), kw.get("w", A), kw.get("c", A), kw.get("ws", A),
                                              kw.get("wsb", slot), None)
    assert call(tiles=0) == 2
    assert call(K=0) == 3 and call(K=9) == 3
    assert call(cb=4) == 4
    assert call(t=None) == 1 and call(w=None) == 1 and call(c=None) == 1
    assert call(t=A + 4) == 6 and call(w=A + 8) == 6
    assert call(wsb=slot - 1) == 7 and call(ws=None) == 7


def test_int8_path_workspace_and_validation(lib):
    a256 = lambda b: (b + 255) // 256 * 256  # noqa: E731
    m, n, M = 1024, 4096, 5
    want = (a256(4 * (m // 128 + 1)) + a256(4 * M * m) + a256(4 * M * n) + a256(4 * M * (n // 16))
            + a256(4 * M * (n // 128)))
    assert B.exl3_gemm_i8_workspace_bytes(m, n, M) == want
    assert B.exl3_gemm_i8_workspace_bytes(m, n, 33) == 0 and B.exl3_gemm_i8_workspace_bytes(100, n, 1) == 0
    call = lambda **kw: lib.exl3_gemm_i8(kw.get("codes", A), kw.get("K", 2), kw.get("cb", 1), kw.get("m", 256),  # noqa: E731
                                         256, A, A, kw.get("M", 1), A, kw.get("qs", A), A, kw.get("ws", A),
                                         kw.get("wsb", 1 << 30), None)
    assert call(M=0) == 5 and call(M=33) == 5
    assert call(m=100) == 2
    assert call(cb=0) == 4 and call(cb=2) == 4 and call(cb=4) == 4
    assert call(K=9) == 3
    assert call(codes=None) == 1 and call(qs=None) == 1
    assert call(wsb=16) == 7
    f = lambda **kw: lib.exl3_gemm_int8act(A, 2, kw.get("cb", 3), 256, 256, A, A, A, kw.get("M", 1), A,  # noqa: E731
                                           kw.get("y", A), A, 1 << 30, None)
    assert f(cb=0) == 4 and f(M=0) == 5 and f(y=None) == 1
    assert lib.exl3_quantize_act(A, 0, 128, A, A, None) == 5
    assert lib.exl3_quantize_act(A, 1, 100, A, A, None) == 2
    assert lib.exl3_quantize_act(A, 1, 128, A, None, None) == 1
    assert lib.exl3_quantize_act(A + 2, 1, 128, A, A, None) == 6


def test_int8_group_workspace_and_validation(lib):
    a256 = lambda b: (b + 255) // 256 * 256  # noqa: E731
    shapes, M = [(1024, 4096), (256, 512)], 3
    want = 256 + sum(a256(4 * M * m) + a256(4 * M * n) + a256(4 * M * (n // 16)) + a256(4 * M * (n // 128))
                     for m, n in shapes)
    assert B.exl3_group_i8_workspace_bytes(shapes, M) == want
    assert B.exl3_group_i8_workspace_bytes([(100, 256)], 1) == 0
    assert B.exl3_group_i8_workspace_bytes(shapes, 33) == 0
    assert B.exl3_group_i8_workspace_bytes(shapes * 33, 1) == 0  # more than EXL3_MAX_GROUP layers
    assert lib.exl3_gemm_int8act_grouped(None, 1, 2, 1, 1, A, 1 << 30, None) == 1


def test_device_status_rejects_null(lib):
    assert lib.exl3_device_status(None, None) == 1


def test_multi_workspace_and_validation(lib):
    shapes = [(256, 384), (1024, 4096), (128, 128)]
    for M in (1, 2, 7):
        assert B.exl3_multi_workspace_bytes(shapes, M) == B.exl3_group_workspace_bytes(shapes, M)
    arr = (B.Exl3LayerKC * 2)()
    for i, (m, n) in enumerate([(256, 256), (128, 384)]):
        arr[i].layer.codes, arr[i].layer.m, arr[i].layer.n = A, m, n
        arr[i].layer.scales, arr[i].layer.x, arr[i].layer.y = A, A, A
        arr[i].K, arr[i].codebook = 2 + i, i

    def call(count=2, M=1, ws=A, wsb=1 << 30):
        return lib.exl3_gemm_multi(arr, count, M, ws, wsb, None)

    assert lib.exl3_gemm_multi(None, 1, 1, A, 1 << 30, None) == 1
    assert call(count=0) == 5 and call(count=B.MAX_GROUP + 1) == 5 and call(M=33) == 5
    arr[1].K = 9
    assert call() == 3
    arr[1].K, arr[1].codebook = 3, 4
    assert call() == 4
    arr[1].codebook = 1
    arr[1].layer.m = 130
    assert call() == 2
    arr[1].layer.m = 128
    arr[1].layer.x = A + 2
    assert call() == 6
    arr[1].layer.x = A
    assert call(wsb=64) == 7 and call(ws=None) == 7


def test_int8_multi_workspace_and_validation(lib):
    shapes = [(256, 384), (1024, 4096), (128, 128)]
    for M in (1, 2, 7):
        assert B.exl3_multi_i8_workspace_bytes(shapes, M) == B.exl3_group_i8_workspace_bytes(shapes, M)
    arr = (B.Exl3LayerKC * 2)()
    for i, (m, n) in enumerate([(256, 256), (128, 384)]):
        arr[i].layer.codes, arr[i].layer.m, arr[i].layer.n = A, m, n
        arr[i].layer.scales, arr[i].layer.x, arr[i].layer.y = A, A, A
        arr[i].K, arr[i].codebook = 2 + i, 1 + 2 * i  # 1MAD, mul1

    def call(count=2, M=1, ws=A, wsb=1 << 30):
        return lib.exl3_gemm_int8act_multi(arr, count, M, ws, wsb, None)

    assert lib.exl3_gemm_int8act_multi(None, 1, 1, A, 1 << 30, None) == 1
    assert call(count=0) == 5 and call(count=B.MAX_GROUP + 1) == 5 and call(M=33) == 5
    arr[1].K = 9
    assert call() == 3
    arr[1].K = 3
    for bad in (0, 2, 4):  # 3INST and MCG have no byte sum; 4 is no code
        arr[1].codebook = bad
        assert call() == 4
    arr[1].codebook = 3
    arr[1].layer.m = 130
    assert call() == 2
    arr[1].layer.m = 128
    arr[1].layer.x = A + 2
    assert call() == 6
    arr[1].layer.x = A
    assert call(wsb=64) == 7 and call(ws=None) == 7
