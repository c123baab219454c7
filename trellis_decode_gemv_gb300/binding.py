"""ctypes binding of libexl3 (include/exl3.h).

Each function has the name of the C entry point it calls and only checks and
marshals torch tensors (device, dtype, contiguity) and passes raw device
pointers plus the current CUDA stream.  Every step of the computation runs in
the library's CUDA kernels; there is no other implementation to fall back on,
and a missing library raises.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

CB_3INST = 0
CB_1MAD = 1
CB_MCG = 2
CB_MUL1 = 3
MAX_BATCH = 32

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None

_STATUS_NAMES = {
    0: "EXL3_OK", 1: "EXL3_ERR_NULL", 2: "EXL3_ERR_SHAPE", 3: "EXL3_ERR_K",
    4: "EXL3_ERR_CODEBOOK", 5: "EXL3_ERR_BATCH", 6: "EXL3_ERR_ALIGN",
    7: "EXL3_ERR_WORKSPACE", 8: "EXL3_ERR_CUDA", 9: "EXL3_ERR_DEVICE_CHECK",
    10: "EXL3_ERR_SCRATCH",
}


class Exl3Error(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def library_path() -> str:
    return os.environ.get("EXL3_LIBRARY", os.path.join(_HERE, "libexl3.so"))


_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
MAX_GROUP = 64


class Exl3Layer(ctypes.Structure):
    """exl3_layer of the header: one layer of a grouped call."""
    _fields_ = [("codes", _P), ("m", _I), ("n", _I), ("s_in", _P), ("s_out", _P),
                ("scales", _P), ("x", _P), ("y", _P)]


class Exl3LayerKC(ctypes.Structure):
    """exl3_layer_kc of the header: a layer with its own K and code."""
    _fields_ = [("layer", Exl3Layer), ("K", _I), ("codebook", _I)]


_SIGNATURES = {
    "exl3_rht_in": ([_P, _P, _P, _I, _I, _P], _I),
    "exl3_rht_out": ([_P, _P, _P, _I, _I, _P], _I),
    "exl3_decode_tiles": ([_P, _I, _I, _I, _I, _P, _P], _I),
    "exl3_workspace_bytes": ([_I, _I, _I], _SZ),
    "exl3_gemv": ([_P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _SZ, _P], _I),
    "exl3_gemm_small": ([_P, _I, _I, _I, _I, _P, _P, _P, _I, _P, _P, _P, _SZ, _P], _I),
    "exl3_gemv_noalloc": ([_P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P], _I),
    "exl3_group_workspace_bytes": ([ctypes.POINTER(Exl3Layer), _I, _I], _SZ),
    "exl3_gemm_grouped": ([ctypes.POINTER(Exl3Layer), _I, _I, _I, _I, _P, _SZ, _P], _I),
    "exl3_multi_workspace_bytes": ([ctypes.POINTER(Exl3LayerKC), _I, _I], _SZ),
    "exl3_gemm_multi": ([ctypes.POINTER(Exl3LayerKC), _I, _I, _P, _SZ, _P], _I),
    "exl3_gemm_workspace_bytes": ([_I, _I, _I], _SZ),
    "exl3_gemm_launches": ([_I, _I, _I], _I),
    "exl3_probe_int": ([_I, _P, _I, _I, _P], _I),
    "exl3_rht_whole": ([_P, _P, _P, _I, _I, _P], _I),
    "exl3_encode_workspace_bytes": ([_I, _I], _SZ),
    "exl3_quantize_act": ([_P, _I, _I, _P, _P, _P], _I),
    "exl3_gemm_i8_workspace_bytes": ([_I, _I, _I], _SZ),
    "exl3_gemm_i8": ([_P, _I, _I, _I, _I, _P, _P, _I, _P, _P, _P, _P, _SZ, _P], _I),
    "exl3_gemm_int8act": ([_P, _I, _I, _I, _I, _P, _P, _P, _I, _P, _P, _P, _SZ, _P], _I),
    "exl3_group_i8_workspace_bytes": ([ctypes.POINTER(Exl3Layer), _I, _I], _SZ),
    "exl3_gemm_int8act_grouped": ([ctypes.POINTER(Exl3Layer), _I, _I, _I, _I, _P, _SZ, _P], _I),
    "exl3_multi_i8_workspace_bytes": ([ctypes.POINTER(Exl3LayerKC), _I, _I], _SZ),
    "exl3_gemm_int8act_multi": ([ctypes.POINTER(Exl3LayerKC), _I, _I, _P, _SZ, _P], _I),
    "exl3_encode_tiles": ([_P, _I, _I, _I, _P, _P, _P, _SZ, _P], _I),
    "exl3_gemm_whole_workspace_bytes": ([_I, _I, _I], _SZ),
    "exl3_gemm_whole": ([_P, _I, _I, _I, _I, _P, _P, _P, _I, _P, _P, _P, _SZ, _P], _I),
    "exl3_gemm_whole_grouped_workspace_bytes": ([ctypes.POINTER(Exl3Layer), _I, _I], _SZ),
    "exl3_gemm_whole_grouped": ([ctypes.POINTER(Exl3Layer), _I, _I, _I, _I, _P, _SZ, _P], _I),
    "exl3_gemm": ([_P, _I, _I, _I, _I, _P, _P, _P, _I, _P, _P, _P, _SZ, _P], _I),
    "exl3_set_path": ([_I], _I),
    "exl3_set_prefill": ([_I], _I),
    "exl3_debug_stall_tensor_wait": ([_I], _I),
    "exl3_device_status": ([_P, _P], _I),
    "exl3_status_string": ([_I], ctypes.c_char_p),
    "exl3_version": ([], ctypes.c_char_p),
}


def header_entry_points() -> list[str]:
    """Names of the functions declared in include/exl3.h."""
    hdr = os.path.join(os.path.dirname(_HERE), "include", "exl3.h")
    text = open(hdr).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(exl3_\w+)\s*\(", text, re.M)))


def load_library():
    """Load libexl3.so (raises if it has not been built)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = library_path()
    if not os.path.exists(path):
        raise Exl3Error(-1, f"{path} is missing: build it with "
                            "`python -m trellis_decode_gemv_gb300.build`")
    lib = ctypes.CDLL(path)
    for name, (args, res) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _LIB = lib
    return lib


def _check(status: int):
    if status != 0:
        msg = load_library().exl3_status_string(status).decode()
        raise Exl3Error(status, msg)


def _ptr(t: torch.Tensor | None, name: str, dtypes, device=None) -> int | None:
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


_HALF = (torch.float16,)
_WORDS = (torch.int32, getattr(torch, "uint32", torch.int32))


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def exl3_status_string(status: int) -> str:
    return load_library().exl3_status_string(status).decode()


def exl3_version() -> str:
    return load_library().exl3_version().decode()


PATH_AUTO, PATH_SHUFFLE, PATH_TENSOR = 0, 1, 2


def exl3_set_path(path: int) -> None:
    """Select the kernel family of exl3_gemv / exl3_gemm_small (process-wide)."""
    _check(load_library().exl3_set_path(path))


PREFILL_AUTO, PREFILL_FUSED, PREFILL_DECODE_ONCE = 0, 1, 2


def exl3_set_prefill(strategy: int) -> None:
    """Select the prefill strategy of exl3_gemm above 32 rows (process-wide)."""
    _check(load_library().exl3_set_prefill(strategy))


def exl3_debug_stall_tensor_wait(on: bool) -> None:
    """Failure-detection test hook of the tensor-core kernel (see the header)."""
    _check(load_library().exl3_debug_stall_tensor_wait(1 if on else 0))


def exl3_device_status(workspace: torch.Tensor, offset: int) -> int:
    """The library's check of the status word at byte `offset` of a workspace:
    0 (EXL3_OK) or 9 (EXL3_ERR_DEVICE_CHECK).  Waits for the current stream."""
    lib = load_library()
    dev = workspace.device
    st = lib.exl3_device_status(_ptr(workspace, "workspace", (torch.uint8,), dev) + offset, _stream(dev))
    if st not in (0, 9):
        _check(st)
    return st


def workspace_status(workspace: torch.Tensor, m: int) -> int:
    """The workspace's device-side status word (non-zero after a timed-out
    device wait).  Synchronizes with the current stream."""
    off = 4 * (m // 128)
    return int(workspace[off:off + 4].view(torch.int32).item())


def exl3_workspace_bytes(m: int, n: int, M: int = 1) -> int:
    return int(load_library().exl3_workspace_bytes(m, n, M))


def alloc_workspace(m: int, n: int, M: int, device) -> torch.Tensor:
    """A zero-filled workspace of exl3_workspace_bytes(m, n, M) bytes."""
    nbytes = exl3_workspace_bytes(m, n, M)
    if nbytes == 0:
        raise Exl3Error(2, "invalid shape or batch for a workspace")
    return torch.zeros(nbytes, dtype=torch.uint8, device=device)


def exl3_rht_in(x: torch.Tensor, s_in: torch.Tensor, out: torch.Tensor | None = None):
    lib = load_library()
    x2 = x if x.dim() == 2 else x.view(1, -1)
    M, n = x2.shape
    if out is None:
        out = torch.empty_like(x2)
    _check(lib.exl3_rht_in(_ptr(x2, "x", _HALF), _ptr(s_in, "s_in", _HALF, x.device),
                           _ptr(out, "x_rot", _HALF, x.device), M, n, _stream(x.device)))
    return out.view_as(x)


def exl3_rht_out(z: torch.Tensor, s_out: torch.Tensor, out: torch.Tensor | None = None):
    lib = load_library()
    z2 = z if z.dim() == 2 else z.view(1, -1)
    M, m = z2.shape
    if out is None:
        out = torch.empty_like(z2)
    _check(lib.exl3_rht_out(_ptr(z2, "z", _HALF), _ptr(s_out, "s_out", _HALF, z.device),
                            _ptr(out, "y", _HALF, z.device), M, m, _stream(z.device)))
    return out.view_as(z)


def exl3_decode_tiles(codes: torch.Tensor, K: int, codebook: int, m: int, n: int,
                      out: torch.Tensor | None = None) -> torch.Tensor:
    lib = load_library()
    if out is None:
        out = torch.empty((m, n), dtype=torch.float16, device=codes.device)
    _check(lib.exl3_decode_tiles(_ptr(codes, "codes", _WORDS), K, codebook, m, n,
                                 _ptr(out, "w_out", _HALF, codes.device), _stream(codes.device)))
    return out


def exl3_gemm_small(codes, K, codebook, m, n, s_in, s_out, scales, x, y=None, workspace=None):
    """y[M, m] = Hb(s_out (.) (scales (.) (W-hat Hb(s_in (.) x[M, n])))).  x is [M, n]."""
    lib = load_library()
    dev = codes.device
    x2 = x if x.dim() == 2 else x.view(1, -1)
    M = x2.shape[0]
    if y is None:
        y = torch.empty((M, m), dtype=torch.float16, device=dev)
    if workspace is None:
        workspace = alloc_workspace(m, n, M, dev)
    _check(lib.exl3_gemm_small(
        _ptr(codes, "codes", _WORDS), K, codebook, m, n,
        _ptr(s_in, "s_in", _HALF, dev), _ptr(s_out, "s_out", _HALF, dev),
        _ptr(scales, "scales", _HALF, dev), M, _ptr(x2, "x", _HALF, dev),
        _ptr(y, "y", _HALF, dev), _ptr(workspace, "workspace", (torch.uint8,), dev),
        workspace.numel(), _stream(dev)))
    return y if x.dim() == 2 else y.view(-1)


def exl3_gemv(codes, K, codebook, m, n, s_in, s_out, scales, x, y=None, workspace=None):
    """Batch-1 layer: x [n] (or [1, n]) -> y [m]."""
    lib = load_library()
    dev = codes.device
    if y is None:
        y = torch.empty(m, dtype=torch.float16, device=dev)
    if workspace is None:
        workspace = alloc_workspace(m, n, 1, dev)
    _check(lib.exl3_gemv(
        _ptr(codes, "codes", _WORDS), K, codebook, m, n,
        _ptr(s_in, "s_in", _HALF, dev), _ptr(s_out, "s_out", _HALF, dev),
        _ptr(scales, "scales", _HALF, dev), _ptr(x, "x", _HALF, dev), _ptr(y, "y", _HALF, dev),
        _ptr(workspace, "workspace", (torch.uint8,), dev), workspace.numel(), _stream(dev)))
    return y


def exl3_gemv_noalloc(codes, K, codebook, m, n, s_in, s_out, scales, x, y=None):
    """exl3_gemv for callers that cannot allocate device memory: the library
    uses its own fixed device scratch array instead of a workspace.  Calls
    that may overlap on the GPU must be serialized by the caller."""
    lib = load_library()
    dev = codes.device
    if y is None:
        y = torch.empty(m, dtype=torch.float16, device=dev)
    # the scratch array's address is per device: make the tensors' device current
    with torch.cuda.device(dev):
        _check(lib.exl3_gemv_noalloc(
            _ptr(codes, "codes", _WORDS), K, codebook, m, n,
            _ptr(s_in, "s_in", _HALF, dev), _ptr(s_out, "s_out", _HALF, dev),
            _ptr(scales, "scales", _HALF, dev), _ptr(x, "x", _HALF, dev), _ptr(y, "y", _HALF, dev),
            _stream(dev)))
    return y


def _layer_array(layers, dev, M):
    """ctypes array of exl3_layer from dicts with codes, m, n, s_in, s_out,
    scales, x ([M, n]) and y ([M, m])."""
    arr = (Exl3Layer * len(layers))()
    for i, L in enumerate(layers):
        arr[i].codes = _ptr(L["codes"], "codes", _WORDS, dev)
        arr[i].m = L["m"]
        arr[i].n = L["n"]
        arr[i].s_in = _ptr(L.get("s_in"), "s_in", _HALF, dev)
        arr[i].s_out = _ptr(L.get("s_out"), "s_out", _HALF, dev)
        arr[i].scales = _ptr(L["scales"], "scales", _HALF, dev)
        arr[i].x = _ptr(L["x"], "x", _HALF, dev)
        arr[i].y = _ptr(L["y"], "y", _HALF, dev)
    return arr


def _kc_array(layers, dev, M):
    plain = _layer_array(layers, dev, M)
    arr = (Exl3LayerKC * len(layers))()
    for i, L in enumerate(layers):
        arr[i].layer = plain[i]
        arr[i].K = int(L["K"])
        arr[i].codebook = int(L["cb"])
    return arr


def exl3_gemm_multi(layers, workspace=None):
    """Independent layers of their own K and code at one batch: each dict as
    for exl3_gemm_grouped plus K and cb.  Same results as one exl3_gemm_small
    per layer; at batch 1 and 2 the layers of the multi-code kernel's (K, code)
    pairs share one kernel chain."""
    lib = load_library()
    dev = layers[0]["codes"].device
    M = layers[0]["x"].shape[0] if layers[0]["x"].dim() == 2 else 1
    arr = _kc_array(layers, dev, M)
    if workspace is None:
        workspace = alloc_group_workspace([(L["m"], L["n"]) for L in layers], M, dev)
    _check(lib.exl3_gemm_multi(arr, len(layers), M, _ptr(workspace, "workspace", (torch.uint8,), dev),
                               workspace.numel(), _stream(dev)))
    return [L["y"] for L in layers]


def exl3_multi_workspace_bytes(shapes, M: int = 1) -> int:
    """Workspace bytes of a multi-code grouped call over layers of (m, n)."""
    arr = (Exl3LayerKC * len(shapes))()
    for i, (m, n) in enumerate(shapes):
        arr[i].layer.m, arr[i].layer.n = m, n
        arr[i].K, arr[i].codebook = 2, 0
    return int(load_library().exl3_multi_workspace_bytes(arr, len(shapes), M))


def exl3_group_workspace_bytes(shapes, M: int = 1) -> int:
    """Workspace bytes of a grouped call over layers of the given (m, n)."""
    arr = (Exl3Layer * len(shapes))()
    for i, (m, n) in enumerate(shapes):
        arr[i].m, arr[i].n = m, n
    return int(load_library().exl3_group_workspace_bytes(arr, len(shapes), M))


def alloc_group_workspace(shapes, M: int, device) -> torch.Tensor:
    nbytes = exl3_group_workspace_bytes(shapes, M)
    if nbytes == 0:
        raise Exl3Error(2, "invalid group for a workspace")
    return torch.zeros(nbytes, dtype=torch.uint8, device=device)


def exl3_gemm_grouped(layers, K, codebook, workspace=None):
    """Independent layers sharing K, the codebook and the batch: each dict has
    codes, m, n, s_in, s_out (or None), scales, x [M, n] and y [M, m] (written).
    Same results as one exl3_gemm_small per layer, in fewer launches."""
    lib = load_library()
    dev = layers[0]["codes"].device
    M = layers[0]["x"].shape[0] if layers[0]["x"].dim() == 2 else 1
    arr = _layer_array(layers, dev, M)
    if workspace is None:
        workspace = alloc_group_workspace([(L["m"], L["n"]) for L in layers], M, dev)
    _check(lib.exl3_gemm_grouped(arr, len(layers), K, codebook, M,
                                 _ptr(workspace, "workspace", (torch.uint8,), dev), workspace.numel(),
                                 _stream(dev)))
    return [L["y"] for L in layers]


def exl3_group_i8_workspace_bytes(shapes, M: int = 1) -> int:
    """Workspace bytes of a grouped int8-activation call over layers of (m, n)."""
    arr = (Exl3Layer * len(shapes))()
    for i, (m, n) in enumerate(shapes):
        arr[i].m, arr[i].n = m, n
    return int(load_library().exl3_group_i8_workspace_bytes(arr, len(shapes), M))


def exl3_multi_i8_workspace_bytes(shapes, M: int = 1) -> int:
    """Workspace bytes of a multi-code int8-activation call over layers of (m, n)."""
    arr = (Exl3LayerKC * len(shapes))()
    for i, (m, n) in enumerate(shapes):
        arr[i].layer.m, arr[i].layer.n = m, n
        arr[i].K, arr[i].codebook = 2, 1
    return int(load_library().exl3_multi_i8_workspace_bytes(arr, len(shapes), M))


def _i8_group_workspace(shapes, M, dev):
    nbytes = exl3_group_i8_workspace_bytes(shapes, M)
    if nbytes == 0:
        raise Exl3Error(2, "invalid group for a workspace")
    return torch.zeros(nbytes, dtype=torch.uint8, device=dev)


def exl3_gemm_int8act_multi(layers, workspace=None):
    """Independent layers on int8 activations, each of its own K and byte-sum
    code (dicts as for exl3_gemm_multi, cb 1MAD or mul1); same results as one
    exl3_gemm_int8act per layer, in one kernel chain."""
    lib = load_library()
    dev = layers[0]["codes"].device
    M = layers[0]["x"].shape[0] if layers[0]["x"].dim() == 2 else 1
    arr = _kc_array(layers, dev, M)
    if workspace is None:
        workspace = _i8_group_workspace([(L["m"], L["n"]) for L in layers], M, dev)
    _check(lib.exl3_gemm_int8act_multi(arr, len(layers), M, _ptr(workspace, "workspace", (torch.uint8,), dev),
                                       workspace.numel(), _stream(dev)))
    return [L["y"] for L in layers]


def exl3_gemm_int8act_grouped(layers, K, codebook, workspace=None):
    """Independent layers on int8 activations (1MAD or mul1), as dicts like
    exl3_gemm_grouped's; same results as one exl3_gemm_int8act per layer."""
    lib = load_library()
    dev = layers[0]["codes"].device
    M = layers[0]["x"].shape[0] if layers[0]["x"].dim() == 2 else 1
    arr = _layer_array(layers, dev, M)
    if workspace is None:
        workspace = _i8_group_workspace([(L["m"], L["n"]) for L in layers], M, dev)
    _check(lib.exl3_gemm_int8act_grouped(arr, len(layers), K, codebook, M,
                                         _ptr(workspace, "workspace", (torch.uint8,), dev), workspace.numel(),
                                         _stream(dev)))
    return [L["y"] for L in layers]


class Exl3Linear:
    """One quantized linear layer, marshalled once.

    Holds the layer's device tensors (codes, signs, scales) and a workspace,
    checked when the object is built; a call then only checks and passes x and
    y.  Same computation as exl3_gemm (any batch up to max_batch):
        y[M, m] = Hb(s_out (.) (scales (.) (W-hat Hb(s_in (.) x[M, n])))).
    """

    def __init__(self, codes, K, codebook, m, n, s_in, s_out, scales, max_batch=1):
        lib = load_library()
        self.device = codes.device
        self.K, self.codebook, self.m, self.n = K, codebook, m, n
        self._keep = (codes, s_in, s_out, scales)
        dev = self.device
        self._args = (_ptr(codes, "codes", _WORDS, dev), K, codebook, m, n,
                      _ptr(s_in, "s_in", _HALF, dev), _ptr(s_out, "s_out", _HALF, dev),
                      _ptr(scales, "scales", _HALF, dev))
        nbytes = lib.exl3_gemm_workspace_bytes(m, n, max_batch)
        if nbytes == 0:
            raise Exl3Error(2, "invalid shape or batch for a workspace")
        self.workspace = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
        self._ws = (self.workspace.data_ptr(), self.workspace.numel())
        self._max_batch = max_batch
        self._fn = lib.exl3_gemm  # exl3_gemm_small up to 32 rows, 128-row passes above

    def __call__(self, x, y=None):
        x2 = x if x.dim() == 2 else x.view(1, -1)
        M = x2.shape[0]
        if M > self._max_batch or x2.shape[1] != self.n:
            raise ValueError(f"x of shape {tuple(x2.shape)} for a layer of n={self.n}, "
                             f"batch up to {self._max_batch}")
        if y is None:
            y = torch.empty((M, self.m), dtype=torch.float16, device=self.device)
        _check(self._fn(*self._args, M, _ptr(x2, "x", _HALF, self.device), _ptr(y, "y", _HALF, self.device),
                        *self._ws, torch.cuda.current_stream(self.device).cuda_stream))
        return y if x.dim() == 2 else y.view(-1)


class Exl3LinearGroup:
    """Independent layers (sharing K, the code and the batch) marshalled once
    for exl3_gemm_grouped: each layer dict has codes, m, n, s_in, s_out,
    scales, x [M, n] and y [M, m] -- x and y stay bound to those tensors, whose
    contents change between calls (decoders write the step's input into x)."""

    def __init__(self, layers, K, codebook):
        lib = load_library()
        self.device = layers[0]["codes"].device
        self.K, self.codebook = K, codebook
        self.M = layers[0]["x"].shape[0] if layers[0]["x"].dim() == 2 else 1
        self._keep = [dict(L) for L in layers]
        self._arr = _layer_array(layers, self.device, self.M)
        self.workspace = alloc_group_workspace([(L["m"], L["n"]) for L in layers], self.M, self.device)
        self._ws = (self.workspace.data_ptr(), self.workspace.numel())
        self._count = len(layers)
        self._fn = lib.exl3_gemm_grouped

    def __call__(self):
        _check(self._fn(self._arr, self._count, self.K, self.codebook, self.M, *self._ws,
                        torch.cuda.current_stream(self.device).cuda_stream))
        return [L["y"] for L in self._keep]


class Exl3LinearMulti:
    """Independent layers of their own K and code (one batch) marshalled once
    for exl3_gemm_multi (or, with int8=True, exl3_gemm_int8act_multi): each
    layer dict as for Exl3LinearGroup plus K and cb; x and y stay bound to
    those tensors."""

    def __init__(self, layers, int8=False):
        lib = load_library()
        self.device = layers[0]["codes"].device
        self.M = layers[0]["x"].shape[0] if layers[0]["x"].dim() == 2 else 1
        self._keep = [dict(L) for L in layers]
        self._arr = _kc_array(layers, self.device, self.M)
        shapes = [(L["m"], L["n"]) for L in layers]
        self.workspace = (_i8_group_workspace(shapes, self.M, self.device) if int8
                          else alloc_group_workspace(shapes, self.M, self.device))
        self._ws = (self.workspace.data_ptr(), self.workspace.numel())
        self._count = len(layers)
        self._fn = lib.exl3_gemm_int8act_multi if int8 else lib.exl3_gemm_multi

    def __call__(self):
        _check(self._fn(self._arr, self._count, self.M, *self._ws,
                        torch.cuda.current_stream(self.device).cuda_stream))
        return [L["y"] for L in self._keep]


def exl3_gemm_workspace_bytes(m: int, n: int, M: int) -> int:
    return int(load_library().exl3_gemm_workspace_bytes(m, n, M))


def exl3_rht_whole(x: torch.Tensor, signs: torch.Tensor, out: torch.Tensor | None = None):
    """QTIP's whole-vector transform of each row: binary16(H_d (signs (.) x) / sqrt(d))."""
    lib = load_library()
    x2 = x if x.dim() == 2 else x.view(1, -1)
    rows, d = x2.shape
    if out is None:
        out = torch.empty_like(x2)
    _check(lib.exl3_rht_whole(_ptr(x2, "x", _HALF), _ptr(signs, "signs", _HALF, x.device),
                              _ptr(out, "out", _HALF, x.device), rows, d, _stream(x.device)))
    return out if x.dim() == 2 else out.view(-1)


def exl3_gemm_whole_workspace_bytes(m: int, n: int, M: int) -> int:
    return int(load_library().exl3_gemm_whole_workspace_bytes(m, n, M))


def exl3_gemm_whole(codes, K, codebook, m, n, s_in, s_out, scales, x, y=None, workspace=None):
    """The layer with whole-vector rotations (power-of-two m, n): x [M, n] -> y [M, m]."""
    lib = load_library()
    dev = codes.device
    x2 = x if x.dim() == 2 else x.view(1, -1)
    M = x2.shape[0]
    if y is None:
        y = torch.empty((M, m), dtype=torch.float16, device=dev)
    if workspace is None:
        nbytes = exl3_gemm_whole_workspace_bytes(m, n, M)
        if nbytes == 0:
            raise Exl3Error(2, "invalid shape or batch for a whole-vector workspace")
        workspace = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
    _check(lib.exl3_gemm_whole(
        _ptr(codes, "codes", _WORDS), K, codebook, m, n,
        _ptr(s_in, "s_in", _HALF, dev), _ptr(s_out, "s_out", _HALF, dev),
        _ptr(scales, "scales", _HALF, dev), M, _ptr(x2, "x", _HALF, dev),
        _ptr(y, "y", _HALF, dev), _ptr(workspace, "workspace", (torch.uint8,), dev),
        workspace.numel(), _stream(dev)))
    return y if x.dim() == 2 else y.view(-1)


def exl3_gemm_whole_grouped_workspace_bytes(shapes, M: int = 1) -> int:
    """Workspace bytes of a grouped whole-vector call over layers of (m, n)."""
    arr = (Exl3Layer * len(shapes))()
    for i, (m, n) in enumerate(shapes):
        arr[i].m, arr[i].n = m, n
    return int(load_library().exl3_gemm_whole_grouped_workspace_bytes(arr, len(shapes), M))


def exl3_gemm_whole_grouped(layers, K, codebook, workspace=None):
    """Independent whole-vector layers sharing K, the codebook and the batch
    (dicts as for exl3_gemm_grouped, power-of-two m and n): same results as
    one exl3_gemm_whole per layer, in one chain of launches."""
    lib = load_library()
    dev = layers[0]["codes"].device
    M = layers[0]["x"].shape[0] if layers[0]["x"].dim() == 2 else 1
    arr = _layer_array(layers, dev, M)
    if workspace is None:
        nbytes = exl3_gemm_whole_grouped_workspace_bytes([(L["m"], L["n"]) for L in layers], M)
        if nbytes == 0:
            raise Exl3Error(2, "invalid group for a whole-vector workspace")
        workspace = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
    _check(lib.exl3_gemm_whole_grouped(arr, len(layers), K, codebook, M,
                                       _ptr(workspace, "workspace", (torch.uint8,), dev), workspace.numel(),
                                       _stream(dev)))
    return [L["y"] for L in layers]


def exl3_encode_workspace_bytes(K: int, ctas: int) -> int:
    return int(load_library().exl3_encode_workspace_bytes(K, ctas))


def exl3_encode_tiles(target: torch.Tensor, K: int, codebook: int, words=None, cost=None, workspace=None):
    """Tail-biting Viterbi encoding of target [tiles, 256] (float32, code units):
    returns (words [tiles, 8K] int32 storage of uint32, cost [tiles] float32)."""
    lib = load_library()
    dev = target.device
    tiles = target.shape[0]
    if words is None:
        words = torch.empty((tiles, 8 * K), dtype=torch.int32, device=dev)
    if cost is None:
        cost = torch.empty(tiles, dtype=torch.float32, device=dev)
    if workspace is None:
        ctas = min(tiles, torch.cuda.get_device_properties(dev).multi_processor_count)
        workspace = torch.empty(exl3_encode_workspace_bytes(K, ctas), dtype=torch.uint8, device=dev)
    _check(lib.exl3_encode_tiles(_ptr(target, "target", (torch.float32,)), tiles, K, codebook,
                                 _ptr(words, "words", _WORDS, dev), _ptr(cost, "cost", (torch.float32,), dev),
                                 _ptr(workspace, "workspace", (torch.uint8,), dev), workspace.numel(),
                                 _stream(dev)))
    return words, cost


def exl3_quantize_act(x_rot: torch.Tensor):
    """int8 activations and per-128-block scales of rotated binary16 activations
    [M, n]: returns (q int8 [M, n], qscale float32 [M, n/128])."""
    lib = load_library()
    x2 = x_rot if x_rot.dim() == 2 else x_rot.view(1, -1)
    M, n = x2.shape
    q = torch.empty((M, n), dtype=torch.int8, device=x_rot.device)
    qs = torch.empty((M, n // 128), dtype=torch.float32, device=x_rot.device)
    _check(lib.exl3_quantize_act(_ptr(x2, "x_rot", _HALF), M, n, _ptr(q, "q", (torch.int8,), x_rot.device),
                                 _ptr(qs, "qscale", (torch.float32,), x_rot.device), _stream(x_rot.device)))
    return q, qs


def exl3_gemm_i8_workspace_bytes(m: int, n: int, M: int) -> int:
    return int(load_library().exl3_gemm_i8_workspace_bytes(m, n, M))


def _i8_workspace(m, n, M, dev, workspace):
    if workspace is not None:
        return workspace
    nbytes = exl3_gemm_i8_workspace_bytes(m, n, M)
    if nbytes == 0:
        raise Exl3Error(2, "invalid shape or batch for an int8 workspace")
    return torch.zeros(nbytes, dtype=torch.uint8, device=dev)


def exl3_gemm_i8(codes, K, codebook, m, n, s_out, scales, q, qscale, y=None, workspace=None):
    """The layer on int8 activations q [M, n] with per-block scales qscale [M, n/128]."""
    lib = load_library()
    dev = codes.device
    q2 = q if q.dim() == 2 else q.view(1, -1)
    M = q2.shape[0]
    if y is None:
        y = torch.empty((M, m), dtype=torch.float16, device=dev)
    workspace = _i8_workspace(m, n, M, dev, workspace)
    _check(lib.exl3_gemm_i8(
        _ptr(codes, "codes", _WORDS), K, codebook, m, n, _ptr(s_out, "s_out", _HALF, dev),
        _ptr(scales, "scales", _HALF, dev), M, _ptr(q2, "q", (torch.int8,), dev),
        _ptr(qscale, "qscale", (torch.float32,), dev), _ptr(y, "y", _HALF, dev),
        _ptr(workspace, "workspace", (torch.uint8,), dev), workspace.numel(), _stream(dev)))
    return y if q.dim() == 2 else y.view(-1)


def exl3_gemm_int8act(codes, K, codebook, m, n, s_in, s_out, scales, x, y=None, workspace=None):
    """The int8-activation layer from binary16 activations x [M, n]."""
    lib = load_library()
    dev = codes.device
    x2 = x if x.dim() == 2 else x.view(1, -1)
    M = x2.shape[0]
    if y is None:
        y = torch.empty((M, m), dtype=torch.float16, device=dev)
    workspace = _i8_workspace(m, n, M, dev, workspace)
    _check(lib.exl3_gemm_int8act(
        _ptr(codes, "codes", _WORDS), K, codebook, m, n, _ptr(s_in, "s_in", _HALF, dev),
        _ptr(s_out, "s_out", _HALF, dev), _ptr(scales, "scales", _HALF, dev), M, _ptr(x2, "x", _HALF, dev),
        _ptr(y, "y", _HALF, dev), _ptr(workspace, "workspace", (torch.uint8,), dev), workspace.numel(),
        _stream(dev)))
    return y if x.dim() == 2 else y.view(-1)


PROBE_KINDS = {0: "IMAD", 1: "LOP3", 2: "SHF", 3: "IDP4A", 4: "PRMT", 5: "IMAD+LOP3", 6: "IMAD+IDP4A+LOP3+SHF"}


def exl3_probe_int(kind: int, out: torch.Tensor, blocks: int, iters: int) -> int:
    """Launch the integer-throughput probe on the current stream of out's
    device; returns the number of instructions it executes (blocks * 8192 *
    iters).  out: int32 tensor of at least blocks * 256 elements."""
    lib = load_library()
    dev = out.device
    if out.numel() < blocks * 256:
        raise ValueError("out holds fewer than blocks * 256 words")
    _check(lib.exl3_probe_int(kind, _ptr(out, "out", _WORDS, dev), blocks, iters, _stream(dev)))
    return blocks * 8192 * iters


def exl3_gemm_launches(m: int, n: int, M: int) -> int:
    """Kernel launches of one exl3_gemm call of this shape and batch on the
    current device under the current path setting."""
    return int(load_library().exl3_gemm_launches(m, n, M))


def exl3_gemm(codes, K, codebook, m, n, s_in, s_out, scales, x, y=None, workspace=None):
    """The layer for any batch M (prefill): x [M, n] -> y [M, m]."""
    lib = load_library()
    dev = codes.device
    x2 = x if x.dim() == 2 else x.view(1, -1)
    M = x2.shape[0]
    if y is None:
        y = torch.empty((M, m), dtype=torch.float16, device=dev)
    if workspace is None:
        nbytes = exl3_gemm_workspace_bytes(m, n, M)
        if nbytes == 0:
            raise Exl3Error(2, "invalid shape or batch for a workspace")
        workspace = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
    _check(lib.exl3_gemm(
        _ptr(codes, "codes", _WORDS), K, codebook, m, n,
        _ptr(s_in, "s_in", _HALF, dev), _ptr(s_out, "s_out", _HALF, dev),
        _ptr(scales, "scales", _HALF, dev), M, _ptr(x2, "x", _HALF, dev),
        _ptr(y, "y", _HALF, dev), _ptr(workspace, "workspace", (torch.uint8,), dev),
        workspace.numel(), _stream(dev)))
    return y if x.dim() == 2 else y.view(-1)
