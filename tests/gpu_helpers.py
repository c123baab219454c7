"""Shared helpers of the GPU parity tests: upload of the seeded synthetic
inputs and the layer tolerance of the correctness criteria (relative L2 error
<= 5e-3 and every |err| <= 1e-2 * max|y_ref| against the oracle's float64
result)."""
import numpy as np
import torch

REL_L2 = 5e-3
MAX_ABS_FRAC = 1e-2


def to_dev(a: np.ndarray, device="cuda"):
    if a is None:
        return None
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def upload(inp: dict, device="cuda") -> dict:
    return {k: to_dev(v, device) for k, v in inp.items()}


def layer_error(y_gpu, y_ref: np.ndarray):
    y = y_gpu.detach().float().cpu().numpy().astype(np.float64).reshape(y_ref.shape)
    assert np.all(np.isfinite(y)), "non-finite output"
    err = y - y_ref
    rel = np.linalg.norm(err) / max(np.linalg.norm(y_ref), 1e-300)
    frac = np.abs(err).max() / max(np.abs(y_ref).max(), 1e-300)
    return rel, frac


def assert_layer_close(y_gpu, y_ref: np.ndarray, what=""):
    rel, frac = layer_error(y_gpu, y_ref)
    assert rel <= REL_L2, f"{what}: relative L2 error {rel:.3e} > {REL_L2}"
    assert frac <= MAX_ABS_FRAC, f"{what}: max |err| / max|y_ref| = {frac:.3e} > {MAX_ABS_FRAC}"
    return rel, frac
