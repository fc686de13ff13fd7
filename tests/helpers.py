"""Shared test helpers: storage <-> torch marshalling and NaN-aware bit comparison."""

import numpy as np
import torch

TORCH_DTYPE = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16, "i32": torch.int32}
ELEM_SIZE = {"f32": 4, "f16": 2, "bf16": 2, "i32": 4}


def to_device(a: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    if dtype == "bf16":
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


def to_host(t: torch.Tensor, dtype: str) -> np.ndarray:
    t = t.detach().cpu()
    if dtype == "bf16":
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.numpy().copy()


def is_nan_bits(a: np.ndarray, dtype: str) -> np.ndarray:
    if dtype in ("f32", "f16"):
        return np.isnan(a)
    if dtype == "bf16":
        return ((a & 0x7F80) == 0x7F80) & ((a & 0x007F) != 0)
    return np.zeros(a.shape, dtype=bool)


def assert_same_bits(got: np.ndarray, want: np.ndarray, dtype: str, what: str = ""):
    """Bit-exact equality, except that any NaN equals any NaN (payloads are not compared)."""
    assert got.shape == want.shape, f"{what}: shape {got.shape} != {want.shape}"
    if got.size == 0:
        return
    gn, wn = is_nan_bits(got, dtype), is_nan_bits(want, dtype)
    assert np.array_equal(gn, wn), f"{what}: NaN positions differ"
    g = got.view(np.uint8).reshape(got.shape[0], -1)
    w = want.view(np.uint8).reshape(want.shape[0], -1)
    ok = gn | (g == w).all(axis=1)
    bad = np.flatnonzero(~ok)
    assert bad.size == 0, (f"{what}: {bad.size} of {got.size} elements differ, first at {bad[:5]}: "
                           f"got {got[bad[:5]]} want {want[bad[:5]]}")
