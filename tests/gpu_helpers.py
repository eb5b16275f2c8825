"""Helpers shared by the GPU parity tests (host <-> device moves and the
attention tolerance).  The tolerance is the one the library is held to:
max |err| <= 1e-2 and mean |err| <= 1e-3 against the float64 oracle."""
from __future__ import annotations

import numpy as np
import torch

MAX_TOL = 1e-2
MEAN_TOL = 1e-3


def dev(a: np.ndarray, kind: str | None = None) -> torch.Tensor:
    """NumPy -> CUDA tensor.  kind 'bf16' reinterprets uint16 bits as bfloat16;
    'u32' reinterprets uint32 as int32."""
    a = np.ascontiguousarray(a)
    if kind == "bf16":
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    if kind == "u32":
        return torch.from_numpy(a.view(np.int32)).cuda()
    return torch.from_numpy(a).cuda()


def host_bits(t: torch.Tensor) -> np.ndarray:
    """CUDA 16-bit tensor -> NumPy uint16 bit patterns."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def assert_attention_close(got: np.ndarray, ref: np.ndarray, what: str = "",
                           max_tol: float = MAX_TOL, mean_tol: float = MEAN_TOL) -> None:
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    assert err.max() <= max_tol, f"{what}: max |err| {err.max():.3e} > {max_tol}"
    assert err.mean() <= mean_tol, f"{what}: mean |err| {err.mean():.3e} > {mean_tol}"


def new_status() -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device="cuda")
