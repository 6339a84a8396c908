"""Test-side marshalling between torch tensors and the oracle's numpy arrays."""
import numpy as np
import torch


def raw(t: torch.Tensor) -> np.ndarray:
    """torch tensor (any device) -> numpy array of the oracle's raw element type."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    if t.dtype == torch.float32:
        return t.numpy().copy()
    if t.dtype == torch.int64:
        return t.numpy().copy()
    raise TypeError(t.dtype)


def dt_name(dtype: torch.dtype) -> str:
    return {torch.float32: "f32", torch.bfloat16: "bf16"}[dtype]


def from_raw(a: np.ndarray, dtype: torch.dtype) -> torch.Tensor:
    if dtype == torch.bfloat16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a))


def to_f64(t: torch.Tensor) -> torch.Tensor:
    return t.detach().cpu().to(torch.float64)
