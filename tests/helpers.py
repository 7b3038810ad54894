"""Conversions between torch tensors and the oracle's numpy arrays (no method
arithmetic here)."""
import numpy as np
import torch


def to_np(t: torch.Tensor) -> np.ndarray:
    """float32 -> float32 array; bfloat16 -> uint16 array of the raw bits;
    E4M3 bytes -> uint8 array."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    if t.dtype == torch.float32:
        return t.numpy().copy()
    if t.dtype in (torch.int32, torch.int64):
        return t.numpy().astype(np.int32)
    if t.dtype == torch.uint8 or t.dtype == getattr(torch, "float8_e4m3fn", None):
        return t.view(torch.uint8).numpy().copy()
    raise TypeError(t.dtype)


def from_np(a: np.ndarray) -> torch.Tensor:
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16)
    return torch.from_numpy(a.copy())


def oracle_inputs(t: dict) -> dict:
    """The generator's torch tensors as oracle arrays (host copies)."""
    return {k: to_np(v) for k, v in t.items()}
