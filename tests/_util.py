"""Small helpers shared by the tests (no attention arithmetic here)."""
import numpy as np
import torch


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw 16-bit patterns of a fp16/bf16 tensor as a numpy uint16 array (CPU copy)."""
    assert t.dtype in (torch.float16, torch.bfloat16)
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def from_bits(a: np.ndarray, dtype: torch.dtype) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(dtype)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().to(torch.float64).numpy()
