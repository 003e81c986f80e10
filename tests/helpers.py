"""Small test helpers: torch tensor <-> numpy storage arrays for the oracle."""
import numpy as np
import torch


def storage(t: torch.Tensor) -> np.ndarray:
    """A CPU numpy view of a tensor's storage: float32 for f32, uint16 bits for f16/bf16."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.float32:
        return t.numpy()
    if t.dtype in (torch.float16, torch.bfloat16):
        return t.view(torch.int16).numpy().view(np.uint16)
    raise TypeError(t.dtype)


def from_storage(a: np.ndarray, dtype: str) -> torch.Tensor:
    if dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16))
    return t.view(torch.float16 if dtype == "f16" else torch.bfloat16)


def as_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().to(torch.float64).numpy()


def nested(a: np.ndarray):
    """numpy array -> nested Python lists of floats (for the brute force)."""
    return a.astype(np.float64).tolist()
