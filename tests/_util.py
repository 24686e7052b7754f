"""Small helpers shared by the tests (comparison only; no kernel arithmetic)."""
import numpy as np
import torch


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor (any device) -> uint16 numpy bit patterns."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """|ord(a) - ord(b)| for bf16 bit patterns, where ord maps sign-magnitude
    patterns onto a monotone integer line (so +0 and -0 are both 0)."""
    def ordered(u):
        u = u.astype(np.int32)
        return np.where(u & 0x8000, -(u & 0x7FFF), u)
    return np.abs(ordered(a) - ordered(b))


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().double().numpy()
