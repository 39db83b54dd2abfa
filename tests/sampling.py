"""Float64 copies of selected (batch, head) slices, for full-size parity tests
that compare sampled heads with the oracle without upcasting whole tensors."""
import numpy as np
import torch


def head_slices(t: torch.Tensor, heads) -> np.ndarray:
    """[B, H, rows, width] (CPU) -> float64 [len(heads), rows, width] for flat heads b*H + h."""
    flat = t.reshape((-1,) + tuple(t.shape[2:]))
    return np.stack([flat[h].to(torch.float64).numpy() for h in heads])
