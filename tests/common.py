"""Helpers shared by the tests: bf16 bit views and error norms (no layer arithmetic here)."""

import numpy as np
import torch


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The raw 16-bit patterns of a bf16 tensor, as numpy uint16 (copied to host)."""
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def max_rel_err(got, ref) -> float:
    """max|got - ref| / max|ref| (the parity norm of the layer's output)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    denom = np.max(np.abs(ref))
    if denom == 0:
        return float(np.max(np.abs(got)))
    return float(np.max(np.abs(got - ref)) / denom)
