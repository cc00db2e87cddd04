"""Helpers for the GPU tests."""
from __future__ import annotations

import numpy as np
import torch

from quantized_swiglu_mlp_gb300.inputs import device_args, operand_to_device  # noqa: F401


def to_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns on the host."""
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
