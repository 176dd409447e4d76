"""Helpers shared by the GPU parity tests: moving seeded bf16 inputs to the device, the
tolerances the parity bar fixes, and error metrics."""

import numpy as np
import torch

from oracle import attention as A

# Tolerances against the fp64 oracle on the same bf16 inputs.
O_MAX_ABS = 1e-2
O_REL_FRO = 5e-3
LSE_MAX_ABS = 1e-3
GRAD_REL_FRO = 2e-2


def to_device(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


def widen(bits: np.ndarray) -> np.ndarray:
    return A.bf16_bits_to_f64(bits)


def rel_fro(x: np.ndarray, ref: np.ndarray) -> float:
    return float(np.linalg.norm((x - ref).ravel()) / max(np.linalg.norm(ref.ravel()), 1e-30))


def max_abs(x: np.ndarray, ref: np.ndarray) -> float:
    return float(np.max(np.abs(x - ref))) if x.size else 0.0
