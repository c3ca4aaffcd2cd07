"""Shared helpers for the GPU parity tests: device upload/download and the tolerance.

The oracle and the CUDA path meet only here, on the same seeded inputs from
``workloads.py``.
"""
from __future__ import annotations

import numpy as np
import torch

# Relative Frobenius error allowed per matrix between the CUDA path and the fp64
# oracle, for the same steps and coefficients on the same inputs.
TOL = 2e-2


def dev(x: np.ndarray, dtype: str = "bf16") -> torch.Tensor:
    """Uploads a float32 array (already representable in dtype) to cuda:0."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    t = t.to(torch.bfloat16) if dtype == "bf16" else t
    return t.cuda()


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel_f(x, ref) -> float:
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    n = np.linalg.norm(ref)
    d = np.linalg.norm(x - ref)
    return float(d / n) if n > 0 else float(d)


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    a = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 2.0 ** (e - 7)
