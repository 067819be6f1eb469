"""Helpers for the GPU parity tests: building/loading the library, moving
tensors to the oracle's numpy formats, and the stated tolerances."""
from __future__ import annotations

import numpy as np
import torch

# Tolerances for y (fp32 accumulation, bf16 operands): max-abs error within
# 1e-2 of the largest reference magnitude, relative Frobenius error <= 5e-3.
Y_MAX_REL = 1e-2
Y_FRO_REL = 5e-3
ALPHA_REL = 1e-6


def load_bd():
    from bit_delta_compressed_gb300 import build
    build.build()
    import bit_delta_compressed_gb300 as bd
    bd.get_lib()
    return bd


def bf16_np(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f32_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy().astype(np.float32)


def bits_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy().view(np.uint32)


def y_errors(y: np.ndarray, ref: np.ndarray):
    y = y.astype(np.float64)
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    max_err = float(np.max(np.abs(y - ref))) if ref.size else 0.0
    fro = float(np.linalg.norm(y - ref)) / max(float(np.linalg.norm(ref)), 1e-300)
    return max_err, scale, fro


def assert_y_close(y: np.ndarray, ref: np.ndarray, what: str = ""):
    assert y.shape == ref.shape, (y.shape, ref.shape)
    assert np.all(np.isfinite(y)), what + ": non-finite output"
    max_err, scale, fro = y_errors(y, ref)
    assert max_err <= Y_MAX_REL * scale, "%s: max err %.3e > %.1e * %.3e" % (what, max_err, Y_MAX_REL, scale)
    assert fro <= Y_FRO_REL, "%s: relative Frobenius error %.3e" % (what, fro)


def assert_alpha_close(a_gpu: float, a_ref: float, what: str = ""):
    if a_ref == 0.0:
        assert a_gpu == 0.0, what
    else:
        assert abs(a_gpu - a_ref) <= ALPHA_REL * abs(a_ref), "%s: alpha %r vs %r" % (what, a_gpu, a_ref)
