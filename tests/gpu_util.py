"""Shared helpers for the GPU parity tests (test infrastructure only)."""

from __future__ import annotations

import numpy as np

import synth

# Tolerances for O and LSE of bf16-input / fp32-accumulate attention against the
# fp64 oracle.
O_MAX_ABS = 2e-2
O_MEAN_ABS = 2e-3
LSE_MAX_ABS = 1e-3


def to_dev(bits: np.ndarray, device="cuda"):
    """uint16 bf16 bit patterns -> CUDA bfloat16 tensor (bit-exact)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).to(device)


def to_dev_i32(a: np.ndarray, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def from_dev(t) -> np.ndarray:
    """CUDA tensor -> float64 numpy (bf16 widened exactly)."""
    import torch
    return t.detach().to(torch.float32).cpu().numpy().astype(np.float64)


def bits_of(t) -> np.ndarray:
    """bf16 CUDA tensor -> uint16 bit patterns."""
    import torch
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def check_close(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    err = np.abs(o_gpu - o_ref)
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite O"
    assert err.max() <= O_MAX_ABS, f"{what}: O max-abs {err.max():.3e}"
    assert err.mean() <= O_MEAN_ABS, f"{what}: O mean-abs {err.mean():.3e}"
    if lse_gpu is not None:
        lerr = np.abs(lse_gpu - lse_ref)
        assert np.all(np.isfinite(lse_gpu)), f"{what}: non-finite LSE"
        assert lerr.max() <= LSE_MAX_ABS, f"{what}: LSE max-abs {lerr.max():.3e}"
    return float(err.max()), float(err.mean())
