"""Helpers for the GPU parity tests (tolerances and bit-exact comparisons)."""

import numpy as np
import torch

# bf16-in / fp32-accumulate outputs against the fp64 oracle
MAX_ABS = 1e-2
MEAN_ABS = 1e-3
LSE_ABS = 2e-3


def assert_close(gpu: torch.Tensor, ref: np.ndarray, what: str = "output"):
    g = gpu.detach().float().cpu().numpy().astype(np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape, (what, g.shape, ref.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    err = np.abs(g - ref)
    mx = float(err.max(initial=0.0))
    mean = float(err.mean()) if err.size else 0.0
    assert mx <= MAX_ABS and mean <= MEAN_ABS, f"{what}: max abs {mx:.3e}, mean abs {mean:.3e}"
    return mx, mean


def assert_lse(gpu: torch.Tensor, ref: np.ndarray, what: str = "lse"):
    g = gpu.detach().double().cpu().numpy()
    ref = np.asarray(ref, dtype=np.float64)
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(g), fin), f"{what}: -inf pattern differs"
    if fin.any():
        err = np.abs(g[fin] - ref[fin]).max()
        assert err <= LSE_ABS, f"{what}: max abs {err:.3e}"


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns (bit-exact comparisons)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy()
