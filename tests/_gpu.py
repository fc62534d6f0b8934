"""Helpers for the GPU parity tests (tolerances and bit-exact comparisons)."""

import numpy as np
import torch

# bf16-in / fp32-accumulate outputs against the fp64 oracle: max-abs 1e-2 and
# mean-abs 1e-3.  An output stored in bf16 with |o| >= 4 sits on a grid of
# spacing 2^-5, so rounding alone can move it by up to 2^-6 = 0.0156 > 1e-2;
# there the element bound is half a bf16 ulp (at the larger of |reference| and
# |output|, since a value just below 4 may round onto the coarser grid above)
# plus 2e-3 of arithmetic slack; below 4 the bound is the flat 1e-2.
MAX_ABS = 1e-2
MEAN_ABS = 1e-3
LSE_ABS = 2e-3
ARITH_SLACK = 2e-3


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    """Half the spacing of the bf16 grid at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(ax)) - 8)


def element_bound(ref: np.ndarray, out: np.ndarray) -> np.ndarray:
    return np.maximum(MAX_ABS, bf16_half_ulp(np.maximum(np.abs(ref), np.abs(out))) + ARITH_SLACK)


def assert_close(gpu: torch.Tensor, ref: np.ndarray, what: str = "output"):
    g = gpu.detach().float().cpu().numpy().astype(np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape, (what, g.shape, ref.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    err = np.abs(g - ref)
    mx = float(err.max(initial=0.0))
    mean = float(err.mean()) if err.size else 0.0
    over = err > element_bound(ref, g)
    if over.any():
        j = np.unravel_index(np.argmax(np.where(over, err, -1.0)), err.shape)
        raise AssertionError(f"{what}: {int(over.sum())} elements over the bound; worst {err[j]:.3e} at "
                             f"ref {ref[j]:.4f}, out {g[j]:.4f}; max abs {mx:.3e}")
    assert mean <= MEAN_ABS, f"{what}: mean abs {mean:.3e}"
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
