"""Helpers shared by the GPU parity tests (comparison and tolerance only)."""
import numpy as np
import torch

# BF16 outputs and gradients vs the fp64 oracle: max-abs 2e-2, mean-abs 2e-3.
MAX_ABS = 2e-2
MEAN_ABS = 2e-3


def dev():
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def assert_close(got, ref, what: str, max_abs: float = MAX_ABS, mean_abs: float = MEAN_ABS):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = np.abs(got - ref)
    mx, mn = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    assert mx <= max_abs and mn <= mean_abs, \
        f"{what}: max-abs {mx:.3e} (limit {max_abs}), mean-abs {mn:.3e} (limit {mean_abs}), " \
        f"max |ref| {float(np.abs(ref).max()) if ref.size else 0:.3f}"
    return mx, mn


def assert_lse_close(got, ref, what: str, tol: float = 1e-3):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    inf_ref = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), inf_ref), f"{what}: -inf pattern differs"
    err = np.abs(got[~inf_ref] - ref[~inf_ref])
    assert err.size == 0 or err.max() <= tol, f"{what}: LSE max-abs {err.max():.3e}"
