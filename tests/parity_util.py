"""Helpers shared by the GPU parity tests: moving seeded inputs to the device,
turning them into the exact fp64 values the oracle reads, and the error
measure the tolerances are stated in."""
import numpy as np
import torch

# Stated tolerances (max normwise relative error, see maxrel):
TOL_F32 = 1e-4   # fp32 I/O
TOL_BF16 = 2e-2  # bf16 I/O with fp32 state


def tol_for(dtype):
    return TOL_F32 if dtype == torch.float32 else TOL_BF16


def f64(t):
    """Exact fp64 copy of a (possibly bf16, possibly CUDA) tensor."""
    return t.detach().to("cpu", torch.float32).double().numpy()


def maxrel(got, ref):
    """max_i |g_i - r_i| / max_i |r_i| (normwise: no division by tiny entries)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "non-finite values in the GPU output"
    scale = np.abs(ref).max() if ref.size else 0.0
    if scale == 0.0:
        return float(np.abs(got).max()) if got.size else 0.0
    return float(np.abs(got - ref).max() / scale)


def to_dev(d, device="cuda"):
    return {k: (None if v is None else v.to(device)) for k, v in d.items()}
