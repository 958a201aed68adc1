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


def elementwise(got, ref):
    """Per-element relative error |g_i - r_i| / max(|r_i|, 1e-6 * max_j |r_j|).

    The floor keeps entries that are zero or nearly so in the reference from
    dividing by ~0.  Returns the largest value with its index, the median and
    the 99.9th percentile."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if ref.size == 0:
        return dict(max=0.0, at=(), median=0.0, p999=0.0)
    scale = np.abs(ref).max()
    den = np.maximum(np.abs(ref), 1e-6 * scale if scale > 0 else 1e-30)
    e = np.abs(got - ref) / den
    at = np.unravel_index(int(np.argmax(e)), e.shape)
    return dict(max=float(e[at]), at=tuple(int(i) for i in at), median=float(np.median(e)),
                p999=float(np.quantile(e, 0.999)))


def check(name, got, ref, tol):
    """Normwise max relative error within tol (the stated bar), with the
    element-wise report printed beside it; the median element-wise error must
    be within tol too, so that a bar met only thanks to a few large entries
    cannot hide errors spread over the small ones."""
    n = maxrel(got, ref)
    e = elementwise(got, ref)
    print(f"{name}: normwise {n:.3e} | element-wise max {e['max']:.3e} at {e['at']}, "
          f"median {e['median']:.3e}, p99.9 {e['p999']:.3e}")
    assert n <= tol, (name, n, tol)
    assert e["median"] <= tol, (name, e, tol)
    return n, e
