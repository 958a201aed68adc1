"""fp64 CPU oracle of the delta-rule fast-weight layer core with DPFP.

TEST INFRASTRUCTURE ONLY.  Only tests/, the smoke check and the benchmark's
CPU-baseline leg may import this package.  The CUDA library never does, and
this package never imports the CUDA library: the two share no code.

Contents
  dpfp(x, nu, eps)                  -- the DPFP feature map, plain C, fp64
  delta_forward(q, k, v, beta, ...) -- O1: the sequential recurrence, plain C
  delta_decode_step(...)            -- one token against a persistent W
  project(x, W_all, H, d_key, d_v)  -- the attention module's projections:
                                       q, k, v per head and beta = sigmoid(.),
                                       numpy fp64
  delta_backward(q, k, v, beta, ...) -- gradients of the recurrence (reverse
                                       sweep over the kept history of W), plain C
  linear_forward(q, k, v, ...)      -- the sum rule (linear attention, with or
                                       without the z normaliser), plain C
  chunked.delta_forward_chunked     -- O2: the chunked (WY / UT) form in numpy,
                                       for tiny brute-force checks of O1
  stack.stack_step, stack.layer_norm -- one token through the token-wise layer
                                       stack (projections, decode step, output
                                       map, LayerNorm, feed-forward), numpy fp64

All arrays are numpy float64 (inputs are converted with np.asarray(...,
dtype=float64), so rounded bf16/fp32 values enter exactly).  fw_oracle.c cites
the passage of the Fast Weights Transformer guide (xdnf.cn/news/308600) that
each routine follows.  Parity is pinned by tests/test_oracle_*.py against
hand-worked examples (tests/golden/), closed forms, invariants, an FFT
identity and the independent chunked form O2; tests/test_oracle_mutants.py
shows that planted mistakes in fw_oracle.c fail those pins, and
tests/test_oracle_stack.py does the same for stack.py.  No function is
left unpinned.
"""
import ctypes
import os

import numpy as np

from .build import build_oracle

_c_double_p = ctypes.POINTER(ctypes.c_double)


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a):
    return None if a is None else a.ctypes.data_as(_c_double_p)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


class OracleLib:
    """The oracle's entry points bound to one compiled copy of fw_oracle.c."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        lib.fwo_dpfp.restype = ctypes.c_int
        lib.fwo_dpfp.argtypes = [_c_double_p, _c_double_p, ctypes.c_int64, ctypes.c_int,
                                 ctypes.c_int, ctypes.c_double]
        lib.fwo_delta_forward.restype = ctypes.c_int
        lib.fwo_delta_forward.argtypes = [_c_double_p] * 7 + [ctypes.c_int64] * 3 + [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int]
        lib.fwo_delta_decode_step.restype = ctypes.c_int
        lib.fwo_delta_decode_step.argtypes = [_c_double_p] * 6 + [ctypes.c_int64] * 2 + [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int]
        lib.fwo_delta_backward.restype = ctypes.c_int
        lib.fwo_delta_backward.argtypes = [_c_double_p] * 12 + [ctypes.c_int64] * 3 + [
            ctypes.c_int] * 3 + [ctypes.c_double, ctypes.c_int]
        lib.fwo_linear_forward.restype = ctypes.c_int
        lib.fwo_linear_forward.argtypes = [_c_double_p] * 8 + [ctypes.c_int64] * 3 + [
            ctypes.c_int] * 4 + [ctypes.c_double, ctypes.c_int]
        self._lib = lib
        self.path = path

    def dpfp(self, x, nu: int = 1, eps: float = 1e-6):
        """phi(x) over the last axis: [..., d_key] -> [..., 2*d_key*nu] (fp64)."""
        x = _f64(x)
        d_key = x.shape[-1]
        rows = int(np.prod(x.shape[:-1])) if x.ndim > 1 else 1
        out = np.empty(x.shape[:-1] + (2 * d_key * nu,), dtype=np.float64)
        rc = self._lib.fwo_dpfp(_p(x), _p(out), rows, d_key, nu, eps)
        if rc != 0:
            raise ValueError(f"oracle dpfp rejected arguments (d_key={d_key}, nu={nu})")
        return out

    def delta_forward(self, q, k, v, beta, W0=None, nu: int = 1, eps: float = 1e-6,
                      nthreads: int = 1):
        """O1, the sequential recurrence.

        q, k: [B,H,L,d_key]; v: [B,H,L,d_v]; beta: [B,H,L]; W0:
        [B,H,d_v,d_dot] or None (zeros).  Returns (y [B,H,L,d_v],
        W_final [B,H,d_v,d_dot]) in fp64.
        """
        q, k, v, beta = _f64(q), _f64(k), _f64(v), _f64(beta)
        B, H, L, d_key = q.shape
        d_v = v.shape[-1]
        d_dot = 2 * d_key * nu
        assert k.shape == q.shape and v.shape == (B, H, L, d_v) and beta.shape == (B, H, L)
        W0 = None if W0 is None else _f64(W0)
        if W0 is not None:
            assert W0.shape == (B, H, d_v, d_dot)
        y = np.empty((B, H, L, d_v), dtype=np.float64)
        W_final = np.empty((B, H, d_v, d_dot), dtype=np.float64)
        rc = self._lib.fwo_delta_forward(_p(q), _p(k), _p(v), _p(beta), _p(W0), _p(W_final),
                                         _p(y), B, H, L, d_key, nu, d_v, eps, int(nthreads))
        if rc != 0:
            raise ValueError("oracle delta_forward rejected arguments")
        return y, W_final

    def delta_decode_step(self, q, k, v, beta, W, nu: int = 1, eps: float = 1e-6,
                          nthreads: int = 1):
        """One token of the token-wise variant.

        q, k: [B,H,d_key]; v: [B,H,d_v]; beta: [B,H]; W: [B,H,d_v,d_dot].
        Returns (y [B,H,d_v], W_next) without modifying the caller's W.
        """
        q, k, v, beta = _f64(q), _f64(k), _f64(v), _f64(beta)
        W = _f64(W).copy()
        B, H, d_key = q.shape
        d_v = v.shape[-1]
        y = np.empty((B, H, d_v), dtype=np.float64)
        rc = self._lib.fwo_delta_decode_step(_p(q), _p(k), _p(v), _p(beta), _p(W), _p(y), B, H,
                                             d_key, nu, d_v, eps, int(nthreads))
        if rc != 0:
            raise ValueError("oracle delta_decode_step rejected arguments")
        return y, W


    def delta_backward(self, q, k, v, beta, gy, W0=None, gW=None, nu: int = 1, eps: float = 1e-6,
                       nthreads: int = 1):
        """Gradients of sum(gy * y) + sum(gW * W_final) for the forward above.

        gy: [B,H,L,d_v]; gW: [B,H,d_v,d_dot] or None (zero).  Returns
        (gq, gk, gv, gbeta, gW0) in fp64.
        """
        q, k, v, beta, gy = _f64(q), _f64(k), _f64(v), _f64(beta), _f64(gy)
        B, H, L, d_key = q.shape
        d_v = v.shape[-1]
        d_dot = 2 * d_key * nu
        W0 = None if W0 is None else _f64(W0)
        gW = None if gW is None else _f64(gW)
        gq, gk = np.empty_like(q), np.empty_like(k)
        gv, gbeta = np.empty_like(v), np.empty_like(beta)
        gW0 = np.empty((B, H, d_v, d_dot), dtype=np.float64)
        rc = self._lib.fwo_delta_backward(_p(q), _p(k), _p(v), _p(beta), _p(W0), _p(gy), _p(gW), _p(gq), _p(gk),
                                          _p(gv), _p(gbeta), _p(gW0), B, H, L, d_key, nu, d_v, eps, int(nthreads))
        if rc != 0:
            raise ValueError("oracle delta_backward rejected arguments")
        return gq, gk, gv, gbeta, gW0

    def linear_forward(self, q, k, v, W0=None, z0=None, nu: int = 1, normalize: bool = True,
                       eps: float = 1e-6, nthreads: int = 1):
        """The sum rule (linear attention) as a recurrence.

        q, k: [B,H,L,d_key]; v: [B,H,L,d_v]; W0: [B,H,d_v,d_dot] or None;
        z0: [B,H,d_dot] or None (zeros).  Returns (y [B,H,L,d_v], W_final,
        z_final) in fp64.
        """
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, H, L, d_key = q.shape
        d_v = v.shape[-1]
        d_dot = 2 * d_key * nu
        assert k.shape == q.shape and v.shape == (B, H, L, d_v)
        W0 = None if W0 is None else _f64(W0)
        z0 = None if z0 is None else _f64(z0)
        y = np.empty((B, H, L, d_v), dtype=np.float64)
        W_final = np.empty((B, H, d_v, d_dot), dtype=np.float64)
        z_final = np.empty((B, H, d_dot), dtype=np.float64)
        rc = self._lib.fwo_linear_forward(_p(q), _p(k), _p(v), _p(W0), _p(z0), _p(W_final), _p(z_final),
                                          _p(y), B, H, L, d_key, nu, d_v, int(bool(normalize)), eps,
                                          int(nthreads))
        if rc != 0:
            raise ValueError("oracle linear_forward rejected arguments")
        return y, W_final, z_final


_default = None


def lib() -> OracleLib:
    """The oracle built from oracle/fw_oracle.c (compiled on first use)."""
    global _default
    if _default is None:
        _default = OracleLib(build_oracle())
    return _default


def dpfp(x, nu: int = 1, eps: float = 1e-6):
    return lib().dpfp(x, nu, eps)


def delta_forward(q, k, v, beta, W0=None, nu: int = 1, eps: float = 1e-6, nthreads: int = 1):
    return lib().delta_forward(q, k, v, beta, W0, nu, eps, nthreads)


def delta_decode_step(q, k, v, beta, W, nu: int = 1, eps: float = 1e-6, nthreads: int = 1):
    return lib().delta_decode_step(q, k, v, beta, W, nu, eps, nthreads)


def linear_forward(q, k, v, W0=None, z0=None, nu: int = 1, normalize: bool = True, eps: float = 1e-6,
                   nthreads: int = 1):
    return lib().linear_forward(q, k, v, W0, z0, nu, normalize, eps, nthreads)


def delta_backward(q, k, v, beta, gy, W0=None, gW=None, nu: int = 1, eps: float = 1e-6, nthreads: int = 1):
    return lib().delta_backward(q, k, v, beta, gy, W0, gW, nu, eps, nthreads)


def project(x, W_all, H: int, d_key: int, d_v: int):
    """The bias-free projections of the attention module (the Fast Weights
    Transformer guide: q, k, v from linear maps of the model width to each
    head's width, beta from a linear map to one scalar per head followed by
    the sigmoid), in fp64: P = x W_all with W_all = [W_q | W_k | W_v | W_beta]
    side by side; head h takes columns h*d .. (h+1)*d - 1 of its block.
    x: [B, L, d_model]; returns q, k [B,H,L,d_key], v [B,H,L,d_v], beta [B,H,L]."""
    x = _f64(x)
    W = _f64(W_all)
    B, L, _ = x.shape
    P = np.matmul(x, W)
    nq, nv = H * d_key, H * d_v

    def heads(a, d):
        return np.ascontiguousarray(a.reshape(B, L, H, d).transpose(0, 2, 1, 3))
    q = heads(P[..., :nq], d_key)
    k = heads(P[..., nq:2 * nq], d_key)
    v = heads(P[..., 2 * nq:2 * nq + nv], d_v)
    beta = np.ascontiguousarray((1.0 / (1.0 + np.exp(-P[..., 2 * nq + nv:2 * nq + nv + H]))).transpose(0, 2, 1))
    return q, k, v, beta
