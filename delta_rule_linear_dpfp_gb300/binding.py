"""Thin Python binding of the C ABI in include/fastweight.h.

Argument marshalling only: every function here checks tensor shapes/dtypes,
allocates missing outputs with PyTorch (device memory is PyTorch's job) and
calls the entry point of the same name in libfastweight.so through ctypes on
the current CUDA stream.  All arithmetic runs in the library's sm_103a
kernels.  There is no fallback: if the library is missing the import of a
function raises, and a non-zero status raises FwError.
"""
import ctypes
import os

import torch

from . import build as _build

FW_OK = 0
FW_ERR_INVALID_ARG = 1
FW_ERR_UNSUPPORTED = 2
FW_ERR_CUDA = 3
FW_ERR_TIMEOUT = 4
FW_DTYPE_F32 = 0
FW_DTYPE_BF16 = 1

#: every entry point include/*.h declares
EXPORTS = ("fw_status_string", "fw_dpfp", "fw_delta_forward_workspace_size", "fw_delta_forward",
           "fw_delta_forward_kernel_count",
           "fw_delta_decode_step", "fw_device_status", "fw_selftest_umma",
           "fw_delta_forward_noalloc", "fw_delta_forward_prepare", "fw_delta_forward_scan",
           "fw_selftest_wait_timeout", "fw_selftest_flag_timeout", "fw_linear_forward_workspace_size",
           "fw_linear_forward",
           "fw_delta_backward_workspace_size", "fw_delta_backward",
           "fw_delta_forward_projected_workspace_size", "fw_delta_forward_projected",
           "fw_decode_stack_workspace_size", "fw_decode_stack_step")

#: the members of fw_stack_layer, in order
STACK_FIELDS = ("W_in", "W_o", "b_o", "ln_gamma", "ln_beta", "W_1", "b_1", "W_2", "b_2", "W")

#: bytes of the library's own scratch array behind fw_delta_forward_noalloc
NOALLOC_SCRATCH_BYTES = 64 << 20

_lib = None


class FwStackLayer(ctypes.Structure):
    """fw_stack_layer of fastweight.h: one layer's device pointers."""
    _fields_ = [(n, ctypes.c_void_p) for n in STACK_FIELDS]


class FwError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__(f"{where}: {status_string(code)}")


def lib_path() -> str:
    return _build.LIB


def load(path: str = None) -> ctypes.CDLL:
    """Load libfastweight.so (built by delta_rule_linear_dpfp_gb300.build)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _build.LIB
    if not os.path.exists(p):
        raise RuntimeError(f"libfastweight.so is not built ({p}); run "
                           "delta_rule_linear_dpfp_gb300.build.build() first")
    lib = ctypes.CDLL(p)
    vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.fw_status_string.restype = ctypes.c_char_p
    lib.fw_status_string.argtypes = [i32]
    lib.fw_dpfp.restype = i32
    lib.fw_dpfp.argtypes = [vp, vp, i64, i32, i32, i32, i32, f32, vp]
    lib.fw_delta_forward_workspace_size.restype = sz
    lib.fw_delta_forward_workspace_size.argtypes = [i32] * 8
    lib.fw_delta_forward.restype = i32
    lib.fw_delta_forward.argtypes = [vp] * 8 + [sz] + [i32] * 8 + [f32, vp]
    lib.fw_delta_forward_kernel_count.restype = i32
    lib.fw_delta_forward_kernel_count.argtypes = [i32] * 8
    lib.fw_delta_decode_step.restype = i32
    lib.fw_delta_decode_step.argtypes = [vp] * 6 + [i32] * 6 + [f32, vp]
    lib.fw_device_status.restype = i32
    lib.fw_device_status.argtypes = [vp]
    lib.fw_delta_forward_prepare.restype = i32
    lib.fw_delta_forward_prepare.argtypes = [vp] * 5 + [sz] + [i32] * 7 + [f32, vp]
    lib.fw_delta_forward_scan.restype = i32
    lib.fw_delta_forward_scan.argtypes = [vp, sz, vp, vp, vp] + [i32] * 7 + [vp]
    lib.fw_delta_forward_noalloc.restype = i32
    lib.fw_delta_forward_noalloc.argtypes = [vp] * 7 + [i32] * 8 + [f32, vp]
    lib.fw_selftest_wait_timeout.restype = i32
    lib.fw_selftest_wait_timeout.argtypes = [i32, vp]
    lib.fw_selftest_flag_timeout.restype = i32
    lib.fw_selftest_flag_timeout.argtypes = [i32, vp]
    lib.fw_linear_forward_workspace_size.restype = sz
    lib.fw_linear_forward_workspace_size.argtypes = [i32] * 9
    lib.fw_linear_forward.restype = i32
    lib.fw_linear_forward.argtypes = [vp] * 9 + [sz] + [i32] * 9 + [f32, vp]
    lib.fw_delta_backward_workspace_size.restype = sz
    lib.fw_delta_backward_workspace_size.argtypes = [i32] * 7
    lib.fw_delta_backward.restype = i32
    lib.fw_delta_backward.argtypes = [vp] * 13 + [sz] + [i32] * 7 + [f32, vp]
    lib.fw_delta_forward_projected_workspace_size.restype = sz
    lib.fw_delta_forward_projected_workspace_size.argtypes = [i32] * 8
    lib.fw_delta_forward_projected.restype = i32
    lib.fw_delta_forward_projected.argtypes = [vp, vp, i32, vp, vp, vp, vp, sz] + [i32] * 8 + [f32, vp]
    lib.fw_decode_stack_workspace_size.restype = sz
    lib.fw_decode_stack_workspace_size.argtypes = [i32] * 6
    lib.fw_decode_stack_step.restype = i32
    lib.fw_decode_stack_step.argtypes = [ctypes.POINTER(FwStackLayer), i32, vp, vp, vp, vp, vp, sz] + [i32] * 8 + [
        f32, f32, vp]
    lib.fw_selftest_umma.restype = i32
    lib.fw_selftest_umma.argtypes = [vp, vp, vp] + [i32] * 5 + [vp]
    if path is None:
        _lib = lib
    return lib


def status_string(code: int) -> str:
    return load().fw_status_string(int(code)).decode()


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.float32:
        return FW_DTYPE_F32
    if t == torch.bfloat16:
        return FW_DTYPE_BF16
    raise TypeError(f"unsupported dtype {t}; use torch.float32 or torch.bfloat16")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(code, where):
    if code != FW_OK:
        raise FwError(code, where)


def _dev(t, name):
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")


def fw_dpfp(x, nu: int = 1, eps: float = 1e-6, out_dtype=None, out=None, stream=None):
    """phi = DPFP(x) over the last axis: [..., d_key] -> [..., 2*d_key*nu]."""
    _dev(x, "x")
    d_key = x.shape[-1]
    out_dtype = out_dtype or x.dtype
    if out is None:
        out = torch.empty(*x.shape[:-1], 2 * d_key * nu, dtype=out_dtype, device=x.device)
    _dev(out, "out")
    rows = x.numel() // d_key if d_key else 0
    rc = load().fw_dpfp(_ptr(x), _ptr(out), rows, d_key, nu, _dtype_code(x.dtype),
                        _dtype_code(out.dtype), eps, _stream(stream))
    _check(rc, "fw_dpfp")
    return out


def fw_delta_forward_workspace_size(B, H, L, d_key, nu, d_v, chunk, io_dtype) -> int:
    code = io_dtype if isinstance(io_dtype, int) else _dtype_code(io_dtype)
    return int(load().fw_delta_forward_workspace_size(B, H, L, d_key, nu, d_v, chunk, code))


def fw_delta_forward_kernel_count(B, H, L, d_key, nu, d_v, chunk, io_dtype) -> int:
    """Kernels fw_delta_forward enqueues for this shape on the current device:
    1 (one cooperative launch) or 2 (prep, then scan) with bf16 I/O; -1 if
    the shape is rejected."""
    code = io_dtype if isinstance(io_dtype, int) else _dtype_code(io_dtype)
    return int(load().fw_delta_forward_kernel_count(B, H, L, d_key, nu, d_v, chunk, code))


def fw_delta_forward(q, k, v, beta, W0=None, nu: int = 1, chunk: int = 64, eps: float = 1e-6,
                     return_state: bool = True, y=None, W_final=None, workspace=None, stream=None):
    """Delta-rule forward over [B,H,L,*] inputs.  Returns (y, W_final or None)."""
    for name, t in (("q", q), ("k", k), ("v", v), ("beta", beta)):
        _dev(t, name)
    B, H, L, d_key = q.shape
    d_v = v.shape[-1]
    d_dot = 2 * d_key * nu
    if k.shape != q.shape or v.shape != (B, H, L, d_v) or beta.shape != (B, H, L):
        raise ValueError("shape mismatch among q, k, v, beta")
    if not (q.dtype == k.dtype == v.dtype == beta.dtype):
        raise ValueError("q, k, v, beta must share the I/O dtype")
    if W0 is not None:
        _dev(W0, "W0")
        if W0.dtype != torch.float32 or W0.shape != (B, H, d_v, d_dot):
            raise ValueError("W0 must be fp32 [B,H,d_v,d_dot]")
    if y is None:
        y = torch.empty(B, H, L, d_v, dtype=q.dtype, device=q.device)
    if W_final is None and return_state:
        W_final = torch.empty(B, H, d_v, d_dot, dtype=torch.float32, device=q.device)
    code = _dtype_code(q.dtype)
    need = fw_delta_forward_workspace_size(B, H, L, d_key, nu, d_v, chunk, code)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().fw_delta_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(W0), _ptr(W_final),
                                 _ptr(y), _ptr(workspace), ws_bytes, B, H, L, d_key, nu, d_v, chunk,
                                 code, eps, _stream(stream))
    _check(rc, "fw_delta_forward")
    return y, W_final


def fw_delta_forward_prepare(q, k, v, beta, workspace, nu: int = 1, chunk: int = 64,
                             eps: float = 1e-6, stream=None):
    """Phase 1 of the bf16 forward: every chunk's preparation into `workspace`
    (a uint8 CUDA tensor of fw_delta_forward_workspace_size bytes)."""
    for name, t in (("q", q), ("k", k), ("v", v), ("beta", beta), ("workspace", workspace)):
        _dev(t, name)
    B, H, L, d_key = q.shape
    d_v = v.shape[-1]
    rc = load().fw_delta_forward_prepare(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(workspace),
                                         workspace.numel() * workspace.element_size(), B, H, L, d_key,
                                         nu, d_v, chunk, eps, _stream(stream))
    _check(rc, "fw_delta_forward_prepare")


def fw_delta_forward_scan(workspace, y, W0=None, W_final=None, nu: int = 1, chunk: int = 64,
                          stream=None):
    """Phase 2 of the bf16 forward: the chunk-by-chunk state scan from the
    prepared `workspace`; writes y [B,H,L,d_v] and W_final (if given)."""
    _dev(workspace, "workspace")
    _dev(y, "y")
    B, H, L, d_v = y.shape
    if W0 is not None:
        _dev(W0, "W0")
    d_dot = (W0 if W0 is not None else W_final).shape[-1] if (W0 is not None or W_final is not None) else None
    if d_dot is None:
        raise ValueError("pass W0 or W_final so the state width is known")
    d_key = d_dot // (2 * nu)
    rc = load().fw_delta_forward_scan(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                      _ptr(W0), _ptr(W_final), _ptr(y), B, H, L, d_key, nu, d_v, chunk,
                                      _stream(stream))
    _check(rc, "fw_delta_forward_scan")
    return y, W_final


def fw_delta_forward_projected_workspace_size(B, L, d_model, H, d_key, nu, d_v, chunk) -> int:
    return int(load().fw_delta_forward_projected_workspace_size(B, L, d_model, H, d_key, nu, d_v, chunk))


def fw_delta_forward_projected(x, W_all, H: int, d_key: int, d_v: int, nu: int = 1, chunk: int = 64,
                               W0=None, eps: float = 1e-6, return_state: bool = True, y=None, W_final=None,
                               workspace=None, stream=None):
    """The layer core from x [B,L,d_model] (bf16) and W_all = [W_q | W_k | W_v |
    W_beta] ([d_model, ldw] bf16, ldw a multiple of 8).  Returns (y, W_final or None)."""
    _dev(x, "x")
    _dev(W_all, "W_all")
    B, L, d_model = x.shape
    ldw = W_all.shape[1]
    d_dot = 2 * d_key * nu
    if W_all.shape[0] != d_model or x.dtype != torch.bfloat16 or W_all.dtype != torch.bfloat16:
        raise ValueError("x [B,L,d_model] and W_all [d_model, ldw] must be bf16 and agree on d_model")
    if W0 is not None:
        _dev(W0, "W0")
    if y is None:
        y = torch.empty(B, H, L, d_v, dtype=torch.bfloat16, device=x.device)
    if W_final is None and return_state:
        W_final = torch.empty(B, H, d_v, d_dot, dtype=torch.float32, device=x.device)
    need = fw_delta_forward_projected_workspace_size(B, L, d_model, H, d_key, nu, d_v, chunk)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().fw_delta_forward_projected(_ptr(x), _ptr(W_all), ldw, _ptr(W0), _ptr(W_final), _ptr(y),
                                           _ptr(workspace), ws_bytes, B, L, d_model, H, d_key, nu, d_v, chunk,
                                           eps, _stream(stream))
    _check(rc, "fw_delta_forward_projected")
    return y, W_final


def fw_decode_stack_workspace_size(B, H, d_key, d_v, d_model, d_ff) -> int:
    return int(load().fw_decode_stack_workspace_size(B, H, d_key, d_v, d_model, d_ff))


def fw_decode_stack_step(x, layers, H: int, d_key: int, d_v: int, nu: int = 1, ln_gamma=None, ln_beta=None,
                         eps: float = 1e-6, ln_eps: float = 1e-5, out=None, workspace=None, stream=None):
    """One token of B sequences through the layer stack.  x: [B, d_model] fp32;
    layers: sequence of dicts keyed by STACK_FIELDS (W_in [d_model, ldw] and
    W_o, W_1, W_2 bf16 [in, out]; b_o, b_1, b_2, ln_gamma, ln_beta fp32 or
    None; W fp32 [B, H, d_v, d_dot], updated in place).  Returns out [B, d_model]
    fp32, the final norm of the last layer's output."""
    _dev(x, "x")
    if x.dtype != torch.float32 or x.dim() != 2:
        raise ValueError("x must be fp32 [B, d_model]")
    B, d_model = x.shape
    d_dot = 2 * d_key * nu
    arr = (FwStackLayer * max(1, len(layers)))()
    ldw_in, d_ff = 0, 64
    for i, ly in enumerate(layers):
        for n in ("W_in", "W_o", "W_1", "W_2"):
            _dev(ly[n], n)
            if ly[n].dtype != torch.bfloat16:
                raise ValueError(f"{n} must be bf16")
        for n in ("b_o", "ln_gamma", "ln_beta", "b_1", "b_2"):
            if ly.get(n) is not None:
                _dev(ly[n], n)
                if ly[n].dtype != torch.float32:
                    raise ValueError(f"{n} must be fp32")
        _dev(ly["W"], "W")
        if ly["W"].dtype != torch.float32 or tuple(ly["W"].shape) != (B, H, d_v, d_dot):
            raise ValueError("W must be fp32 [B, H, d_v, d_dot]")
        if i == 0:
            ldw_in, d_ff = ly["W_in"].shape[1], ly["W_1"].shape[1]
        if (tuple(ly["W_in"].shape) != (d_model, ldw_in) or tuple(ly["W_o"].shape) != (H * d_v, d_model) or
                tuple(ly["W_1"].shape) != (d_model, d_ff) or tuple(ly["W_2"].shape) != (d_ff, d_model)):
            raise ValueError(f"layer {i}: weight shapes disagree")
        for n in STACK_FIELDS:
            setattr(arr[i], n, None if ly.get(n) is None else ly[n].data_ptr())
    for name, t in (("ln_gamma", ln_gamma), ("ln_beta", ln_beta)):
        if t is not None:
            _dev(t, name)
    if out is None:
        out = torch.empty(B, d_model, dtype=torch.float32, device=x.device)
    need = fw_decode_stack_workspace_size(B, H, d_key, d_v, d_model, d_ff)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().fw_decode_stack_step(arr, len(layers), _ptr(x), _ptr(ln_gamma), _ptr(ln_beta), _ptr(out),
                                     _ptr(workspace), ws_bytes, B, H, d_key, nu, d_v, d_model, d_ff, ldw_in, eps,
                                     ln_eps, _stream(stream))
    _check(rc, "fw_decode_stack_step")
    return out


def fw_delta_backward_workspace_size(B, H, L, d_key, nu, d_v, io_dtype) -> int:
    code = io_dtype if isinstance(io_dtype, int) else _dtype_code(io_dtype)
    return int(load().fw_delta_backward_workspace_size(B, H, L, d_key, nu, d_v, code))


def fw_delta_backward(q, k, v, beta, dy, W0=None, dW_final=None, nu: int = 1, eps: float = 1e-6,
                      return_dW0: bool = True, workspace=None, stream=None):
    """Gradients of the delta-rule forward: given dy [B,H,L,d_v] (and dW_final),
    returns (dq, dk, dv, dbeta, dW0 or None)."""
    for name, t in (("q", q), ("k", k), ("v", v), ("beta", beta), ("dy", dy)):
        _dev(t, name)
    B, H, L, d_key = q.shape
    d_v = v.shape[-1]
    d_dot = 2 * d_key * nu
    if k.shape != q.shape or v.shape != (B, H, L, d_v) or beta.shape != (B, H, L) or dy.shape != v.shape:
        raise ValueError("shape mismatch among q, k, v, beta, dy")
    if not (q.dtype == k.dtype == v.dtype == beta.dtype == dy.dtype):
        raise ValueError("q, k, v, beta, dy must share the I/O dtype")
    for name, t in (("W0", W0), ("dW_final", dW_final)):
        if t is not None:
            _dev(t, name)
            if t.dtype != torch.float32 or tuple(t.shape) != (B, H, d_v, d_dot):
                raise ValueError(f"{name} must be fp32 [B,H,d_v,d_dot]")
    dq, dk, dv, dbeta = (torch.empty_like(t) for t in (q, k, v, beta))
    dW0 = torch.empty(B, H, d_v, d_dot, dtype=torch.float32, device=q.device) if return_dW0 else None
    code = _dtype_code(q.dtype)
    need = fw_delta_backward_workspace_size(B, H, L, d_key, nu, d_v, code)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().fw_delta_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(W0), _ptr(dy), _ptr(dW_final),
                                  _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dbeta), _ptr(dW0), _ptr(workspace), ws_bytes,
                                  B, H, L, d_key, nu, d_v, code, eps, _stream(stream))
    _check(rc, "fw_delta_backward")
    return dq, dk, dv, dbeta, dW0


def fw_linear_forward_workspace_size(B, H, L, d_key, nu, d_v, chunk, normalize=True,
                                     io_dtype=torch.bfloat16) -> int:
    code = io_dtype if isinstance(io_dtype, int) else _dtype_code(io_dtype)
    return int(load().fw_linear_forward_workspace_size(B, H, L, d_key, nu, d_v, chunk, int(bool(normalize)),
                                                       code))


def fw_linear_forward(q, k, v, W0=None, z0=None, nu: int = 1, normalize: bool = True, chunk: int = 64,
                      eps: float = 1e-6, return_state: bool = True, y=None, W_final=None, z_final=None,
                      workspace=None, stream=None):
    """The sum rule (linear attention) over [B,H,L,*] bf16 inputs.
    Returns (y, W_final or None, z_final or None)."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        _dev(t, name)
    B, H, L, d_key = q.shape
    d_v = v.shape[-1]
    d_dot = 2 * d_key * nu
    if k.shape != q.shape or v.shape != (B, H, L, d_v):
        raise ValueError("shape mismatch among q, k, v")
    if not (q.dtype == k.dtype == v.dtype):
        raise ValueError("q, k, v must share the I/O dtype")
    for name, t, shape in (("W0", W0, (B, H, d_v, d_dot)), ("z0", z0, (B, H, d_dot))):
        if t is not None:
            _dev(t, name)
            if t.dtype != torch.float32 or tuple(t.shape) != shape:
                raise ValueError(f"{name} must be fp32 {list(shape)}")
    if y is None:
        y = torch.empty(B, H, L, d_v, dtype=q.dtype, device=q.device)
    if W_final is None and return_state:
        W_final = torch.empty(B, H, d_v, d_dot, dtype=torch.float32, device=q.device)
    if z_final is None and return_state and normalize:
        z_final = torch.empty(B, H, d_dot, dtype=torch.float32, device=q.device)
    code = _dtype_code(q.dtype)
    need = fw_linear_forward_workspace_size(B, H, L, d_key, nu, d_v, chunk, normalize, code)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().fw_linear_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(W0), _ptr(z0), _ptr(W_final), _ptr(z_final),
                                  _ptr(y), _ptr(workspace), ws_bytes, B, H, L, d_key, nu, d_v, chunk,
                                  int(bool(normalize)), code, eps, _stream(stream))
    _check(rc, "fw_linear_forward")
    return y, W_final, z_final


def fw_delta_forward_noalloc(q, k, v, beta, W0=None, nu: int = 1, chunk: int = 64,
                             eps: float = 1e-6, return_state: bool = True, y=None, W_final=None,
                             stream=None):
    """fw_delta_forward without a caller-provided workspace: the library uses
    its own fixed scratch array (NOALLOC_SCRATCH_BYTES per GPU) and allocates
    nothing.  For callers that cannot allocate device memory when they call
    the forward.  Outputs passed in as y / W_final are used as they are;
    missing ones are created here with PyTorch before the call."""
    for name, t in (("q", q), ("k", k), ("v", v), ("beta", beta)):
        _dev(t, name)
    B, H, L, d_key = q.shape
    d_v = v.shape[-1]
    d_dot = 2 * d_key * nu
    if k.shape != q.shape or v.shape != (B, H, L, d_v) or beta.shape != (B, H, L):
        raise ValueError("shape mismatch among q, k, v, beta")
    if W0 is not None:
        _dev(W0, "W0")
        if W0.dtype != torch.float32 or W0.shape != (B, H, d_v, d_dot):
            raise ValueError("W0 must be fp32 [B,H,d_v,d_dot]")
    if y is None:
        y = torch.empty(B, H, L, d_v, dtype=q.dtype, device=q.device)
    if W_final is None and return_state:
        W_final = torch.empty(B, H, d_v, d_dot, dtype=torch.float32, device=q.device)
    rc = load().fw_delta_forward_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(W0),
                                         _ptr(W_final), _ptr(y), B, H, L, d_key, nu, d_v, chunk,
                                         _dtype_code(q.dtype), eps, _stream(stream))
    _check(rc, "fw_delta_forward_noalloc")
    return y, W_final


def fw_delta_decode_step(q, k, v, beta, W, nu: int = 1, eps: float = 1e-6, y=None, stream=None):
    """One token per (b,h): q, k [B,H,d_key]; v [B,H,d_v]; beta [B,H]; W fp32
    [B,H,d_v,d_dot] updated in place.  Returns y [B,H,d_v]."""
    for name, t in (("q", q), ("k", k), ("v", v), ("beta", beta), ("W", W)):
        _dev(t, name)
    B, H, d_key = q.shape
    d_v = v.shape[-1]
    if W.dtype != torch.float32 or W.shape != (B, H, d_v, 2 * d_key * nu):
        raise ValueError("W must be fp32 [B,H,d_v,d_dot]")
    if y is None:
        y = torch.empty(B, H, d_v, dtype=q.dtype, device=q.device)
    rc = load().fw_delta_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(W), _ptr(y), B, H,
                                     d_key, nu, d_v, _dtype_code(q.dtype), eps, _stream(stream))
    _check(rc, "fw_delta_decode_step")
    return y


def fw_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status code."""
    return int(load().fw_device_status(_stream(stream)))


def fw_selftest_umma(A, B, a_mn: int = 0, b_mn: int = 0, swap_mn: int = 0, stream=None):
    """D = A B^T through one tcgen05 MMA chain (A [128,K], B [N,K] fp32 CUDA
    tensors holding bf16-representable values).  Returns D [128,N] fp32."""
    _dev(A, "A")
    _dev(B, "B")
    K = A.shape[1]
    N = B.shape[0]
    D = torch.empty(128, N, dtype=torch.float32, device=A.device)
    rc = load().fw_selftest_umma(_ptr(A), _ptr(B), _ptr(D), N, K, a_mn, b_mn, swap_mn, _stream(stream))
    _check(rc, "fw_selftest_umma")
    return D


def fw_selftest_wait_timeout(limit_us: int = 2000, stream=None):
    """Run the bounded-wait failure path once (see include/fastweight_selftest.h)."""
    _check(load().fw_selftest_wait_timeout(int(limit_us), _stream(stream)), "fw_selftest_wait_timeout")


def fw_selftest_flag_timeout(limit_us: int = 2000, stream=None):
    """Run the ready-flag wait's failure path once (see include/fastweight_selftest.h)."""
    _check(load().fw_selftest_flag_timeout(int(limit_us), _stream(stream)), "fw_selftest_flag_timeout")
