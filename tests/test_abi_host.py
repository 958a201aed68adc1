"""The C-ABI library on the host (no GPU needed): it builds, loads, exports
every symbol include/fastweight.h declares, and rejects bad arguments before
touching CUDA."""
import ctypes
import glob
import os
import re

import pytest

from delta_rule_linear_dpfp_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))

# a non-null, 16-byte aligned address that is never dereferenced: every call
# below fails its host-side checks before any CUDA call
FAKE = ctypes.c_void_p(0x10000)
MISALIGNED = ctypes.c_void_p(0x10008)


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def declared_symbols():
    names = set()
    for h in HEADERS:
        names |= set(re.findall(r"FW_API[^;(]*?\b(fw_\w+)\s*\(", open(h).read()))
    return sorted(names)


def test_header_declares_the_binding_exports():
    assert declared_symbols() == sorted(binding.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def _prototypes():
    """name -> parameter count of every FW_API function in include/*.h."""
    protos = {}
    for h in HEADERS:
        text = open(h).read()
        for m in re.finditer(r"FW_API[^;(]*?\b(fw_\w+)\s*\(([^)]*)\)", text):
            params = [p for p in m.group(2).split(",") if p.strip() and p.strip() != "void"]
            protos[m.group(1)] = len(params)
    return protos


def test_binding_signatures_match_the_headers(lib):
    for name, n in _prototypes().items():
        assert len(getattr(lib, name).argtypes) == n, name


def test_status_strings(lib):
    for code in range(5):
        assert binding.status_string(code).startswith("FW_")
    assert binding.status_string(99) == "unknown fw_status"


def test_dpfp_argument_checks(lib):
    E, U, OK = binding.FW_ERR_INVALID_ARG, binding.FW_ERR_UNSUPPORTED, binding.FW_OK
    call = lib.fw_dpfp
    assert call(None, FAKE, 4, 64, 1, 0, 0, 1e-6, None) == E
    assert call(FAKE, None, 4, 64, 1, 0, 0, 1e-6, None) == E
    assert call(MISALIGNED, FAKE, 4, 64, 1, 0, 0, 1e-6, None) == E
    assert call(FAKE, FAKE, -1, 64, 1, 0, 0, 1e-6, None) == E
    assert call(FAKE, FAKE, 4, 64, 0, 0, 0, 1e-6, None) == E
    assert call(FAKE, FAKE, 4, 64, 128, 0, 0, 1e-6, None) == E      # nu > 2*d_key-1
    assert call(FAKE, FAKE, 4, 64, 1, 7, 0, 1e-6, None) == E        # unknown dtype
    assert call(FAKE, FAKE, 4, 64, 1, 0, 0, -1.0, None) == E        # eps < 0
    assert call(FAKE, FAKE, 4, 64, 1, 0, 0, float("nan"), None) == E
    assert call(FAKE, FAKE, 4, 12, 1, 0, 0, 1e-6, None) == U        # d_key not compiled
    assert call(FAKE, FAKE, 0, 64, 1, 0, 0, 1e-6, None) == OK       # empty: nothing enqueued
    assert call(None, None, 0, 64, 1, 0, 0, 1e-6, None) == OK       # empty tensors may be NULL


def _fwd(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, beta=FAKE, W0=None, Wf=None, y=FAKE, ws=None, wsb=0, B=2, H=2,
             L=8, d_key=64, nu=1, d_v=64, chunk=64, io=1, eps=1e-6)
    a.update(kw)
    return lib.fw_delta_forward(a["q"], a["k"], a["v"], a["beta"], a["W0"], a["Wf"], a["y"],
                                a["ws"], a["wsb"], a["B"], a["H"], a["L"], a["d_key"], a["nu"],
                                a["d_v"], a["chunk"], a["io"], a["eps"], None)


def test_forward_argument_checks(lib):
    E, U, OK = binding.FW_ERR_INVALID_ARG, binding.FW_ERR_UNSUPPORTED, binding.FW_OK
    for name in ("q", "k", "v", "beta", "y"):
        assert _fwd(lib, **{name: None}) == E, name
        assert _fwd(lib, **{name: MISALIGNED}) == E, name
    assert _fwd(lib, W0=MISALIGNED) == E
    assert _fwd(lib, Wf=MISALIGNED) == E
    assert _fwd(lib, B=-1) == E
    assert _fwd(lib, d_v=0) == E
    assert _fwd(lib, nu=0) == E
    assert _fwd(lib, chunk=48) == E
    assert _fwd(lib, io=3) == E
    assert _fwd(lib, eps=-1e-6) == E
    assert _fwd(lib, d_key=24) == U
    assert _fwd(lib, d_key=128, nu=2) == U           # bf16: padded d_dot 512 > 384
    assert _fwd(lib, d_key=64, nu=3, d_v=256) == U   # bf16: d_v outside {16, 32, 64, 128}
    assert _fwd(lib, d_key=128, nu=5, io=0) == U     # fp32: d_dot 1280 > 1024
    need = lib.fw_delta_forward_workspace_size(2, 2, 8, 64, 1, 64, 64, 1)
    if need > 0:
        assert _fwd(lib, ws=None, wsb=0) == E
        assert _fwd(lib, ws=FAKE, wsb=need - 1) == E
    # empty batch: nothing to do, nothing enqueued, NULL pointers allowed
    assert _fwd(lib, B=0, ws=FAKE, wsb=1 << 40) == OK
    assert _fwd(lib, B=0, q=None, k=None, v=None, beta=None, y=None) == OK


def test_forward_workspace_query(lib):
    ws = lib.fw_delta_forward_workspace_size
    assert ws(2, 2, 8, 64, 1, 64, 64, 0) == 0          # fp32 path needs none
    assert ws(2, 2, 8, 64, 1, 64, 48, 1) == 0          # rejected chunk -> 0
    assert ws(2, 2, 8, 24, 1, 64, 64, 1) == 0          # unsupported d_key -> 0
    a = ws(2, 8, 2048, 64, 3, 64, 64, 1)
    b = ws(4, 8, 2048, 64, 3, 64, 64, 1)
    assert b >= a


def test_decode_argument_checks(lib):
    E, U = binding.FW_ERR_INVALID_ARG, binding.FW_ERR_UNSUPPORTED
    call = lib.fw_delta_decode_step
    base = [FAKE] * 6 + [4, 2, 64, 2, 128, 1, 1e-6, None]
    for i in range(6):
        args = list(base)
        args[i] = None
        assert call(*args) == E
        args[i] = MISALIGNED
        assert call(*args) == E
    args = list(base)
    args[9] = 0                                        # nu = 0
    assert call(*args) == E
    args = list(base)
    args[8] = 20                                       # d_key not compiled
    assert call(*args) == U
    args = list(base)
    args[8], args[9] = 128, 5                          # d_dot = 1280 > 1024
    assert call(*args) == U


def test_phase_argument_checks(lib):
    E, U, OK = binding.FW_ERR_INVALID_ARG, binding.FW_ERR_UNSUPPORTED, binding.FW_OK
    prep, scan = lib.fw_delta_forward_prepare, lib.fw_delta_forward_scan
    need = lib.fw_delta_forward_workspace_size(2, 2, 8, 64, 1, 64, 64, 1)
    assert need > 0
    args = [FAKE] * 5 + [need, 2, 2, 8, 64, 1, 64, 64, 1e-6, None]
    for i in range(5):                   # q, k, v, beta, workspace
        bad = list(args)
        bad[i] = None
        assert prep(*bad) == E
        bad[i] = MISALIGNED
        assert prep(*bad) == E
    bad = list(args)
    bad[5] = need - 1                    # workspace too small
    assert prep(*bad) == E
    bad = list(args)
    bad[9] = 24                          # d_key not compiled
    assert prep(*bad) == U
    bad = list(args)
    bad[12] = 48                         # chunk
    assert prep(*bad) == E
    sargs = [FAKE, need, None, None, FAKE, 2, 2, 8, 64, 1, 64, 64, None]
    bad = list(sargs)
    bad[0] = None
    assert scan(*bad) == E
    bad = list(sargs)
    bad[4] = None                        # y
    assert scan(*bad) == E
    bad = list(sargs)
    bad[2] = MISALIGNED                  # W0
    assert scan(*bad) == E
    bad = list(sargs)
    bad[5] = 0                           # empty batch: nothing to do
    assert scan(*bad) == OK


def test_linear_argument_checks(lib):
    E, U, OK = binding.FW_ERR_INVALID_ARG, binding.FW_ERR_UNSUPPORTED, binding.FW_OK
    f, ws = lib.fw_linear_forward, lib.fw_linear_forward_workspace_size
    need = ws(2, 2, 8, 64, 1, 64, 64, 1, 1)
    assert need > 0
    assert ws(2, 2, 8, 64, 1, 64, 64, 1, 0) == 0            # fp32 I/O is not compiled
    assert ws(2, 2, 8, 64, 1, 64, 64, 2, 1) == 0            # normalize must be 0 or 1
    assert ws(2, 2, 8, 64, 1, 64, 64, 0, 1) < need          # no normaliser block
    base = [FAKE] * 9 + [need, 2, 2, 8, 64, 1, 64, 64, 1, 1, 1e-6, None]

    def call(**kw):
        a = list(base)
        names = ["q", "k", "v", "W0", "z0", "Wf", "zf", "y", "ws", "wsb", "B", "H", "L", "d_key", "nu",
                 "d_v", "chunk", "normalize", "io", "eps", "stream"]
        for key, val in kw.items():
            a[names.index(key)] = val
        return f(*a)

    for name in ("q", "k", "v", "y", "ws"):
        assert call(**{name: None}) == E
        assert call(**{name: MISALIGNED}) == E
    for name in ("W0", "z0", "Wf", "zf"):
        assert call(**{name: MISALIGNED}) == E
    assert call(wsb=need - 1) == E
    assert call(normalize=3) == E
    assert call(io=0) == U
    assert call(d_key=24) == U
    assert call(d_key=128, nu=2) == U                       # padded d_dot 512 > 384
    assert call(nu=0) == E
    assert call(chunk=48) == E
    assert call(eps=-1.0) == E
    assert call(B=0, q=None, k=None, v=None, y=None, ws=None) == OK


def _stack(lib, layers=None, n=1, **kw):
    a = dict(x=FAKE, g=None, b=None, out=FAKE, ws=FAKE, wsb=1 << 30, B=4, H=2, d_key=16, nu=1, d_v=32, d_model=128,
             d_ff=128, ldw=136, eps=1e-6, ln_eps=1e-5)
    a.update(kw)
    if layers is None:
        ly = binding.FwStackLayer(*([0x10000] * len(binding.STACK_FIELDS)))
        layers = (binding.FwStackLayer * 1)(ly)
    return lib.fw_decode_stack_step(layers, n, a["x"], a["g"], a["b"], a["out"], a["ws"], a["wsb"], a["B"], a["H"],
                                    a["d_key"], a["nu"], a["d_v"], a["d_model"], a["d_ff"], a["ldw"], a["eps"],
                                    a["ln_eps"], None)


def test_stack_argument_checks(lib):
    E, U, OK = binding.FW_ERR_INVALID_ARG, binding.FW_ERR_UNSUPPORTED, binding.FW_OK
    ws = lib.fw_decode_stack_workspace_size
    assert ws(4, 2, 16, 32, 128, 128) > 0
    assert ws(4, 2, 16, 32, 96, 128) == 0          # d_model not a multiple of 128
    assert ws(4, 2, 16, 32, 2048, 128) == 0        # d_model above 1024
    assert ws(4, 2, 16, 24, 128, 128) == 0         # H d_v not a multiple of 64
    assert ws(4, 2, 12, 32, 128, 128) == 0         # d_key not compiled
    assert _stack(lib, x=None) == E
    assert _stack(lib, out=MISALIGNED) == E
    assert _stack(lib, ws=None) == E
    assert _stack(lib, wsb=16) == E                # workspace too small
    assert _stack(lib, ldw=100) == E               # N = 2 (2 16 + 32 + 1) = 130 > 100
    assert _stack(lib, ldw=140) == E               # not a multiple of 8
    assert _stack(lib, eps=-1.0) == E
    assert _stack(lib, ln_eps=float("nan")) == E
    assert _stack(lib, n=-1) == E
    assert _stack(lib, d_model=96) == U
    assert _stack(lib, d_ff=100) == U
    assert _stack(lib, nu=32) == E                 # nu > 2 d_key - 1
    assert _stack(lib, d_key=64, nu=9) == U        # d_dot 1152 > 1024
    bad = binding.FwStackLayer(*([0x10000] * len(binding.STACK_FIELDS)))
    bad.W = None                                    # the layer's fast weights missing
    assert _stack(lib, layers=(binding.FwStackLayer * 1)(bad)) == E
    bad.W, bad.b_o = 0x10000, 0x10004               # a misaligned bias
    assert _stack(lib, layers=(binding.FwStackLayer * 1)(bad)) == E
    assert _stack(lib, B=0, x=None, out=None, ws=None, wsb=0) == OK   # empty: nothing enqueued


def test_backward_workspace_limits(lib):
    ws = lib.fw_delta_backward_workspace_size
    assert ws(2, 2, 16, 64, 1, 64, 1) > 0
    assert ws(2, 2, 16, 128, 4, 200, 1) > 0       # d_dot 1024, d_v not a multiple of the row block
    assert ws(2, 2, 16, 128, 5, 64, 1) == 0       # d_dot 1280 > 1024
    assert ws(2, 2, 16, 12, 1, 64, 1) == 0        # d_key not compiled
    assert ws(65536, 65536, 1, 64, 1, 64, 1) == 0  # B H past 2^30 (and past int): rejected, not wrapped


def _chunked_ws(BH, L, d_dot, d_v):
    # phi(k), phi(q), the per-token records, then per chunk M, T, P, K K^T (64 x 64 each) and G, S, dS'
    # (d_v x d_dot each), then X, U, dX, dU per token (fp32 throughout)
    rows, nC = BH * L, -(-L // 64)
    return 4 * (2 * rows * d_dot + rows * (2 * d_dot + 4) + 4 * BH * nC * 64 * 64 + 3 * BH * nC * d_v * d_dot
                + 4 * rows * d_v)


def _serial_ws(BH, L, d_dot, d_v):
    # u_t per token, phi(k), phi(q), then each block of 16 rows' per-token records
    rows = BH * L
    return 4 * (rows * d_v + 2 * rows * d_dot + -(-d_v // 16) * rows * (2 * d_dot + 4))


def test_backward_path_choice_by_workspace(lib):
    """The backward takes the chunk-parallel path for d_dot <= 512, d_v <= 128
    and at most 65535 chunks of 64 tokens, the token-serial one past that;
    the workspace size says which."""
    ws = lib.fw_delta_backward_workspace_size
    assert ws(4, 8, 512, 64, 1, 64, 1) == _chunked_ws(32, 512, 128, 64) == 92_536_832   # the bench shape
    assert ws(1, 2, 30, 64, 4, 128, 0) == _chunked_ws(2, 30, 512, 128)                  # both limits met
    assert ws(1, 1, 70, 128, 3, 32, 0) == _serial_ws(1, 70, 768, 32)                    # d_dot 768
    assert ws(1, 2, 25, 16, 1, 129, 0) == _serial_ws(2, 25, 32, 129)                    # d_v 129
    L = 64 * 65535
    assert ws(1, 1, L, 8, 1, 16, 1) == _chunked_ws(1, L, 16, 16)
    assert ws(1, 1, L + 1, 8, 1, 16, 1) == _serial_ws(1, L + 1, 16, 16)                 # 65536 chunks


def test_size_queries_at_integer_limits(lib):
    """Sequence lengths whose chunk count would wrap in int, and key widths
    whose 2 d_key would, are refused by the size queries (0), not computed."""
    big = 2**31 - 1
    assert lib.fw_delta_forward_workspace_size(1, 1, big, 64, 1, 64, 64, 1) == 0
    assert lib.fw_delta_backward_workspace_size(1, 1, big, 64, 1, 64, 1) == 0
    assert lib.fw_linear_forward_workspace_size(1, 1, big, 64, 1, 64, 64, 1, 1) == 0
    assert lib.fw_delta_backward_workspace_size(1, 1, 16, big, 3, 64, 1) == 0
    assert lib.fw_delta_forward_workspace_size(1, 1, 2**31 - 65, 64, 1, 64, 64, 1) > 0   # the longest L taken
