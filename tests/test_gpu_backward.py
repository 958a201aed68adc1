"""GPU parity of the delta-rule backward (fw_delta_backward) against the fp64
oracle's backward (itself pinned to finite differences of the forward), on
the same seeded inputs, through the C ABI: the chunk-parallel form for
d_dot <= 512 and d_v <= 128, the token-serial kernel past that.
Tolerances: max normwise relative error per gradient tensor, 1e-4 for fp32
I/O and 2e-2 for bf16 I/O."""
import numpy as np
import pytest
import torch

import oracle
from delta_rule_linear_dpfp_gb300 import binding as fw
from delta_rule_linear_dpfp_gb300 import build, inputs
from tests.parity_util import f64, maxrel, to_dev, tol_for

pytestmark = pytest.mark.gpu

NT = oracle.default_threads()


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build.build()
    fw.load()
    yield
    assert fw.fw_device_status() == fw.FW_OK


def _grads(B, H, L, d_key, nu, d_v, io, with_state, seed):
    d = inputs.random_forward_inputs(B, H, L, d_key, nu, d_v, io, w0_var=0.01 if with_state else None, seed=seed)
    g = torch.Generator().manual_seed(seed + 1000)
    dt = inputs.torch_dtype(io)
    dy = torch.randn(B, H, L, d_v, generator=g).to(dt)
    dWf = torch.randn(B, H, d_v, 2 * d_key * nu, generator=g) if with_state else None
    dd = to_dev(d)
    got = fw.fw_delta_backward(dd["q"], dd["k"], dd["v"], dd["beta"], dy.cuda(), W0=dd["W0"],
                               dW_final=None if dWf is None else dWf.cuda(), nu=nu)
    torch.cuda.synchronize()
    want = oracle.delta_backward(f64(d["q"]), f64(d["k"]), f64(d["v"]), f64(d["beta"]), f64(dy),
                                 None if d["W0"] is None else f64(d["W0"]), None if dWf is None else f64(dWf),
                                 nu, 1e-6, NT)
    return got, want, dt


CASES = [  # B, H, L, d_key, nu, d_v
    (1, 2, 64, 16, 1, 16),
    (2, 2, 100, 64, 1, 64),
    (1, 2, 70, 32, 3, 32),
    (1, 1, 40, 64, 3, 64),
    (1, 1, 33, 128, 1, 16),
    (2, 1, 20, 8, 5, 128),
    (1, 3, 45, 32, 1, 40),      # row blocks of 16, 16 and 8
    (1, 2, 30, 64, 4, 128),     # d_dot 512 with d_v 128: 8 row blocks
    (1, 1, 70, 128, 3, 32),     # d_dot 768: past the chunked form's limit, token by token
    (1, 2, 25, 16, 1, 150),     # d_v 150: token by token, 10 row blocks, the last of 6 rows
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "b{}h{}l{}dk{}nu{}dv{}".format(*c))
@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("with_state", [False, True])
def test_backward_parity(case, io, with_state):
    got, want, dt = _grads(*case, io, with_state, seed=sum(case))
    names = ["dq", "dk", "dv", "dbeta", "dW0"]
    for name, a, b in zip(names, got, want):
        assert tuple(a.shape) == b.shape, name
        err = maxrel(f64(a), b)
        assert err <= tol_for(dt), (name, err)


def test_backward_empty_sequence():
    # no token: dL/dW0 = dL/dW_final
    d = to_dev(inputs.random_forward_inputs(2, 2, 0, 64, 1, 64, "bf16", w0_var=0.01, seed=1))
    dWf = torch.randn(2, 2, 64, 128, device="cuda")
    out = fw.fw_delta_backward(d["q"], d["k"], d["v"], d["beta"], torch.empty(2, 2, 0, 64, dtype=torch.bfloat16,
                                                                                 device="cuda"), W0=d["W0"],
                               dW_final=dWf, nu=1)
    torch.cuda.synchronize()
    assert torch.equal(out[4], dWf)


def test_backward_zero_beta():
    # beta = 0: the state never changes, so dv = 0 and dk = 0 exactly
    d = inputs.random_forward_inputs(1, 2, 50, 64, 1, 64, "f32", w0_var=0.01, seed=2)
    d["beta"].zero_()
    dd = to_dev(d)
    dy = torch.randn(1, 2, 50, 64, device="cuda")
    dq, dk, dv, db, dW0 = fw.fw_delta_backward(dd["q"], dd["k"], dd["v"], dd["beta"], dy, W0=dd["W0"], nu=1)
    assert torch.count_nonzero(dv) == 0 and torch.count_nonzero(dk) == 0
    assert torch.all(torch.isfinite(dq)) and torch.all(torch.isfinite(db))


def test_backward_deterministic():
    # fixed summation orders and no races: repeated calls give the same bits (bf16 and fp32 I/O)
    for io in ("bf16", "f32"):
        d = to_dev(inputs.random_forward_inputs(2, 4, 150, 64, 1, 64, io, w0_var=0.01, seed=11))
        dy = torch.randn(2, 4, 150, 64, generator=torch.Generator().manual_seed(3)).to(inputs.torch_dtype(io)).cuda()
        dWf = torch.randn(2, 4, 64, 128, generator=torch.Generator().manual_seed(4)).cuda()
        first = fw.fw_delta_backward(d["q"], d["k"], d["v"], d["beta"], dy, W0=d["W0"], dW_final=dWf, nu=1)
        for _ in range(4):
            again = fw.fw_delta_backward(d["q"], d["k"], d["v"], d["beta"], dy, W0=d["W0"], dW_final=dWf, nu=1)
            for a, b in zip(first, again):
                assert torch.equal(a, b)


def test_backward_bench_workload():
    # the bench row's shape and launch configuration: B4 H8 L512 d_key 64 nu 1 d_v 64, bf16, W0 = 0
    d = inputs.forward_inputs("b4h8_l512")
    dd = to_dev(d)
    dy = torch.randn(4, 8, 512, 64, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    got = fw.fw_delta_backward(dd["q"], dd["k"], dd["v"], dd["beta"], dy.cuda(), nu=1)
    torch.cuda.synchronize()
    want = oracle.delta_backward(f64(d["q"]), f64(d["k"]), f64(d["v"]), f64(d["beta"]), f64(dy), None, None, 1,
                                 1e-6, NT)
    for name, a, b in zip(["dq", "dk", "dv", "dbeta", "dW0"], got, want):
        err = maxrel(f64(a), b)
        assert err <= tol_for(torch.bfloat16), (name, err)
