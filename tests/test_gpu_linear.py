"""GPU parity of the sum rule (linear attention with the DPFP kernel,
fw_linear_forward) against the fp64 oracle on the same seeded inputs, through
the C ABI.  Tolerance: max normwise relative error 2e-2 (bf16 I/O, fp32
state); state shapes and layouts exact."""
import numpy as np
import pytest
import torch

import oracle
from delta_rule_linear_dpfp_gb300 import binding as fw
from delta_rule_linear_dpfp_gb300 import build, inputs
from tests.parity_util import TOL_BF16, f64, maxrel, to_dev

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


def _check(d, nu, normalize, chunk=64, zero_query=None):
    dd = to_dev(d)
    if zero_query is not None:
        b, h, t = zero_query
        d["q"][b, h, t] = 0
        dd["q"][b, h, t] = 0
    y, Wf, zf = fw.fw_linear_forward(dd["q"], dd["k"], dd["v"], W0=dd["W0"], z0=dd["z0"], nu=nu,
                                     normalize=normalize, chunk=chunk)
    torch.cuda.synchronize()
    yo, Wo, zo = oracle.linear_forward(f64(d["q"]), f64(d["k"]), f64(d["v"]),
                                       None if d["W0"] is None else f64(d["W0"]),
                                       None if d["z0"] is None else f64(d["z0"]), nu, normalize, 1e-6, NT)
    assert tuple(y.shape) == yo.shape and tuple(Wf.shape) == Wo.shape
    ey, ew = maxrel(f64(y), yo), maxrel(f64(Wf), Wo)
    assert ey <= TOL_BF16 and ew <= TOL_BF16, (ey, ew)
    if normalize:
        assert tuple(zf.shape) == zo.shape
        assert maxrel(f64(zf), zo) <= TOL_BF16
    else:
        assert zf is None
    return f64(y), yo


# B, H, L, d_key, nu, d_v, chunk: several chunks, ragged tails, every compiled d_v,
# the largest state that fits with the normaliser block
CASES = [
    (2, 4, 200, 64, 1, 64, 64),
    (1, 3, 130, 32, 3, 128, 64),
    (2, 2, 70, 16, 2, 16, 32),
    (1, 2, 64, 128, 1, 32, 64),
    (1, 2, 97, 64, 3, 64, 16),
    (1, 1, 50, 8, 15, 16, 64),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "b{}h{}l{}dk{}nu{}dv{}c{}".format(*c))
@pytest.mark.parametrize("normalize", [True, False])
@pytest.mark.parametrize("with_state", [False, True])
def test_linear_parity(case, normalize, with_state):
    B, H, L, d_key, nu, d_v, chunk = case
    d = inputs.linear_inputs(B, H, L, d_key, nu, d_v, with_state=with_state, seed=sum(case))
    _check(d, nu, normalize, chunk)


def test_linear_zero_denominator():
    # q = 0 -> phi(q) = 0: the normalised output is exactly 0 there (no NaN)
    d = inputs.linear_inputs(1, 2, 100, 64, 1, 64, seed=3)
    y, yo = _check(d, 1, True, zero_query=(0, 1, 70))
    assert np.all(y[0, 1, 70] == 0.0) and np.all(yo[0, 1, 70] == 0.0)
    assert np.all(np.isfinite(y))


def test_linear_first_output_is_v():
    # normalised from a zero state with q_1 = k_1: y_1 = v_1 (bf16 rounding of phi aside)
    d = inputs.linear_inputs(2, 2, 64, 64, 1, 32, seed=4)
    d["q"][:, :, 0] = d["k"][:, :, 0]
    dd = to_dev(d)
    y, _, _ = fw.fw_linear_forward(dd["q"], dd["k"], dd["v"], nu=1, normalize=True)
    assert maxrel(f64(y[:, :, 0]), f64(d["v"][:, :, 0])) <= TOL_BF16


def test_linear_empty_sequence_returns_initial_state():
    d = inputs.linear_inputs(2, 2, 0, 64, 1, 64, with_state=True, seed=5)
    dd = to_dev(d)
    y, Wf, zf = fw.fw_linear_forward(dd["q"], dd["k"], dd["v"], W0=dd["W0"], z0=dd["z0"], nu=1, normalize=True)
    torch.cuda.synchronize()
    assert y.numel() == 0
    assert torch.equal(Wf.cpu(), d["W0"]) and torch.equal(zf.cpu(), d["z0"])


def test_linear_chunk_invariance():
    # the chunk length only tiles the work: results agree to rounding
    d = to_dev(inputs.linear_inputs(1, 4, 192, 64, 1, 64, with_state=True, seed=6))
    outs = [fw.fw_linear_forward(d["q"], d["k"], d["v"], W0=d["W0"], z0=d["z0"], nu=1, normalize=True,
                                 chunk=c)[0] for c in (16, 32, 64)]
    for o in outs[1:]:
        assert maxrel(f64(o), f64(outs[0])) <= TOL_BF16


@pytest.mark.parametrize("normalize", [True, False])
def test_linear_bench_shapes(normalize):
    # the bench row's shapes: B4 H8 L512 d_key 64 nu 1 d_v 64, bf16, from zero state
    _check(inputs.linear_inputs(4, 8, 512, 64, 1, 64, seed=0), 1, normalize)
