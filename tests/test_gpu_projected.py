"""GPU parity of the forward from the token activations
(fw_delta_forward_projected: the tcgen05 projection prologue, then the
chunked forward) against the fp64 oracle (oracle.project, then the
sequential recurrence) on the same seeded bf16 x and weights, through the C
ABI.  Tolerance: max normwise relative error 2e-2 (bf16 I/O, fp32 state)."""
import pytest
import torch

import oracle
from delta_rule_linear_dpfp_gb300 import binding as fw
from delta_rule_linear_dpfp_gb300 import build, inputs
from tests.parity_util import TOL_BF16, f64, maxrel

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


CASES = [  # B, H, L, d_model, d_key, d_v, nu, w0
    (1, 8, 1024, 512, 64, 64, 1, False),     # the projected workload's shapes
    (2, 4, 200, 128, 32, 64, 2, True),       # ragged token count (400) and column count (516)
    (1, 2, 77, 64, 16, 16, 3, False),
    (3, 3, 50, 192, 64, 32, 1, True),
    (1, 8, 4096, 512, 64, 64, 1, True),      # the forward as one launch: the separate projection GEMM first
    (1, 2, 300, 256, 128, 64, 1, False),     # d_key 128: the separate projection GEMM first
]


def test_projected_path_choice():
    """The projections are folded into the prep where the forward runs as its
    two kernels (d_key, d_v <= 64); otherwise they run as a GEMM first."""
    assert fw.fw_delta_forward_kernel_count(1, 8, 1024, 64, 1, 64, 64, torch.bfloat16) == 2
    assert fw.fw_delta_forward_kernel_count(1, 8, 4096, 64, 1, 64, 64, torch.bfloat16) == 1


@pytest.mark.parametrize("case", CASES, ids=lambda c: "b{}h{}l{}dm{}dk{}dv{}nu{}w{}".format(*c))
def test_projected_parity(case):
    B, H, L, d_model, d_key, d_v, nu, w0 = case
    d = inputs.layer_inputs(B, H, L, d_model, d_key, d_v, nu, w0_var=0.01 if w0 else None, seed=sum(case[:7]))
    W0 = None if d["W0"] is None else d["W0"].cuda()
    y, Wf = fw.fw_delta_forward_projected(d["x"].cuda(), d["W_all"].cuda(), H, d_key, d_v, nu=nu, W0=W0)
    torch.cuda.synchronize()
    q, k, v, beta = oracle.project(f64(d["x"]), f64(d["W_all"]), H, d_key, d_v)
    yo, Wo = oracle.delta_forward(q, k, v, beta, None if d["W0"] is None else f64(d["W0"]), nu, 1e-6, NT)
    ey, ew = maxrel(f64(y), yo), maxrel(f64(Wf), Wo)
    assert ey <= TOL_BF16 and ew <= TOL_BF16, (ey, ew)


def test_projected_equals_forward_on_its_projections():
    # the projected path = the plain forward on bf16(x W_all), to bf16 rounding of q, k, v, beta
    B, H, L, d_model, d_key, d_v = 1, 4, 256, 256, 64, 64
    d = inputs.layer_inputs(B, H, L, d_model, d_key, d_v, seed=9)
    x, W = d["x"].cuda(), d["W_all"].cuda()
    y1, W1 = fw.fw_delta_forward_projected(x, W, H, d_key, d_v)
    q, k, v, beta = (torch.from_numpy(a).to(torch.bfloat16).cuda().contiguous()
                     for a in oracle.project(f64(d["x"]), f64(d["W_all"]), H, d_key, d_v))
    y2, W2 = fw.fw_delta_forward(q, k, v, beta, nu=1)
    assert maxrel(f64(y1), f64(y2)) <= TOL_BF16 and maxrel(f64(W1), f64(W2)) <= TOL_BF16


def test_projected_argument_checks():
    lib = fw.load()
    ws = lib.fw_delta_forward_projected_workspace_size
    assert ws(1, 64, 512, 8, 64, 1, 64, 64) > 0
    assert ws(1, 64, 500, 8, 64, 1, 64, 64) == 0            # d_model not a multiple of 64
    d = inputs.layer_inputs(1, 2, 64, 64, 16, 16, seed=1)
    x, W = d["x"].cuda(), d["W_all"].cuda()
    with pytest.raises(fw.FwError):
        fw.fw_delta_forward_projected(x, W[:, :8].contiguous(), 2, 16, 16)   # ldw too small
