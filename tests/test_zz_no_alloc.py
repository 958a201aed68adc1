"""fw_delta_forward_noalloc, the forward for callers that cannot allocate
device memory at call time (a host program whose memory pool owns the GPU and
forbids further cudaMalloc, or a serving loop that cannot take the implicit
synchronisation of cudaMalloc / cudaFree).  It runs on the library's own
fixed scratch array instead of a caller workspace.

The file name sorts last so that a run that stops at the first failure has
run every other test before this one.  It must pass alone in a fresh process
and after the rest of the suite."""
import ctypes

import pytest
import torch

from delta_rule_linear_dpfp_gb300 import binding as fw
from delta_rule_linear_dpfp_gb300 import build, inputs
from tests.parity_util import f64, maxrel, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build.build()
    fw.load()


def test_noalloc_matches_workspace_forward_twice():
    """Two calls in a row through the C ABI agree with fw_delta_forward (which
    gets a caller workspace) within the bf16 tolerance of the parity tests;
    the second call runs on the scratch left over from the first."""
    d = to_dev(inputs.random_forward_inputs(2, 4, 200, 64, 2, 64, "bf16", 0.01, seed=21))
    e = to_dev(inputs.random_forward_inputs(2, 4, 200, 64, 2, 64, "bf16", None, seed=22))
    for case in (d, e):
        y_ref, W_ref = fw.fw_delta_forward(case["q"], case["k"], case["v"], case["beta"],
                                           W0=case["W0"], nu=2, chunk=64)
        y1, W1 = fw.fw_delta_forward_noalloc(case["q"], case["k"], case["v"], case["beta"],
                                             W0=case["W0"], nu=2, chunk=64)
        y2, W2 = fw.fw_delta_forward_noalloc(case["q"], case["k"], case["v"], case["beta"],
                                             W0=case["W0"], nu=2, chunk=64)
        torch.cuda.synchronize()
        assert fw.fw_device_status() == fw.FW_OK
        for y_, W_ in ((y1, W1), (y2, W2)):
            assert maxrel(f64(y_), f64(y_ref)) <= 2e-2
            assert maxrel(f64(W_), f64(W_ref)) <= 2e-2


def test_noalloc_rejects_shapes_beyond_the_scratch():
    """A shape whose workspace exceeds the fixed array is refused up front
    (nothing is enqueued: the pointers below are never read)."""
    B, H, L, d_key, nu, d_v, C = 64, 16, 4096, 64, 3, 64, 64
    need = fw.fw_delta_forward_workspace_size(B, H, L, d_key, nu, d_v, C, torch.bfloat16)
    assert need > fw.NOALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(0x10000)
    rc = fw.load().fw_delta_forward_noalloc(fake, fake, fake, fake, None, None, fake, B, H, L,
                                            d_key, nu, d_v, C, fw.FW_DTYPE_BF16, 1e-6, None)
    assert rc == fw.FW_ERR_UNSUPPORTED
