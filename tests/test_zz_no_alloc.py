"""fw_delta_forward_noalloc, the forward for callers that cannot allocate
device memory at call time (a host program whose memory pool owns the GPU and
forbids further cudaMalloc, or a serving loop that cannot take the implicit
synchronisation of cudaMalloc / cudaFree).  It runs on the library's own
fixed scratch array instead of a caller workspace.

The file name sorts last so that a run that stops at the first failure has
run every other test before this one.  It must pass alone in a fresh process
and after the rest of the suite."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from delta_rule_linear_dpfp_gb300 import binding as fw
from delta_rule_linear_dpfp_gb300 import build, inputs
from tests.parity_util import TOL_BF16, f64, maxrel, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build.build()
    fw.load()


def test_noalloc_matches_workspace_forward_twice():
    """Two calls in a row through the C ABI give exactly what fw_delta_forward
    (which gets a caller workspace) gives: the same kernels on the same inputs
    are deterministic, so the comparison is bit for bit; the second call runs
    on the scratch left over from the first."""
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
            assert torch.equal(y_, y_ref) and torch.equal(W_, W_ref)


def test_noalloc_against_the_oracle():
    """The entry point's outputs against the fp64 oracle, within the bf16 bar."""
    h = inputs.random_forward_inputs(1, 2, 130, 32, 1, 32, "bf16", 0.01, seed=23)
    d = to_dev(h)
    y, W = fw.fw_delta_forward_noalloc(d["q"], d["k"], d["v"], d["beta"], W0=d["W0"], nu=1, chunk=64)
    torch.cuda.synchronize()
    y_ref, W_ref = oracle.delta_forward(f64(h["q"]), f64(h["k"]), f64(h["v"]), f64(h["beta"]),
                                        f64(h["W0"]), 1, 1e-6)
    assert maxrel(f64(y), y_ref) <= TOL_BF16 and maxrel(f64(W), W_ref) <= TOL_BF16


def test_noalloc_allocates_no_device_memory():
    """With the outputs already allocated, a call leaves the device's free
    memory unchanged: the library takes nothing from the device allocator."""
    d = to_dev(inputs.random_forward_inputs(2, 4, 256, 64, 1, 64, "bf16", None, seed=24))
    y = torch.empty(2, 4, 256, 64, dtype=torch.bfloat16, device="cuda")
    W = torch.empty(2, 4, 64, 128, dtype=torch.float32, device="cuda")
    fw.fw_delta_forward_noalloc(d["q"], d["k"], d["v"], d["beta"], nu=1, chunk=64, y=y, W_final=W)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        fw.fw_delta_forward_noalloc(d["q"], d["k"], d["v"], d["beta"], nu=1, chunk=64, y=y, W_final=W)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert np.isfinite(f64(y)).all()


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
