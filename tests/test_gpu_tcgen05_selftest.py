"""The tcgen05 building blocks of the bf16 forward (operand layouts with the
128-byte swizzle, K-major and MN-major matrix descriptors, the instruction
descriptor, the tensor-memory accumulator layout, commit and mbarrier
completion) against a plain matrix product.  If one of these conventions were
wrong, the forward's parity tests would fail without saying why; these say
which one."""
import numpy as np
import pytest
import torch

from delta_rule_linear_dpfp_gb300 import binding as fw
from delta_rule_linear_dpfp_gb300 import build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build.build()
    fw.load()


def _operands(N, K, seed):
    g = torch.Generator().manual_seed(seed)
    # small integers times powers of two: exact in bf16 and in the fp32 sums
    A = (torch.randint(-8, 9, (128, K), generator=g).float() / 4.0)
    B = (torch.randint(-8, 9, (N, K), generator=g).float() / 8.0)
    return A, B


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (1, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("N", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("K", [16, 64, 128])
def test_umma_matches_matmul(a_mn, b_mn, N, K):
    A, B = _operands(N, K, seed=N * 1000 + K + 7 * a_mn + 3 * b_mn)
    D = fw.fw_selftest_umma(A.cuda(), B.cuda(), a_mn=a_mn, b_mn=b_mn)
    torch.cuda.synchronize()
    assert fw.fw_device_status() == fw.FW_OK
    ref = A.double() @ B.double().T
    assert np.array_equal(D.cpu().double().numpy(), ref.numpy())


def test_swapped_mn_offsets_are_detected():
    """With the leading and stride offsets of an MN-major descriptor exchanged
    the product comes out wrong: the test can tell the two conventions apart."""
    A, B = _operands(64, 128, seed=1)
    D = fw.fw_selftest_umma(A.cuda(), B.cuda(), a_mn=1, b_mn=1, swap_mn=1)
    torch.cuda.synchronize()
    assert fw.fw_device_status() == fw.FW_OK
    ref = A.double() @ B.double().T
    assert not np.array_equal(D.cpu().double().numpy(), ref.numpy())


def test_bounded_wait_reports_timeout_and_context_survives():
    """A wait on an mbarrier nothing arrives at gives up after its bound, the
    status word reports FW_ERR_TIMEOUT once, and the GPU keeps working."""
    assert fw.fw_device_status() == fw.FW_OK
    fw.fw_selftest_wait_timeout(3000)
    assert fw.fw_device_status() == fw.FW_ERR_TIMEOUT
    assert fw.fw_device_status() == fw.FW_OK            # cleared by the read
    A, B = _operands(64, 64, seed=5)
    D = fw.fw_selftest_umma(A.cuda(), B.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(D.cpu().double().numpy(), (A.double() @ B.double().T).numpy())


def test_flag_wait_reports_timeout_and_context_survives():
    """A wait on a ready flag nothing sets (the single-launch forward's hand-over
    between CTAs) gives up after its bound, the status word reports
    FW_ERR_TIMEOUT once, and the single-launch forward still runs correctly."""
    assert fw.fw_device_status() == fw.FW_OK
    fw.fw_selftest_flag_timeout(3000)
    assert fw.fw_device_status() == fw.FW_ERR_TIMEOUT
    assert fw.fw_device_status() == fw.FW_OK
    from delta_rule_linear_dpfp_gb300 import inputs
    assert fw.fw_delta_forward_kernel_count(2, 8, 2048, 64, 3, 64, 64, torch.bfloat16) == 1
    d = {k: (None if v is None else v.cuda()) for k, v in inputs.forward_inputs("b2h8_l2048_nu3").items()}
    y1, W1 = fw.fw_delta_forward(d["q"], d["k"], d["v"], d["beta"], W0=d["W0"], nu=3)
    y2, W2 = fw.fw_delta_forward(d["q"], d["k"], d["v"], d["beta"], W0=d["W0"], nu=3)
    torch.cuda.synchronize()
    assert fw.fw_device_status() == fw.FW_OK
    assert torch.equal(y1, y2) and torch.equal(W1, W2)
