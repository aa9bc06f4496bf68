"""Failure detection on the GPU without faulting it.

Every barrier wait in the pipeline kernels is bounded; when one runs out the
kernel records SWG_ERR_DEVICE_TIMEOUT in the device error word, frees its
tensor memory and exits.  swg_selftest_wait_timeout makes that happen on
purpose (a barrier nothing completes, a 1 ms limit); the context must stay
usable afterwards.  Host-side failures are injected on the host.
"""
import pytest
import torch

import oracle
import swiglu_mlp_gb300 as swg
import synth
from helpers import check_half, to_f64

pytestmark = pytest.mark.gpu

TIMEOUT = 6        # SWG_ERR_DEVICE_TIMEOUT
NO_MEMORY = 5      # SWG_ERR_NO_MEMORY


def _small_gemm_ok():
    M, N, K = 200, 256, 192
    A, B, _ = synth.gemm_bf16(M, N, K, seed=501)
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    swg.gemm(0, 0, M, N, K, 1.0, A.cuda(), K, B.cuda(), N, 0.0, D, N, swg.BF16)
    assert swg.get_device_error() == 0
    check_half(to_f64(D), oracle.gemm(0, 0, M, N, K, 1.0, A, K, B, N, 0.0), "after timeout")


def test_bounded_wait_reports_timeout_and_context_survives():
    assert swg.get_device_error() == 0
    swg.selftest_wait_timeout(1_000_000)          # 1 ms
    assert swg.get_device_error() == TIMEOUT
    assert swg.get_device_error() == 0            # read-and-clear
    _small_gemm_ok()


def test_timeouts_on_two_streams_in_a_row():
    s = torch.cuda.Stream()
    for _ in range(2):
        swg.selftest_wait_timeout(500_000, stream=s)
        assert swg.get_device_error(s) == TIMEOUT
    _small_gemm_ok()


def test_workspace_allocation_failure_is_reported(monkeypatch):
    """Split-K needs the library workspace; a failed allocation returns
    SWG_ERR_NO_MEMORY before any launch, and the next call works."""
    M, N, K = 32, 2048, 4096
    A, B, C = synth.gemm_bf16(M, N, K, seed=502, c=True)
    Ad, Bd, Cd = A.cuda(), B.cuda(), C.cuda()
    swg.shutdown()                                # drop any cached workspace
    monkeypatch.setenv("SWG_TEST_FAIL_ALLOC", "1")
    before = swg.launch_count()
    with pytest.raises(swg.SwgError) as e:
        swg.gemm_ex(0, 0, M, N, K, 1.0, Ad, K, Bd, N, 1.0, Cd, N, swg.BF16, 4)
    assert e.value.status == NO_MEMORY
    assert swg.launch_count() == before
    torch.cuda.synchronize()
    assert torch.equal(Cd.cpu(), C)               # nothing written
    monkeypatch.delenv("SWG_TEST_FAIL_ALLOC")
    swg.gemm_ex(0, 0, M, N, K, 1.0, Ad, K, Bd, N, 1.0, Cd, N, swg.BF16, 4)
    assert swg.get_device_error() == 0
    check_half(to_f64(Cd), oracle.gemm(0, 0, M, N, K, 1.0, A, K, B, N, 1.0, C, N), "after")
