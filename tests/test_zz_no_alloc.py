"""gemm_splitk_noalloc: the split-K GEMM that allocates no device memory.

Some callers cannot call cudaMalloc once they are running (a host framework
that already holds nearly all device memory in its own pool, or a serving
loop that forbids device allocation because it can synchronise the GPU).
gemm_splitk_noalloc serves them by keeping its FP32 partial sums in a fixed
array inside the library.  These tests call it through the C ABI twice in a
row, on different shapes, and compare each result with gemm_ex's (the
workspace-allocating path with the same split factor); they also check the
size limit and that repeated calls leave device free memory unchanged.

This file is collected last so that a stop-at-first-failure run has already
run every other test.
"""
import ctypes

import pytest
import torch

import swiglu_mlp_gb300 as swg
import synth
from helpers import check_f32, check_half, to_f64

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 * 1024 * 1024     # SWG_NOALLOC_SCRATCH_BYTES


def _both(tA, tB, M, N, K, alpha, beta, code, split_k, seed):
    """Runs gemm_ex and gemm_splitk_noalloc on the same inputs; returns both D."""
    tin = torch.float16 if code in (swg.F16, swg.F16_F32OUT) else torch.bfloat16
    tout = torch.float32 if code in (swg.F16_F32OUT, swg.BF16_F32OUT) else tin
    g = synth.generator(seed)
    A = synth.normal(synth.stored_shape(tA, M, K), g, dtype=tin).cuda()
    B = synth.normal(synth.stored_shape(tB, K, N), g, dtype=tin).cuda()
    C = synth.normal((M, N), g, dtype=tout).cuda()
    D_ref, D_new = C.clone(), C.clone()
    swg.gemm_ex(tA, tB, M, N, K, alpha, A, A.shape[1], B, B.shape[1], beta, D_ref, N, code,
                split_k)
    swg.gemm_splitk_noalloc(tA, tB, M, N, K, alpha, A, A.shape[1], B, B.shape[1], beta, D_new,
                            N, code, split_k)
    assert swg.get_device_error() == 0
    return to_f64(D_ref), to_f64(D_new)


def test_two_calls_match_existing_entry_point():
    # call 1: the skinny split-K shape, automatic split, beta = 1, bf16 out
    ref, new = _both(0, 0, 64, 4096, 16384, 1.0, 1.0, swg.BF16, 0, seed=101)
    check_half(new, ref, "noalloc call 1")
    # call 2: another shape and split reuses the shared array
    ref, new = _both(1, 1, 40, 600, 1000, 0.5, 0.0, swg.BF16_F32OUT, 3, seed=102)
    check_f32(new, ref, 1000, "noalloc call 2")


def test_rejects_partials_larger_than_the_fixed_array():
    M, N, K, split_k = 64, 16384, 4096, 16
    assert split_k * M * N * 4 > SCRATCH_BYTES
    A = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((K, N), dtype=torch.bfloat16, device="cuda")
    C = torch.full((M, N), 3.0, dtype=torch.bfloat16, device="cuda")
    before = swg.launch_count()
    rc = swg.load().gemm_splitk_noalloc(0, 0, M, N, K, ctypes.c_float(1.0), A.data_ptr(), K,
                                        B.data_ptr(), N, ctypes.c_float(0.0), C.data_ptr(), N,
                                        swg.BF16, split_k, None)
    assert rc == 3                        # SWG_ERR_UNSUPPORTED
    assert swg.launch_count() == before
    torch.cuda.synchronize()
    assert torch.all(C == 3.0)


def test_repeated_calls_leave_device_memory_unchanged():
    M, N, K = 32, 4096, 8192
    A, B, C = synth.gemm_bf16(M, N, K, seed=103, c=True)
    A, B, C = A.cuda(), B.cuda(), C.cuda()
    swg.gemm_splitk_noalloc(0, 0, M, N, K, 1.0, A, K, B, N, 1.0, C, N, swg.BF16)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        swg.gemm_splitk_noalloc(0, 0, M, N, K, 1.0, A, K, B, N, 1.0, C, N, swg.BF16)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert swg.get_device_error() == 0
