"""gemm_splitk_noalloc: gemm_ex for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc once they are running: a host framework
that already holds nearly all device memory in its own pool, or a serving loop
that forbids device allocation because it can synchronise the whole GPU.
gemm_splitk_noalloc serves them: it runs the kernels gemm_ex plans for the
same arguments, but keeps split-K partial sums in a fixed array inside the
library instead of a cudaMalloc'd workspace.

These tests call it through the C ABI twice in a row, on different shapes and
kernels, and require each result to equal gemm_ex's bit for bit and to match
the FP64 oracle within the tolerance the other parity tests use.  Outputs sit
inside guard bands, and the fixed array inside its own (SWG_TEST_WS_GUARD=1
is set for this module before its first call).  They also check the size
limit, that repeated calls leave device free memory unchanged, and -- in a
fresh process -- that the first call commits no more than the array and the
library's code.

This file is collected last, so that a stop-at-first-failure run has already
run every other test; it passes alone in a fresh process as well.
"""
import ctypes
import json
import os
import subprocess
import sys

import pytest
import torch

import oracle
import swiglu_mlp_gb300 as swg
import synth
from helpers import Guarded, check_f32, check_half, to_f64

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 * 1024 * 1024     # SWG_NOALLOC_SCRATCH_BYTES
GUARD_BYTES = 2 * 64 * 1024          # the array's two guard bands
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _guarded_array():
    old = os.environ.get("SWG_TEST_WS_GUARD")
    os.environ["SWG_TEST_WS_GUARD"] = "1"
    yield
    if old is None:
        os.environ.pop("SWG_TEST_WS_GUARD", None)
    else:
        os.environ["SWG_TEST_WS_GUARD"] = old


TYPES = {  # code -> (input dtype, output dtype, oracle input type, oracle C type)
    swg.BF16: (torch.bfloat16, torch.bfloat16, "bf16", "bf16"),
    swg.BF16_F32OUT: (torch.bfloat16, torch.float32, "bf16", "f32"),
    swg.E4M3_BF16OUT: (torch.float8_e4m3fn, torch.bfloat16, "e4m3", "bf16"),
}


def _both(tA, tB, M, N, K, alpha, beta, code, split_k, seed):
    """Runs gemm_ex, then gemm_splitk_noalloc, on the same inputs and guarded
    copies of the same C; returns (D from gemm_ex, D from the no-allocation
    call, the oracle's D)."""
    tin, tout, oin, oout = TYPES[code]
    g = synth.generator(seed)
    if tin == torch.float8_e4m3fn:
        A = (torch.randn(M, K, generator=g)).to(tin)
        B = (torch.randn(N, K, generator=g) * 0.5).to(tin)
    else:
        A = synth.normal(synth.stored_shape(tA, M, K), g, dtype=tin)
        B = synth.normal(synth.stored_shape(tB, K, N), g, dtype=tin)
    C = synth.normal((M, N), g, dtype=tout)
    Ad, Bd = A.cuda(), B.cuda()
    outs = []
    for fn in (swg.gemm_ex, swg.gemm_splitk_noalloc):
        Cg = Guarded(M, N, tout, init=C)
        fn(tA, tB, M, N, K, alpha, Ad, A.shape[1], Bd, B.shape[1], beta, Cg.view, Cg.ld, code,
           split_k)
        assert swg.get_device_error() == 0
        outs.append(Cg.cpu(f"{fn.__name__} {M}x{N}x{K}"))
    yhat = oracle.gemm(tA, tB, M, N, K, alpha, A, A.shape[1], B, B.shape[1], beta, C, N,
                       in_type=oin, c_type=oout)
    return outs[0], outs[1], yhat


def test_two_calls_match_existing_entry_point():
    # call 1: the skinny split-K shape with four K ranges (few rows: the
    # transposed product, partials in the fixed array), beta = 1, bf16 out
    ref, new, yhat = _both(0, 0, 64, 4096, 16384, 1.0, 1.0, swg.BF16, 4, seed=101)
    assert torch.equal(new, ref)
    check_half(to_f64(new), yhat, "noalloc call 1")
    # call 2: right after it, another shape and kernel (M > 64: 128- or
    # 256-row tiles whose last partial tile is a TMA store into the array),
    # three forced splits, beta = 0, FP32 out
    ref, new, yhat = _both(1, 1, 296, 520, 1000, 0.5, 0.0, swg.BF16_F32OUT, 3, seed=102)
    assert torch.equal(new, ref)
    check_f32(to_f64(new), yhat, 1000, "noalloc call 2")
    assert swg.debug_workspace_guards() == 0


def test_e4m3_few_rows():
    """8-bit operands: the e4m3 few-rows split-K kernel with its partials in
    the fixed array."""
    ref, new, yhat = _both(0, 1, 16, 1000, 4096, 1.0 / 32, 0.5, swg.E4M3_BF16OUT, 0, seed=103)
    assert torch.equal(new, ref)
    check_half(to_f64(new), yhat, "noalloc e4m3")
    assert swg.debug_workspace_guards() == 0


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
    A, B, C = synth.gemm_bf16(M, N, K, seed=104, c=True)
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


_PROBE = r"""
import json, sys
sys.path.insert(0, sys.argv[1])
import torch
import swiglu_mlp_gb300 as swg
M, N, K = 32, 2048, 8192
g = torch.Generator().manual_seed(7)
A = torch.randn(M, K, generator=g).to(torch.bfloat16).cuda()
B = torch.randn(K, N, generator=g).to(torch.bfloat16).cuda()
C = torch.randn(M, N, generator=g).to(torch.bfloat16).cuda()
torch.cuda.synchronize()
free0 = torch.cuda.mem_get_info()[0]
swg.gemm_splitk_noalloc(0, 0, M, N, K, 1.0, A, K, B, N, 1.0, C, N, swg.BF16)
torch.cuda.synchronize()
free1 = torch.cuda.mem_get_info()[0]
for _ in range(3):
    swg.gemm_splitk_noalloc(0, 0, M, N, K, 1.0, A, K, B, N, 1.0, C, N, swg.BF16)
torch.cuda.synchronize()
free2 = torch.cuda.mem_get_info()[0]
print(json.dumps({"free0": free0, "free1": free1, "free2": free2,
                  "err": swg.get_device_error()}))
"""


def test_first_call_in_a_fresh_process_commits_only_the_array_and_code():
    """With CUDA's lazy module loading the first call is where the library's
    device image -- its kernels and the fixed array -- becomes resident.  The
    drop in free device memory at that call is at most the array plus the
    library's code (48 MiB allowed for the code); later calls change nothing."""
    env = dict(os.environ)
    env.pop("SWG_TEST_WS_GUARD", None)
    r = subprocess.run([sys.executable, "-c", _PROBE, ROOT], capture_output=True, text=True,
                       env=env, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads(r.stdout.strip().splitlines()[-1])
    assert d["err"] == 0
    drop = d["free0"] - d["free1"]
    assert 0 <= drop <= SCRATCH_BYTES + GUARD_BYTES + 48 * 1024 * 1024, d
    assert d["free2"] == d["free1"], d
