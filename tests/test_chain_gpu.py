"""Chains of calls on one stream with no host synchronisation between them.

Every tcgen05 kernel is launched with programmatic stream serialisation: it
may be scheduled while the kernel before it still runs, and it must not touch
global memory until that kernel has completed.  These chains put each hazard
between consecutive launches -- a read of what the previous call wrote, a
write of what the previous call read, two split-K calls sharing one workspace
-- and require the unsynchronised chain to give the same bits as the chain run
with a full synchronisation after every call (every kernel here is
deterministic).  The chain's single-GEMM result is also checked against the
oracle.
"""
import pytest
import torch

import oracle
import swiglu_mlp_gb300 as swg
import synth
from helpers import check_half, to_f64

pytestmark = pytest.mark.gpu


def _inputs(n, seed):
    g = synth.generator(seed)
    A = synth.normal((n, n), g)
    B = synth.normal((n, n), g, std=n ** -0.5)
    B2 = synth.normal((n, n), g, std=n ** -0.5)
    return A, B, B2


def _chain(A, B, B2, sync):
    """D1 = A B; D2 = D1 B (reads D1); D1 = A B2 (overwrites what the previous
    call read); D3 = D2 B2; then D3 + D1 in torch."""
    n = A.shape[0]
    dev = "cuda"
    Ad, Bd, B2d = A.to(dev), B.to(dev), B2.to(dev)
    D1 = torch.empty((n, n), dtype=torch.bfloat16, device=dev)
    D2 = torch.empty_like(D1)
    D3 = torch.empty_like(D1)
    steps = [
        lambda: swg.gemm(0, 0, n, n, n, 1.0, Ad, n, Bd, n, 0.0, D1, n, swg.BF16),
        lambda: swg.gemm(0, 0, n, n, n, 1.0, D1, n, Bd, n, 0.0, D2, n, swg.BF16),
        lambda: swg.gemm(0, 0, n, n, n, 1.0, Ad, n, B2d, n, 0.0, D1, n, swg.BF16),
        lambda: swg.gemm(0, 0, n, n, n, 1.0, D2, n, B2d, n, 0.0, D3, n, swg.BF16),
    ]
    for f in steps:
        f()
        if sync:
            torch.cuda.synchronize()
    D4 = D3 + D1                    # a torch kernel after ours on the same stream
    torch.cuda.synchronize()
    return D1.cpu(), D2.cpu(), D3.cpu(), D4.cpu()


@pytest.mark.parametrize("n", [384, 1024])
def test_gemm_chain_hazards(n):
    A, B, B2 = _inputs(n, seed=500 + n)
    ref = _chain(A, B, B2, sync=True)
    got = _chain(A, B, B2, sync=False)
    assert swg.get_device_error() == 0
    for r, x in zip(ref, got):
        assert torch.equal(r, x)
    rows = [0, 1, n // 2, n - 1]
    yhat = oracle.gemm(0, 0, n, n, n, 1.0, A, n, B2, n, 0.0, rows=rows)
    check_half(to_f64(got[0])[rows], yhat, "chain: D1 = A B2 after the overwrite")


def _splitk_chain(sync):
    """Two skinny split-K calls sharing the stream's workspace, the second
    reading the first's output, then a fused SwiGLU and a GEMM of its output."""
    M, N, K = 32, 2048, 8192
    A, B, C = synth.gemm_bf16(M, N, K, seed=520, c=True)
    g = synth.generator(521)
    B2 = synth.normal((N, N), g, std=N ** -0.5)
    Ad, Bd, Cd, B2d = A.cuda(), B.cuda(), C.cuda(), B2.cuda()
    E = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    _, W1, W2 = synth.swiglu(1, N, 512, seed=522)
    Wf = swg.interleave_weights(W1.cuda(), W2.cuda())
    Y = torch.empty((M, 512), dtype=torch.bfloat16, device="cuda")
    F = torch.empty((M, 512), dtype=torch.bfloat16, device="cuda")
    Wd = synth.normal((512, 512), g, std=512 ** -0.5).cuda()
    torch.cuda.synchronize()
    steps = [
        lambda: swg.gemm(0, 0, M, N, K, 1.0, Ad, K, Bd, N, 1.0, Cd, N, swg.BF16),
        lambda: swg.gemm_ex(0, 0, M, N, N, 1.0, Cd, N, B2d, N, 0.0, E, N, swg.BF16, 4),
        lambda: swg.swiglu_mlp(E, Wf, Y, M, 512, N),
        lambda: swg.gemm(0, 0, M, 512, 512, 1.0, Y, 512, Wd, 512, 0.0, F, 512, swg.BF16),
    ]
    for f in steps:
        f()
        if sync:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    return Cd.cpu(), E.cpu(), Y.cpu(), F.cpu()


def test_splitk_and_swiglu_chain_hazards():
    ref = _splitk_chain(sync=True)
    got = _splitk_chain(sync=False)
    assert swg.get_device_error() == 0
    for r, x in zip(ref, got):
        assert torch.equal(r, x)
