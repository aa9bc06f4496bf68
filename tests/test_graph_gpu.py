"""Capture into a CUDA graph and replay.

Every entry point only enqueues kernels (no host synchronisation), and a
split-K workspace stays allocated once a stream has one, so a sequence of
calls can be captured into a CUDA graph after it has run once on the same
stream.  These tests capture a large CTA-pair GEMM, a skinny split-K GEMM
(workspace and dependent reduction), the fused SwiGLU and the full MLP,
and check that replays reproduce the eager results bit for bit, also after
the inputs are overwritten in place.  They also check that a call that would
have to allocate while its stream is capturing is refused and launches
nothing.
"""
import ctypes

import pytest
import torch

import swiglu_mlp_gb300 as swg
import synth

pytestmark = pytest.mark.gpu


def _problem(seed):
    g = synth.generator(seed)
    n = 1024
    P = {
        "A": synth.normal((n, n), g).cuda(),
        "B": synth.normal((n, n), g, std=n ** -0.5).cuda(),
        "As": synth.normal((32, 8192), g).cuda(),
        "Bs": synth.normal((8192, 2048), g, std=0.05).cuda(),
        "X": synth.normal((512, 896), g).cuda(),
    }
    _, W1, W2 = synth.swiglu(1, 896, 1536, seed=seed + 1)
    P["Wf"] = swg.interleave_weights(W1.cuda(), W2.cuda())
    P["Wd"] = synth.normal((1536, 896), g, std=0.02).cuda()
    return P


def _outputs():
    bf = torch.bfloat16
    return {
        "D": torch.empty((1024, 1024), dtype=bf, device="cuda"),
        "Ds": torch.empty((32, 2048), dtype=bf, device="cuda"),
        "Y": torch.empty((512, 1536), dtype=bf, device="cuda"),
        "Y2": torch.empty((512, 1536), dtype=bf, device="cuda"),
        "O": torch.empty((512, 896), dtype=bf, device="cuda"),
    }


def _work(P, O):
    swg.gemm(0, 0, 1024, 1024, 1024, 1.0, P["A"], 1024, P["B"], 1024, 0.0, O["D"], 1024,
             swg.BF16)
    swg.gemm(0, 0, 32, 2048, 8192, 1.0, P["As"], 8192, P["Bs"], 2048, 0.0, O["Ds"], 2048,
             swg.BF16)
    swg.swiglu_mlp(P["X"], P["Wf"], O["Y"], 512, 1536, 896)
    swg.swiglu_mlp_forward(P["X"], P["Wf"], P["Wd"], O["Y2"], O["O"], 512, 1536, 896, 0.0)


def _snapshot(O):
    return {k: v.cpu() for k, v in O.items()}


def test_capture_and_replay_bitwise():
    s = torch.cuda.Stream()
    P, O = _problem(700), _outputs()
    with torch.cuda.stream(s):
        _work(P, O)                               # warm-up: workspace, attributes
    torch.cuda.synchronize()
    eager = _snapshot(O)
    for v in O.values():
        v.zero_()
    torch.cuda.synchronize()

    g = torch.cuda.CUDAGraph()
    before = swg.launch_count()
    with torch.cuda.graph(g, stream=s):
        _work(P, O)
    captured = swg.launch_count() - before
    assert captured >= 7                          # GEMM, GEMM + reduction, SwiGLU, SwiGLU + GEMM
    for v in O.values():
        v.zero_()
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert swg.get_device_error() == 0
    for k, v in _snapshot(O).items():
        assert torch.equal(v, eager[k]), k

    # New input values in the same buffers: the replay recomputes.
    P2 = _problem(701)
    for k in ("A", "B", "As", "Bs", "X", "Wf", "Wd"):
        P[k].copy_(P2[k])
    with torch.cuda.stream(s):
        _work(P2, O)
    torch.cuda.synchronize()
    eager2 = _snapshot(O)
    for v in O.values():
        v.zero_()
    torch.cuda.synchronize()
    g.replay()
    g.replay()                                    # replays back to back
    torch.cuda.synchronize()
    for k, v in _snapshot(O).items():
        assert torch.equal(v, eager2[k]), k
    assert any(not torch.equal(eager[k], eager2[k]) for k in eager)


@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")
def test_allocation_while_capturing_is_refused():
    """A split-K call with nine explicit K ranges (the workspace path) on a
    stream that has no workspace yet would have to allocate one: while that stream is capturing, the call returns
    SWG_ERR_UNSUPPORTED and launches nothing."""
    s = torch.cuda.Stream()
    P, O = _problem(702), _outputs()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    before = swg.launch_count()
    rc = None
    with torch.cuda.graph(g, stream=s):
        rc = swg.load().gemm_ex(0, 0, 32, 2048, 8192, ctypes.c_float(1.0), P["As"].data_ptr(),
                                8192, P["Bs"].data_ptr(), 2048, ctypes.c_float(0.0),
                                O["Ds"].data_ptr(), 2048, swg.BF16, 9,
                                ctypes.c_void_p(s.cuda_stream))
    assert rc == 3                                # SWG_ERR_UNSUPPORTED
    assert swg.launch_count() == before
    # Outside the capture the same call allocates and runs.
    with torch.cuda.stream(s):
        swg.gemm_ex(0, 0, 32, 2048, 8192, 1.0, P["As"], 8192, P["Bs"], 2048, 0.0, O["Ds"], 2048,
                    swg.BF16, 9)
    torch.cuda.synchronize()
    assert swg.get_device_error() == 0
