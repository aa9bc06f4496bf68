"""Concurrent use: several streams, several host threads.

The split-K workspace is per (device, stream) and the per-device state is
created under a mutex, so calls on different streams may overlap on the GPU
and calls from different host threads may overlap in the library (ctypes
releases the interpreter lock around each call).  Every result must equal,
bit for bit, the same call made alone on the default stream.
"""
import threading

import pytest
import torch

import swiglu_mlp_gb300 as swg
import synth

pytestmark = pytest.mark.gpu


def _case(seed):
    g = synth.generator(seed)
    A = synth.normal((48, 8192), g).cuda()
    B = synth.normal((8192, 3072), g, std=0.05).cuda()
    X = synth.normal((384, 1024), g).cuda()
    W = synth.normal((1024, 2048), g, std=0.03).cuda()
    return A, B, X, W


def _run(case, D, Y, stream):
    A, B, X, W = case
    swg.gemm(0, 0, 48, 3072, 8192, 1.0, A, 8192, B, 3072, 0.0, D, 3072, swg.BF16, stream=stream)
    swg.swiglu_mlp(X, W, Y, 384, 1024, 1024, stream=stream)


def _buffers():
    return (torch.empty((48, 3072), dtype=torch.bfloat16, device="cuda"),
            torch.empty((384, 1024), dtype=torch.bfloat16, device="cuda"))


def _reference(cases):
    refs = []
    for c in cases:
        D, Y = _buffers()
        _run(c, D, Y, torch.cuda.current_stream())
        torch.cuda.synchronize()
        refs.append((D.cpu(), Y.cpu()))
    return refs


def test_streams_overlap_split_k():
    """Split-K GEMMs and SwiGLU on four streams at once, each stream with its
    own workspace, repeated without synchronisation."""
    cases = [_case(800 + i) for i in range(4)]
    refs = _reference(cases)
    streams = [torch.cuda.Stream() for _ in cases]
    bufs = [_buffers() for _ in cases]
    torch.cuda.synchronize()
    for _ in range(5):
        for c, s, (D, Y) in zip(cases, streams, bufs):
            _run(c, D, Y, s)
    torch.cuda.synchronize()
    assert swg.get_device_error() == 0
    for (D, Y), (rD, rY) in zip(bufs, refs):
        assert torch.equal(D.cpu(), rD)
        assert torch.equal(Y.cpu(), rY)


def test_host_threads_call_concurrently():
    """Four host threads, each with its own stream, call the library in a
    loop at the same time."""
    cases = [_case(810 + i) for i in range(4)]
    refs = _reference(cases)
    errors = []
    results = [None] * len(cases)

    def worker(i):
        try:
            s = torch.cuda.Stream()
            D, Y = _buffers()
            with torch.cuda.stream(s):
                for _ in range(20):
                    _run(cases[i], D, Y, s)
            s.synchronize()
            results[i] = (D.cpu(), Y.cpu())
        except Exception as e:          # reported below, on the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(cases))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not any(t.is_alive() for t in threads)
    assert not errors, errors
    assert swg.get_device_error() == 0
    for (D, Y), (rD, rY) in zip(results, refs):
        assert torch.equal(D, rD)
        assert torch.equal(Y, rY)
