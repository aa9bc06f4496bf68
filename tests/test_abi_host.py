"""Host-side checks of the C ABI that need no GPU.

The library must load on a machine without a GPU, export every function that
include/swiglu_mlp.h declares, and reject bad arguments before any CUDA call
(so these checks return the documented status codes here too).
"""
import ctypes
import os
import re

import pytest

import swiglu_mlp_gb300 as swg
from swiglu_mlp_gb300 import build as swg_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "swiglu_mlp.h")

OK, INVALID, MISALIGNED, UNSUPPORTED, CUDA_ERR = 0, 1, 2, 3, 4
P = 0x10000           # a fake, 16-byte-aligned device address (never dereferenced)


@pytest.fixture(scope="module")
def lib():
    swg_build.build()
    return swg.load()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"SWG_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def test_header_declares_the_entry_points():
    names = set(declared_functions())
    assert {"gemm", "swiglu_mlp", "gemm_ex", "swiglu_interleave", "swg_status_string",
            "swg_get_device_error", "swg_launch_count", "swg_shutdown"} <= names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} not exported"
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    assert swg.status_string(0) == "SWG_OK"
    assert swg.status_string(2) == "SWG_ERR_MISALIGNED"
    assert swg.status_string(6) == "SWG_ERR_DEVICE_TIMEOUT"
    assert swg.status_string(99) == "SWG_ERR_UNKNOWN"


def g(lib, **kw):
    a = dict(tA=0, tB=0, M=128, N=128, K=64, alpha=1.0, A=P, lda=64, B=P, ldb=128, beta=0.0,
             C=P, ldc=128, dtype=1)
    a.update(kw)
    return lib.gemm(a["tA"], a["tB"], a["M"], a["N"], a["K"], a["alpha"], a["A"], a["lda"],
                    a["B"], a["ldb"], a["beta"], a["C"], a["ldc"], a["dtype"], None)


def test_gemm_validation(lib):
    assert g(lib, dtype=7) == UNSUPPORTED
    assert g(lib, tA=2) == INVALID
    assert g(lib, M=-1) == INVALID
    assert g(lib, K=-5) == INVALID
    assert g(lib, M=0) == OK and g(lib, N=0) == OK          # no-ops, no CUDA call
    assert g(lib, A=None) == INVALID
    assert g(lib, B=None) == INVALID
    assert g(lib, C=None) == INVALID
    assert g(lib, lda=63) == INVALID                        # op N: lda >= K
    assert g(lib, tA=1, lda=64) == INVALID                  # op T: lda >= M = 128
    assert g(lib, ldb=120) == INVALID                       # op N: ldb >= N
    assert g(lib, tB=1, ldb=32) == INVALID                  # op T: ldb >= K
    assert g(lib, ldc=100) == INVALID
    assert g(lib, A=P + 2) == MISALIGNED
    assert g(lib, C=P + 8) == MISALIGNED
    assert g(lib, lda=68) == MISALIGNED                     # 136 bytes
    assert g(lib, ldc=130) == MISALIGNED
    assert g(lib, M=2 ** 31, ldc=2 ** 31) == UNSUPPORTED
    assert lib.gemm_ex(0, 0, 128, 128, 64, 1.0, P, 64, P, 128, 0.0, P, 128, 1, -1, None) == INVALID
    # Calls that pass validation would launch; with fake pointers that is only
    # allowed where there is no GPU (they then fail at the first CUDA call).
    if not _has_gpu():
        assert g(lib, K=0, A=None, B=None, lda=0, ldb=0) == CUDA_ERR   # K = 0 needs no A, B
        assert g(lib, dtype=0, ldc=132) == CUDA_ERR                    # f32: 528 B rows aligned


def _has_gpu():
    import torch
    return torch.cuda.is_available()


@pytest.mark.skipif(_has_gpu(), reason="checks the no-GPU path")
def test_valid_call_without_gpu_reports_cuda_error(lib):
    assert g(lib) == CUDA_ERR
    # The runtime error behind it is recorded for this thread and named.
    code = lib.swg_last_cuda_error()
    assert code not in (0, 10000)
    name = lib.swg_cuda_error_name(code).decode()
    assert name.startswith("cuda") and "Error" in name
    assert lib.swg_cuda_error_name(0).decode() == "none"


@pytest.mark.skipif(_has_gpu(), reason="checks the no-GPU path")
def test_binding_error_names_the_cuda_error():
    import swiglu_mlp_gb300 as swg
    with pytest.raises(swg.SwgError) as info:
        swg.gemm(0, 0, 128, 128, 64, 1.0, P, 64, P, 128, 0.0, P, 128, swg.BF16)
    assert info.value.status == CUDA_ERR
    assert info.value.cuda_error != 0
    assert "[CUDA" in str(info.value)


def test_swiglu_validation(lib):
    f = lib.swiglu_mlp
    assert f(P, P, P, -1, 64, 64, None) == INVALID
    assert f(P, P, P, 0, 64, 64, None) == OK
    assert f(P, P, None, 8, 64, 64, None) == INVALID
    assert f(None, P, P, 8, 64, 64, None) == INVALID
    assert f(P, P, P, 8, 60, 64, None) == MISALIGNED        # N % 8
    assert f(P, P, P, 8, 64, 60, None) == MISALIGNED        # K % 8
    assert f(P + 4, P, P, 8, 64, 64, None) == MISALIGNED
    assert f(P, P, P, 8, 2 ** 30, 64, None) == UNSUPPORTED


def test_interleave_validation(lib):
    f = lib.swiglu_interleave
    assert f(P, P, P, -1, 8, None) == INVALID
    assert f(P, P, P, 0, 8, None) == OK
    assert f(None, P, P, 4, 8, None) == INVALID
    assert f(P, P, P, 4, 6, None) == MISALIGNED
    assert f(P, P + 2, P, 4, 8, None) == MISALIGNED


def test_python_binding_raises(lib):
    with pytest.raises(swg.SwgError) as e:
        swg.gemm(0, 0, -1, 1, 1, 1.0, P, 8, P, 8, 0.0, P, 8, swg.BF16, stream=0)
    assert e.value.status == INVALID


def test_shutdown_is_idempotent(lib):
    swg.shutdown()
    swg.shutdown()


def test_selftest_timeout_argument_checks(lib):
    assert lib.swg_selftest_wait_timeout(0, None) == INVALID
    assert lib.swg_selftest_wait_timeout(-5, None) == INVALID
    assert lib.swg_selftest_wait_timeout(2_000_000_000, None) == INVALID


def test_noalloc_rejects_bad_arguments_before_any_cuda_call(lib):
    """gemm_splitk_noalloc validates exactly as gemm_ex does, before its
    once-per-device set-up, so argument errors are reported without a GPU."""
    def n(**kw):
        a = dict(tA=0, tB=0, M=64, N=4096, K=16384, A=P, lda=16384, B=P, ldb=4096, C=P,
                 ldc=4096, dtype=1, split_k=0)
        a.update(kw)
        return lib.gemm_splitk_noalloc(a["tA"], a["tB"], a["M"], a["N"], a["K"],
                                       ctypes.c_float(1.0), a["A"], a["lda"], a["B"], a["ldb"],
                                       ctypes.c_float(1.0), a["C"], a["ldc"], a["dtype"],
                                       a["split_k"], None)
    assert n(M=-1) == INVALID
    assert n(split_k=-2) == INVALID
    assert n(tA=2) == INVALID
    assert n(A=0) == INVALID
    assert n(ldc=4000) == INVALID
    assert n(dtype=9) == UNSUPPORTED
    assert n(C=P + 8) == MISALIGNED
    assert n(lda=16388) == MISALIGNED
    assert n(M=0) == OK and n(N=0) == OK
    # e4m3 rules are gemm_ex's too: op(A) = A and op(B) = B^T only
    assert n(dtype=4, tB=0, ldb=16384) == UNSUPPORTED


def test_debug_workspace_guards_needs_an_output(lib):
    assert lib.swg_debug_workspace_guards(None, None) == INVALID
