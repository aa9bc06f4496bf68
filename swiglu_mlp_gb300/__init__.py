"""Python binding of ``libswiglu_mlp.so`` (C ABI in ``include/swiglu_mlp.h``).

Argument marshalling only: every step of the computation runs in the
library's CUDA kernels.  There is no fallback of any kind; if the shared
library has not been built this module raises on first use.

Functions with the C names take the C arguments (pointers may be given as
ints or as tensors, whose ``data_ptr()`` is used; ``stream`` may be a
``torch.cuda.Stream``, a raw handle, or None for the current torch stream).
Each raises :class:`SwgError` when the library returns a non-zero status.
The ``*_into`` helpers derive sizes and strides from row-major torch tensors.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "SwgError", "OP_N", "OP_T", "F16_F32OUT", "BF16", "F16", "BF16_F32OUT", "E4M3_BF16OUT",
    "E4M3_F32OUT", "swiglu_mlp_fp8",
    "gemm", "gemm_ex", "gemm_splitk_noalloc", "swiglu_mlp", "swiglu_mlp_dual", "swiglu_mlp_forward", "swiglu_interleave", "status_string",
    "get_device_error", "debug_workspace_guards", "launch_count", "shutdown", "gemm_into", "selftest_wait_timeout",
    "swiglu_mlp_into", "interleave_weights", "library_path", "load",
]

OP_N, OP_T = 0, 1
F16_F32OUT, BF16, F16, BF16_F32OUT, E4M3_BF16OUT, E4M3_F32OUT = 0, 1, 2, 3, 4, 5
STATUS = {0: "SWG_OK", 1: "SWG_ERR_INVALID_ARG", 2: "SWG_ERR_MISALIGNED",
          3: "SWG_ERR_UNSUPPORTED", 4: "SWG_ERR_CUDA", 5: "SWG_ERR_NO_MEMORY",
          6: "SWG_ERR_DEVICE_TIMEOUT"}

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libswiglu_mlp.so")
_lock = threading.Lock()
_lib = None


class SwgError(RuntimeError):
    """A non-zero status from the C ABI; for SWG_ERR_CUDA the message also
    names the CUDA error behind it (swg_last_cuda_error)."""

    def __init__(self, status: int, where: str, cuda_error: int = 0, cuda_name: str = ""):
        self.status = int(status)
        self.cuda_error = int(cuda_error)
        msg = f"{where}: {STATUS.get(self.status, 'SWG_ERR_UNKNOWN')} ({self.status})"
        if self.cuda_error:
            msg += f" [CUDA {self.cuda_error}: {cuda_name}]"
        super().__init__(msg)


def library_path() -> str:
    return _LIB_PATH


def load():
    """Loads the shared library (once).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(_LIB_PATH)
        i64, i32, f32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_void_p
        lib.gemm.argtypes = [i32, i32, i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64, i32, vp]
        lib.gemm.restype = i32
        lib.gemm_ex.argtypes = [i32, i32, i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64, i32,
                                i32, vp]
        lib.gemm_ex.restype = i32
        lib.gemm_splitk_noalloc.argtypes = [i32, i32, i64, i64, i64, f32, vp, i64, vp, i64,
                                            f32, vp, i64, i32, i32, vp]
        lib.gemm_splitk_noalloc.restype = i32
        lib.swiglu_mlp.argtypes = [vp, vp, vp, i64, i64, i64, vp]
        lib.swiglu_mlp.restype = i32
        lib.swiglu_mlp_fp8.argtypes = [vp, vp, vp, i64, i64, i64, f32, vp]
        lib.swiglu_mlp_fp8.restype = i32
        lib.swiglu_mlp_dual.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp]
        lib.swiglu_mlp_dual.restype = i32
        lib.swiglu_mlp_forward.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, f32, vp]
        lib.swiglu_mlp_forward.restype = i32
        lib.swiglu_interleave.argtypes = [vp, vp, vp, i64, i64, vp]
        lib.swiglu_interleave.restype = i32
        lib.swg_status_string.argtypes = [i32]
        lib.swg_status_string.restype = ctypes.c_char_p
        lib.swg_get_device_error.argtypes = [vp]
        lib.swg_get_device_error.restype = i32
        lib.swg_selftest_wait_timeout.argtypes = [i64, vp]
        lib.swg_selftest_wait_timeout.restype = i32
        lib.swg_launch_count.argtypes = []
        lib.swg_launch_count.restype = ctypes.c_uint64
        lib.swg_shutdown.argtypes = []
        lib.swg_shutdown.restype = None
        lib.swg_last_cuda_error.argtypes = []
        lib.swg_last_cuda_error.restype = i32
        lib.swg_cuda_error_name.argtypes = [i32]
        lib.swg_cuda_error_name.restype = ctypes.c_char_p
        lib.swg_debug_workspace_guards.argtypes = [vp, ctypes.POINTER(i64)]
        lib.swg_debug_workspace_guards.restype = i32
        _lib = lib
        return lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


_raw_stream = None    # torch's accessor of the current raw stream handle, once found


def _current_stream():
    """The calling thread's current torch stream on the current device as a
    raw handle (None without CUDA).  torch's raw accessor is used when it has
    one: building a torch.cuda.Stream object per call costs several
    microseconds of host time."""
    global _raw_stream
    import torch
    if _raw_stream is None:
        if not torch.cuda.is_available():
            return None
        get = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        _raw_stream = get if get is not None else (
            lambda dev: torch.cuda.current_stream(dev).cuda_stream)
    return _raw_stream(torch.cuda.current_device())


def _stream(s):
    if s is None:
        return _current_stream()
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(rc: int, where: str) -> int:
    if rc != 0:
        code, name = 0, ""
        if rc == 4:                     # SWG_ERR_CUDA
            code = load().swg_last_cuda_error()
            name = load().swg_cuda_error_name(code).decode()
        raise SwgError(rc, where, code, name)
    return rc


def gemm(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, dtype, stream=None):
    """D = alpha * op(A) op(B) + beta * C, in place over C (see the C header)."""
    return _check(load().gemm(int(transA), int(transB), int(M), int(N), int(K), float(alpha),
                              _ptr(A), int(lda), _ptr(B), int(ldb), float(beta), _ptr(C),
                              int(ldc), int(dtype), _stream(stream)), "gemm")


def gemm_ex(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, dtype, split_k,
            stream=None):
    return _check(load().gemm_ex(int(transA), int(transB), int(M), int(N), int(K), float(alpha),
                                 _ptr(A), int(lda), _ptr(B), int(ldb), float(beta), _ptr(C),
                                 int(ldc), int(dtype), int(split_k), _stream(stream)), "gemm_ex")


def gemm_splitk_noalloc(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, dtype,
                        split_k=0, stream=None):
    """Split-K GEMM that allocates no device memory: its partial sums live in
    a fixed array inside the library (see the C header for the size limit and
    the sharing rules)."""
    return _check(load().gemm_splitk_noalloc(int(transA), int(transB), int(M), int(N), int(K),
                                             float(alpha), _ptr(A), int(lda), _ptr(B), int(ldb),
                                             float(beta), _ptr(C), int(ldc), int(dtype),
                                             int(split_k), _stream(stream)),
                  "gemm_splitk_noalloc")


def swiglu_mlp(A, W_fused, Y, M, N, K, stream=None):
    """Y = SiLU(A W1) (.) (A W2) over the interleaved W_fused (see the C header)."""
    return _check(load().swiglu_mlp(_ptr(A), _ptr(W_fused), _ptr(Y), int(M), int(N), int(K),
                                    _stream(stream)), "swiglu_mlp")


def swiglu_mlp_fp8(A, W_fused_t, Y, M, N, K, scale, stream=None):
    """Y = SiLU(s A W1) (.) (s A W2) from e4m3 A [M, K] and the transposed
    interleaved e4m3 weight [2N, K] (see the C header)."""
    return _check(load().swiglu_mlp_fp8(_ptr(A), _ptr(W_fused_t), _ptr(Y), int(M), int(N),
                                        int(K), float(scale), _stream(stream)), "swiglu_mlp_fp8")


def swiglu_mlp_dual(A, W1, W2, Y, M, N, K, stream=None):
    """Y = SiLU(A W1) (.) (A W2) from separate K x N weights (see the C header)."""
    return _check(load().swiglu_mlp_dual(_ptr(A), _ptr(W1), _ptr(W2), _ptr(Y), int(M), int(N),
                                         int(K), _stream(stream)), "swiglu_mlp_dual")


def swiglu_mlp_forward(A, W_fused, W_down, Y, Out, M, N, K, beta=0.0, stream=None):
    """Out = (SiLU(A W1) (.) (A W2)) W_down + beta * Out (see the C header)."""
    return _check(load().swiglu_mlp_forward(_ptr(A), _ptr(W_fused), _ptr(W_down), _ptr(Y),
                                            _ptr(Out), int(M), int(N), int(K), float(beta),
                                            _stream(stream)), "swiglu_mlp_forward")


def swiglu_interleave(W1, W2, W_fused, K, N, stream=None):
    return _check(load().swiglu_interleave(_ptr(W1), _ptr(W2), _ptr(W_fused), int(K), int(N),
                                           _stream(stream)), "swiglu_interleave")


def status_string(status: int) -> str:
    return load().swg_status_string(int(status)).decode()


def get_device_error(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device error word."""
    return load().swg_get_device_error(_stream(stream))


def selftest_wait_timeout(limit_ns: int, stream=None) -> int:
    """Runs a kernel whose bounded wait is made to run out (see the C header)."""
    return _check(load().swg_selftest_wait_timeout(int(limit_ns), _stream(stream)),
                  "swg_selftest_wait_timeout")


def debug_workspace_guards(stream=None) -> int:
    """Changed guard bytes around the current device's split-K workspaces
    (only those created under SWG_TEST_WS_GUARD=1; see the C header)."""
    bad = ctypes.c_int64(0)
    _check(load().swg_debug_workspace_guards(_stream(stream), ctypes.byref(bad)),
           "swg_debug_workspace_guards")
    return int(bad.value)


def launch_count() -> int:
    return int(load().swg_launch_count())


def shutdown() -> None:
    load().swg_shutdown()


# ---------------------------------------------------------------- tensor helpers

def _dtype_code(in_dtype, out_dtype) -> int:
    import torch
    table = {(torch.float16, torch.float32): F16_F32OUT, (torch.bfloat16, torch.bfloat16): BF16,
             (torch.float16, torch.float16): F16, (torch.bfloat16, torch.float32): BF16_F32OUT}
    try:
        return table[(in_dtype, out_dtype)]
    except KeyError:
        raise SwgError(3, f"gemm_into: unsupported dtypes {in_dtype} -> {out_dtype}") from None


def _row_major_ld(t, name):
    if t.dim() != 2 or t.stride(1) != 1:
        raise SwgError(1, f"{name} must be a 2-D row-major tensor (unit column stride)")
    return t.stride(0)


def gemm_into(C, A, B, transA=0, transB=0, alpha=1.0, beta=0.0, split_k=None, stream=None):
    """C <- alpha * op(A) op(B) + beta * C for 2-D row-major tensors."""
    M = A.shape[1] if transA else A.shape[0]
    K = A.shape[0] if transA else A.shape[1]
    N = B.shape[0] if transB else B.shape[1]
    Kb = B.shape[1] if transB else B.shape[0]
    if Kb != K or tuple(C.shape) != (M, N) or A.dtype != B.dtype:
        raise SwgError(1, "gemm_into: inconsistent shapes or dtypes")
    code = _dtype_code(A.dtype, C.dtype)
    args = (transA, transB, M, N, K, alpha, A, _row_major_ld(A, "A"), B, _row_major_ld(B, "B"),
            beta, C, _row_major_ld(C, "C"), code)
    if split_k is None:
        gemm(*args, stream=stream)
    else:
        gemm_ex(*args, split_k, stream=stream)
    return C


def swiglu_mlp_into(Y, A, W_fused, stream=None):
    """Y <- SiLU(A W1) (.) (A W2) with W_fused the interleaved [K, 2N] weight."""
    M, K = A.shape
    N = W_fused.shape[1] // 2
    if W_fused.shape[0] != K or tuple(Y.shape) != (M, N):
        raise SwgError(1, "swiglu_mlp_into: inconsistent shapes")
    for t, n in ((A, "A"), (W_fused, "W_fused"), (Y, "Y")):
        if not t.is_contiguous():
            raise SwgError(1, f"swiglu_mlp_into: {n} must be contiguous")
    swiglu_mlp(A, W_fused, Y, M, N, K, stream=stream)
    return Y


def interleave_weights(W1, W2, stream=None):
    """W_fused[K, 2N] with even columns W1 (Gate) and odd columns W2 (Up)."""
    import torch
    K, N = W1.shape
    if tuple(W2.shape) != (K, N) or not (W1.is_contiguous() and W2.is_contiguous()):
        raise SwgError(1, "interleave_weights: W1, W2 must be contiguous and the same shape")
    Wf = torch.empty((K, 2 * N), dtype=W1.dtype, device=W1.device)
    swiglu_interleave(W1, W2, Wf, K, N, stream=stream)
    return Wf
