"""FP64 CPU oracle for the GEMM and fused-SwiGLU hot path.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The product library under
``swiglu_mlp_gb300/`` never imports this package, and this package imports
nothing from it.

The arithmetic lives in ``oracle.c`` (plain C, double precision); this module
only compiles it with gcc and marshals numpy arrays.  What each function
computes, with the passage it follows:

* :func:`gemm` — D = alpha * op(A) op(B) + beta * C_old, element by element,
  op = identity or transpose, row-major storage with a row stride
  ("GEMM o Coração Matemático", §1 and §2; C is not read when beta == 0, §2.1).
* :func:`swiglu` — Y = SiLU(A W1) (.) (A W2), SiLU(x) = x / (1 + e^-x), from
  SEPARATE W1 and W2 ("Sobreposição de Ativação em Nível de Tile para
  Inferência Eficiente de LLM", Definição do Problema; Metodologia, Kernel-2).
* :func:`interleave` — W_fused with even columns from W1 (Gate) and odd columns
  from W2 (Up) (same page, Metodologia, Kernel-2).
* :func:`mlp` — the full gated MLP, (SiLU(A W1) (.) (A W2)) W_down + beta * Out
  ("GEMM o Coração Matemático", §13.3, with the gated activation above).
* :func:`swiglu_typed`, :func:`interleave_t8` — the same SwiGLU on 8-bit
  (e4m3) operands with a per-tensor scale, and the transposed interleave the
  8-bit kernel reads ("GEMM o Coração Matemático", §12.4 on quantised operands
  with a scale; the e4m3 field layout is the OCP 8-bit floating-point E4M3
  format, which the pages do not define, pinned against torch's
  float8_e4m3fn).
* :func:`silu`, :func:`f16_to_f64`, :func:`bf16_to_f64`, :func:`e4m3_to_f64`,
  :func:`round_bf16` — the scalar pieces.

Every function is pinned by ``tests/test_oracle_pins.py`` against values and
properties fixed outside the oracle (the page's worked example, exact integer
brute force, algebraic identities, closed forms of SiLU, and numpy/torch
decoders for the storage formats).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

TYPES = {"f16": 0, "bf16": 1, "f32": 2, "e4m3": 3}


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` (gcc, no fast-math, no FMA
    contraction, so x86 and Arm hosts give identical doubles)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, f64, vp, i32 = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
            lib.orc_gemm.argtypes = [i32, i32, i64, i64, i64, f64, vp, i64, i32,
                                     vp, i64, i32, f64, vp, i64, i32, vp, i64, vp, i64,
                                     vp, i32]
            lib.orc_gemm.restype = i32
            lib.orc_swiglu.argtypes = [vp, i64, vp, vp, i64, i64, i64, i64, vp, i64, vp, i64,
                                       vp, i32]
            lib.orc_swiglu.restype = i32
            lib.orc_mlp.argtypes = [vp, vp, vp, vp, vp, f64, i64, i64, i64, vp, i64, vp, i32,
                                    i32]
            lib.orc_mlp.restype = i32
            lib.orc_swiglu_typed.argtypes = [vp, vp, vp, i32, f64, i64, i64, i64, vp, i64, vp,
                                             i64, vp, i32]
            lib.orc_swiglu_typed.restype = i32
            lib.orc_interleave_t8.argtypes = [vp, vp, vp, i64, i64]
            lib.orc_interleave_t8.restype = None
            lib.orc_e4m3_to_f64.argtypes = [ctypes.c_uint8]
            lib.orc_e4m3_to_f64.restype = f64
            lib.orc_interleave.argtypes = [vp, vp, vp, i64, i64]
            lib.orc_interleave.restype = None
            lib.orc_round_bf16.argtypes = [f64]
            lib.orc_round_bf16.restype = f64
            lib.orc_silu.argtypes = [f64]
            lib.orc_silu.restype = f64
            lib.orc_f16_to_f64.argtypes = [ctypes.c_uint16]
            lib.orc_f16_to_f64.restype = f64
            lib.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.orc_bf16_to_f64.restype = f64
            lib.orc_num_cores.restype = i32
            _lib = lib
    return _lib


def _as_buffer(x, kind: str) -> np.ndarray:
    """A C-contiguous numpy view of the stored values.  Half formats are passed
    as their 16-bit patterns (uint16/int16/float16 arrays, or torch tensors of
    dtype float16/bfloat16); f32 as float32."""
    if x is None:
        return None
    if hasattr(x, "detach"):               # a torch CPU tensor
        import torch
        t = x.detach().contiguous()
        if t.dtype in (torch.float16, torch.bfloat16):
            t = t.view(torch.int16)
        elif t.dtype == getattr(torch, "float8_e4m3fn", None):
            t = t.view(torch.uint8)
        x = t.numpy()
    a = np.ascontiguousarray(x)
    if kind == "e4m3":
        if a.dtype.itemsize != 1:
            raise TypeError(f"e4m3 operand must hold 8-bit patterns, got {a.dtype}")
        return a.view(np.uint8)
    if kind in ("f16", "bf16"):
        if a.dtype.itemsize != 2:
            raise TypeError(f"{kind} operand must hold 16-bit patterns, got {a.dtype}")
        return a.view(np.uint16)
    if a.dtype != np.float32:
        raise TypeError(f"f32 operand must be float32, got {a.dtype}")
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data


def _rows(rows, M):
    """Index subset (rows or columns) as int64, or (None, M) for all."""
    if rows is None:
        return None, M
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    if r.size and (r.min() < 0 or r.max() >= M):
        raise IndexError("index out of range")
    return r, int(r.size)


def gemm(transA: int, transB: int, M: int, N: int, K: int, alpha: float,
         A, lda: int, B, ldb: int, beta: float, C=None, ldc: int = 0,
         in_type: str = "bf16", c_type: str = "bf16", rows=None,
         threads: int = 0, cols=None) -> np.ndarray:
    """D = alpha * op(A) op(B) + beta * C_old in double; returns the rows
    ``rows`` (all when None) and columns ``cols`` (all when None) as a float64
    array of shape (len(rows), len(cols)).
    A is stored M x K (transA = 0) or K x M (transA = 1) with row stride lda;
    B is stored K x N (transB = 0) or N x K (transB = 1) with row stride ldb;
    C is M x N with row stride ldc and is not read when beta == 0."""
    lib = _load()
    a = _as_buffer(A, in_type)
    b = _as_buffer(B, in_type)
    c = _as_buffer(C, c_type) if beta != 0.0 else None
    r, n_rows = _rows(rows, M)
    cs, n_cols = _rows(cols, N)
    out = np.empty((n_rows, n_cols), dtype=np.float64)
    rc = lib.orc_gemm(int(transA), int(transB), M, N, K, float(alpha),
                      _ptr(a), lda, TYPES[in_type], _ptr(b), ldb, TYPES[in_type],
                      float(beta), _ptr(c), ldc, TYPES[c_type],
                      _ptr(r), n_rows, _ptr(cs), n_cols, out.ctypes.data, int(threads))
    if rc != 0:
        raise ValueError("oracle gemm rejected its arguments")
    return out


def swiglu(A, W1, W2, M: int, N: int, K: int, rows=None, threads: int = 0,
           lda: int | None = None, ldw: int | None = None, cols=None) -> np.ndarray:
    """Y = SiLU(A W1) (.) (A W2) in double, from bf16 A (M x K) and separate
    bf16 W1, W2 (K x N); returns float64 rows ``rows`` x columns ``cols`` (all
    when None)."""
    lib = _load()
    a = _as_buffer(A, "bf16")
    w1 = _as_buffer(W1, "bf16")
    w2 = _as_buffer(W2, "bf16")
    r, n_rows = _rows(rows, M)
    cs, n_cols = _rows(cols, N)
    out = np.empty((n_rows, n_cols), dtype=np.float64)
    rc = lib.orc_swiglu(_ptr(a), lda if lda is not None else K, _ptr(w1), _ptr(w2),
                        ldw if ldw is not None else N, M, N, K, _ptr(r), n_rows,
                        _ptr(cs), n_cols, out.ctypes.data, int(threads))
    if rc != 0:
        raise ValueError("oracle swiglu rejected its arguments")
    return out


def mlp(A, W1, W2, Wd, M: int, N: int, K: int, beta: float = 0.0, Out_old=None, rows=None,
        threads: int = 0, round_y: bool = False) -> np.ndarray:
    """Out = (SiLU(A W1) (.) (A W2)) W_down + beta * Out_old in double: A is
    M x K, W1 and W2 K x N, W_down N x K, Out_old M x K, all bf16 (Out_old read
    only when beta != 0).  The gated activation Y stays in double, or with
    round_y is rounded to bf16 (round-to-nearest-even, :func:`round_bf16`)
    before the down projection, as the product stores it."""
    lib = _load()
    a, w1, w2, wd = (_as_buffer(x, "bf16") for x in (A, W1, W2, Wd))
    o = _as_buffer(Out_old, "bf16") if beta != 0.0 else None
    r, n_rows = _rows(rows, M)
    out = np.empty((n_rows, K), dtype=np.float64)
    rc = lib.orc_mlp(_ptr(a), _ptr(w1), _ptr(w2), _ptr(wd), _ptr(o), float(beta), M, N, K,
                     _ptr(r), n_rows, out.ctypes.data, int(threads), 1 if round_y else 0)
    if rc != 0:
        raise ValueError("oracle mlp rejected its arguments")
    return out


def swiglu_typed(A, W1, W2, M: int, N: int, K: int, in_type: str = "e4m3",
                 scale: float = 1.0, rows=None, cols=None, threads: int = 0) -> np.ndarray:
    """Y = SiLU(scale * A W1) (.) (scale * A W2) in double for operands of
    storage type in_type (e.g. e4m3) with a per-tensor dequantisation scale."""
    lib = _load()
    a, w1, w2 = (_as_buffer(x, in_type) for x in (A, W1, W2))
    r, n_rows = _rows(rows, M)
    cs, n_cols = _rows(cols, N)
    out = np.empty((n_rows, n_cols), dtype=np.float64)
    rc = lib.orc_swiglu_typed(_ptr(a), _ptr(w1), _ptr(w2), TYPES[in_type], float(scale), M, N,
                              K, _ptr(r), n_rows, _ptr(cs), n_cols, out.ctypes.data,
                              int(threads))
    if rc != 0:
        raise ValueError("oracle swiglu_typed rejected its arguments")
    return out


def interleave_t8(W1, W2, K: int, N: int) -> np.ndarray:
    """2N x K uint8 patterns: row 2n = W1 column n, row 2n+1 = W2 column n."""
    lib = _load()
    w1 = _as_buffer(W1, "e4m3")
    w2 = _as_buffer(W2, "e4m3")
    out = np.empty((2 * N, K), dtype=np.uint8)
    lib.orc_interleave_t8(_ptr(w1), _ptr(w2), out.ctypes.data, K, N)
    return out


def e4m3_to_f64(bits: int) -> float:
    return _load().orc_e4m3_to_f64(int(bits) & 0xFF)


def interleave(W1, W2, K: int, N: int) -> np.ndarray:
    """W_fused (K x 2N uint16 bit patterns): even columns W1, odd columns W2."""
    lib = _load()
    w1 = _as_buffer(W1, "bf16")
    w2 = _as_buffer(W2, "bf16")
    out = np.empty((K, 2 * N), dtype=np.uint16)
    lib.orc_interleave(_ptr(w1), _ptr(w2), out.ctypes.data, K, N)
    return out


def round_bf16(x: float) -> float:
    """x rounded once to the nearest bfloat16 value, ties to even."""
    return _load().orc_round_bf16(float(x))


def silu(x: float) -> float:
    return _load().orc_silu(float(x))


def f16_to_f64(bits: int) -> float:
    return _load().orc_f16_to_f64(int(bits) & 0xFFFF)


def bf16_to_f64(bits: int) -> float:
    return _load().orc_bf16_to_f64(int(bits) & 0xFFFF)


def num_cores() -> int:
    return _load().orc_num_cores()
