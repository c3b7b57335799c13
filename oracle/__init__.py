"""fp64 CPU oracle for the fused GEMM + epilogue -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library and its
Python binding) never imports, links or calls it, and it imports nothing from
the product.

The arithmetic lives in ``oracle.c`` (plain C, fp64, threads over output
rows); this module compiles it with gcc and marshals numpy arrays through
ctypes.  ``schedule.py`` holds the grouped tile ordering written from the page
"I3. Fuse a GEMM epilogue and change tile scheduling".

Element types are passed as codes: F16 = 1, BF16 = 2, F32 = 3, E4M3 = 4.  16-bit
values are numpy ``uint16`` arrays holding the raw bit patterns, fp8 e4m3 values
``uint8`` bit patterns; F32 is ``float32``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

F16, BF16, F32, E4M3 = 1, 2, 3, 4
EPI_RELU, EPI_GATE, EPI_LINEAR, EPI_RESIDUAL, EPI_QUANT = 0, 1, 2, 3, 4

# Negative controls: deliberate mistakes the oracle can be asked to make, so
# that the tests can show each pin rejects a plausible slip.  OK = the oracle.
OK = 0
MUT_RELU_FIRST, MUT_BIAS_ROW, MUT_BIAS_IN_SUM, MUT_DROP_GEMM = 1, 2, 3, 4
MUT_TRANSPOSE_B, MUT_DROP_LAST_K, MUT_GATE_SIGN, MUT_RESID_AFTER = 5, 6, 7, 8
MUT_SCALE_FIRST = 9
MUTANTS = {"relu_first": MUT_RELU_FIRST, "bias_row": MUT_BIAS_ROW,
           "bias_in_sum": MUT_BIAS_IN_SUM, "drop_gemm": MUT_DROP_GEMM,
           "transpose_b": MUT_TRANSPOSE_B, "drop_last_k": MUT_DROP_LAST_K,
           "gate_sign": MUT_GATE_SIGN, "resid_after": MUT_RESID_AFTER,
           "scale_first": MUT_SCALE_FIRST}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into _oracle.so (gcc, -O3, no fast-math, no FP contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O3", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
             "-shared", "-pthread", _SRC, "-o", tmp, "-lm"],
            check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            lib.orc_gemm_epilogue.restype = ctypes.c_int
            lib.orc_gemm_epilogue.argtypes = (
                [ctypes.c_void_p] * 7
                + [ctypes.c_int64] * 3 + [ctypes.c_void_p, ctypes.c_int64]
                + [ctypes.c_int] * 6 + [ctypes.c_double, ctypes.c_int])
            lib.orc_encode.restype = None
            lib.orc_encode.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int]
            lib.orc_decode.restype = None
            lib.orc_decode.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int]
            _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def _ptr(a):
    return None if a is None else a.ctypes.data


def _storage(t):
    return {F32: np.float32, E4M3: np.uint8}.get(t, np.uint16)


def _bits(a, t):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    want = _storage(t)
    if a.dtype != want:
        raise TypeError(f"oracle expects {np.dtype(want)} storage for type code {t}, got {a.dtype}")
    return a


def encode(x, t: int) -> np.ndarray:
    """Round fp64 values to type ``t`` (RNE), returning raw bits (uint16) or float32."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=_storage(t))
    _load().orc_encode(_ptr(x), _ptr(out), x.size, t)
    return out


def decode(a, t: int) -> np.ndarray:
    """Decode raw bits (uint16) or float32 of type ``t`` to fp64."""
    a = _bits(a, t)
    out = np.empty(a.shape, dtype=np.float64)
    _load().orc_decode(_ptr(a), _ptr(out), a.size, t)
    return out


class Result:
    """Rounded output, the unrounded fp64 value, and sum_k |A B| per element."""

    def __init__(self, out, ref, absdot, threads):
        self.out = out          # rounded to the output type (bits or float32)
        self.ref = ref          # fp64 value before the final rounding
        self.absdot = absdot    # fp64 sum of |A[i,k] B[k,j]|
        self.threads = threads  # threads the oracle used


def gemm_epilogue(A, B, bias, M: int, N: int, K: int, ab_type: int, bias_type: int,
                  out_type: int, epi: int, Y=None, rows=None, threads: int | None = None,
                  want_ref: bool = True, mutant: int = OK, scale: float = 1.0,
                  y_type: int | None = None) -> Result:
    """Run the oracle on all rows, or on the listed ``rows`` of the M x N output.  ``y_type`` is
    the element type of the gate's Y (or the residual R); by default the operand type."""
    y_type = ab_type if y_type is None else y_type
    A = _bits(A, ab_type) if K > 0 else (None if A is None else _bits(A, ab_type))
    B = _bits(B, ab_type) if K > 0 else (None if B is None else _bits(B, ab_type))
    bias = _bits(bias, bias_type)
    if epi in (EPI_GATE, EPI_RESIDUAL):
        Y = _bits(Y, y_type)
    if rows is None:
        nrows, rows_arr = M, None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        if rows_arr.size and (rows_arr.min() < 0 or rows_arr.max() >= M):
            raise IndexError("row index out of range")
        nrows = rows_arr.size
    out = np.empty((nrows, N), dtype=_storage(out_type))
    ref = np.empty((nrows, N), dtype=np.float64) if want_ref else None
    absdot = np.empty((nrows, N), dtype=np.float64) if want_ref else None
    th = threads or default_threads()
    used = _load().orc_gemm_epilogue(
        _ptr(A), _ptr(B), _ptr(bias), _ptr(Y if epi in (EPI_GATE, EPI_RESIDUAL) else None),
        _ptr(out), _ptr(ref), _ptr(absdot), M, N, K, _ptr(rows_arr), nrows,
        ab_type, bias_type, out_type, y_type, epi, mutant, float(scale), th)
    if used < 0:
        raise ValueError("oracle rejected its arguments")
    return Result(out, ref, absdot, used)


def bias_relu(A, B, bias, M, N, K, ab_type, bias_type, out_type, **kw) -> Result:
    """out = RNE(max(0, A @ B + bias)) -- fp64 sum, bias once after the sum."""
    return gemm_epilogue(A, B, bias, M, N, K, ab_type, bias_type, out_type, EPI_RELU, **kw)


def addmm_gate(A, B, bias, Y, M, N, K, ab_type, bias_type, out_type, **kw) -> Result:
    """X = A @ B + bias;  out = RNE(X + X * Y) -- X never rounded before the gate."""
    return gemm_epilogue(A, B, bias, M, N, K, ab_type, bias_type, out_type, EPI_GATE, Y=Y, **kw)


def bias_residual_relu(A, B, bias, R, M, N, K, ab_type, bias_type, out_type, **kw) -> Result:
    """out = RNE(max(0, A @ B + bias + R)) -- the residual added before the activation."""
    return gemm_epilogue(A, B, bias, M, N, K, ab_type, bias_type, out_type, EPI_RESIDUAL, Y=R, **kw)


def bias_relu_quant(A, B, bias, M, N, K, ab_type, bias_type, scale, **kw) -> Result:
    """out = e4m3(clamp(scale * max(0, A @ B + bias), -448, 448)), fp8 output (uint8 bits)."""
    return gemm_epilogue(A, B, bias, M, N, K, ab_type, bias_type, E4M3, EPI_QUANT, scale=scale, **kw)


def linear(A, B, bias, M, N, K, ab_type, bias_type, out_type, **kw) -> Result:
    """out = RNE(A @ B + bias) with no activation."""
    return gemm_epilogue(A, B, bias, M, N, K, ab_type, bias_type, out_type, EPI_LINEAR, **kw)
