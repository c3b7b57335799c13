"""ctypes binding of libfgemm.so: the C ABI of include/fgemm.h under the same names.

Argument marshalling only: pointers are taken from ints, torch tensors
(``data_ptr()``) or numpy arrays; the stream from an int, a ``torch.cuda.Stream``
or, by default, torch's current stream.  Every status other than FGEMM_OK raises
``FgemmError``.  There is no fallback: if the library is missing this module
raises on first use.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfgemm.so")

# dtype word (include/fgemm.h)
F16, BF16, E4M3 = 0x1, 0x2, 0x3
BIAS_SAME, BIAS_F32, BIAS_BF16 = 0x00, 0x10, 0x20
OUT_SAME, OUT_F32, OUT_E4M3, OUT_BF16, OUT_F16 = 0x000, 0x100, 0x200, 0x300, 0x400
Y_SAME, Y_F16, Y_BF16 = 0x0000, 0x1000, 0x2000

# status codes
OK, ERR_INVALID_VALUE, ERR_UNSUPPORTED_DTYPE, ERR_MISALIGNED = 0, 1, 2, 3
ERR_NO_DEVICE, ERR_LAUNCH, ERR_TIMEOUT, ERR_WORKSPACE = 4, 5, 6, 7

# epilogue codes (fgemm_plan)
EPI_RELU, EPI_GATE, EPI_RESIDUAL_RELU, EPI_RELU_QUANT = 0, 1, 2, 3

# paths
PATH_AUTO, PATH_TC, PATH_SKINNY, PATH_GENERIC, PATH_KZERO, PATH_NONE = 0, 1, 2, 3, 4, 5
PATH_NAMES = {PATH_TC: "tc", PATH_SKINNY: "skinny", PATH_GENERIC: "generic",
              PATH_KZERO: "kzero", PATH_NONE: "none"}


class FgemmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {fgemm_status_string(status)} ({status})")


class Opts(ctypes.Structure):
    """fgemm_opts: zero fields mean defaults."""
    _fields_ = [("group_m", ctypes.c_int), ("path", ctypes.c_int), ("split_k", ctypes.c_int),
                ("max_ctas", ctypes.c_int), ("timeout_ms", ctypes.c_int),
                ("cta_pair", ctypes.c_int), ("tail_split", ctypes.c_int),
                ("skinny_tiles", ctypes.c_int), ("stages", ctypes.c_int),
                ("inject_stall", ctypes.c_int), ("bias_init", ctypes.c_int),
                ("full_last_n", ctypes.c_int), ("y_blocks", ctypes.c_int),
                ("k_rows", ctypes.c_int), ("bias_mma", ctypes.c_int), ("pdl", ctypes.c_int),
                ("raster", ctypes.c_int), ("epi_warps", ctypes.c_int)]


class PlanInfo(ctypes.Structure):
    """fgemm_plan_info."""
    _fields_ = [("path", ctypes.c_int), ("grid", ctypes.c_int), ("cluster", ctypes.c_int),
                ("tiles", ctypes.c_int), ("work_items", ctypes.c_int), ("tail_split", ctypes.c_int),
                ("resident_pairs", ctypes.c_int), ("last_tile_n", ctypes.c_int),
                ("y_blocks", ctypes.c_int), ("k_rows", ctypes.c_int), ("row_barriers", ctypes.c_int),
                ("bias_init", ctypes.c_int), ("epi_warps", ctypes.c_int)]


_lock = threading.Lock()
_lib = None
_vp, _i64, _int, _sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
_SIGS = {
    "fgemm_bias_relu": (_int, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _vp]),
    "fgemm_addmm_gate": (_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _vp]),
    "fgemm_bias_residual_relu": (_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _vp]),
    "fgemm_bias_residual_relu_ex": (_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _vp,
                                           ctypes.POINTER(Opts), ctypes.POINTER(_int)]),
    "fgemm_bias_relu_quant": (_int, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, ctypes.c_float,
                                     _vp]),
    "fgemm_bias_relu_quant_ex": (_int, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, ctypes.c_float,
                                        _vp, ctypes.POINTER(Opts), ctypes.POINTER(_int)]),
    "fgemm_bias_relu_ex": (_int, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _vp,
                                  ctypes.POINTER(Opts), ctypes.POINTER(_int)]),
    "fgemm_addmm_gate_ex": (_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _vp,
                                   ctypes.POINTER(Opts), ctypes.POINTER(_int)]),
    "fgemm_unfused_workspace_bytes": (_sz, [_i64, _i64, _int, _int]),
    "fgemm_unfused_bias_relu": (_int, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _vp, _sz,
                                       _int, _vp]),
    "fgemm_unfused_addmm_gate": (_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _vp,
                                        _sz, _int, _vp]),
    "fgemm_unfused_bias_relu_noalloc": (_int, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _int,
                                               _vp]),
    "fgemm_device_status": (_int, [_vp, ctypes.POINTER(_int)]),
    "fgemm_status_string": (ctypes.c_char_p, [_int]),
    "fgemm_plan": (_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _int,
                          ctypes.POINTER(Opts), ctypes.POINTER(PlanInfo)]),
    "fgemm_plan_on": (_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _int,
                             ctypes.POINTER(Opts), _int, _int, ctypes.POINTER(PlanInfo)]),
    "fgemm_tile_of": (_int, [_i64, _i64, _i64, _int, ctypes.POINTER(_i64), ctypes.POINTER(_i64)]),
}


def lib():
    """Load libfgemm.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with gemm_epilogue_gb300.build.build()")
            handle = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIGS.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
    return _lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):
        return x.ctypes.data
    raise TypeError(f"cannot take a pointer of {type(x)}")


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(st: int, where: str) -> None:
    if st != OK:
        raise FgemmError(st, where)


def _opts(opts) -> Opts | None:
    if opts is None or isinstance(opts, Opts):
        return opts
    o = Opts()
    fields = {name for name, _ in Opts._fields_}
    for k, v in dict(opts).items():
        if k not in fields:  # a misspelt key would otherwise be dropped without a word
            raise ValueError(f"unknown fgemm_opts field {k!r}")
        setattr(o, k, int(v))
    return o


def fgemm_status_string(status: int) -> str:
    return lib().fgemm_status_string(status).decode()


def fgemm_bias_relu(A, B, bias, out, M, N, K, dtype, stream=None) -> None:
    _check(lib().fgemm_bias_relu(_ptr(A), _ptr(B), _ptr(bias), _ptr(out), M, N, K, dtype,
                                 _stream(stream)), "fgemm_bias_relu")


def fgemm_addmm_gate(A, B, bias, Y, out, M, N, K, dtype, stream=None) -> None:
    _check(lib().fgemm_addmm_gate(_ptr(A), _ptr(B), _ptr(bias), _ptr(Y), _ptr(out), M, N, K,
                                  dtype, _stream(stream)), "fgemm_addmm_gate")


def fgemm_bias_residual_relu(A, B, bias, R, out, M, N, K, dtype, stream=None) -> None:
    _check(lib().fgemm_bias_residual_relu(_ptr(A), _ptr(B), _ptr(bias), _ptr(R), _ptr(out), M, N,
                                          K, dtype, _stream(stream)), "fgemm_bias_residual_relu")


def fgemm_bias_residual_relu_ex(A, B, bias, R, out, M, N, K, dtype, stream=None, opts=None) -> int:
    taken = ctypes.c_int(-1)
    o = _opts(opts)
    _check(lib().fgemm_bias_residual_relu_ex(_ptr(A), _ptr(B), _ptr(bias), _ptr(R), _ptr(out), M, N,
                                             K, dtype, _stream(stream),
                                             ctypes.byref(o) if o else None, ctypes.byref(taken)),
           "fgemm_bias_residual_relu_ex")
    return taken.value


def fgemm_bias_relu_quant(A, B, bias, out, M, N, K, dtype, scale, stream=None) -> None:
    _check(lib().fgemm_bias_relu_quant(_ptr(A), _ptr(B), _ptr(bias), _ptr(out), M, N, K, dtype,
                                       float(scale), _stream(stream)), "fgemm_bias_relu_quant")


def fgemm_bias_relu_quant_ex(A, B, bias, out, M, N, K, dtype, scale, stream=None, opts=None) -> int:
    taken = ctypes.c_int(-1)
    o = _opts(opts)
    _check(lib().fgemm_bias_relu_quant_ex(_ptr(A), _ptr(B), _ptr(bias), _ptr(out), M, N, K, dtype,
                                          float(scale), _stream(stream),
                                          ctypes.byref(o) if o else None, ctypes.byref(taken)),
           "fgemm_bias_relu_quant_ex")
    return taken.value


def fgemm_bias_relu_ex(A, B, bias, out, M, N, K, dtype, stream=None, opts=None) -> int:
    """Returns the path that ran (PATH_*)."""
    taken = ctypes.c_int(-1)
    o = _opts(opts)
    _check(lib().fgemm_bias_relu_ex(_ptr(A), _ptr(B), _ptr(bias), _ptr(out), M, N, K, dtype,
                                    _stream(stream), ctypes.byref(o) if o else None,
                                    ctypes.byref(taken)), "fgemm_bias_relu_ex")
    return taken.value


def fgemm_addmm_gate_ex(A, B, bias, Y, out, M, N, K, dtype, stream=None, opts=None) -> int:
    taken = ctypes.c_int(-1)
    o = _opts(opts)
    _check(lib().fgemm_addmm_gate_ex(_ptr(A), _ptr(B), _ptr(bias), _ptr(Y), _ptr(out), M, N, K,
                                     dtype, _stream(stream), ctypes.byref(o) if o else None,
                                     ctypes.byref(taken)), "fgemm_addmm_gate_ex")
    return taken.value


def fgemm_unfused_workspace_bytes(M, N, dtype, inter_f32=0) -> int:
    return int(lib().fgemm_unfused_workspace_bytes(M, N, dtype, int(inter_f32)))


def fgemm_unfused_bias_relu(A, B, bias, out, M, N, K, dtype, workspace, workspace_bytes,
                            inter_f32=0, stream=None) -> None:
    _check(lib().fgemm_unfused_bias_relu(_ptr(A), _ptr(B), _ptr(bias), _ptr(out), M, N, K, dtype,
                                         _ptr(workspace), workspace_bytes, int(inter_f32),
                                         _stream(stream)), "fgemm_unfused_bias_relu")


def fgemm_unfused_addmm_gate(A, B, bias, Y, out, M, N, K, dtype, workspace, workspace_bytes,
                             inter_f32=0, stream=None) -> None:
    _check(lib().fgemm_unfused_addmm_gate(_ptr(A), _ptr(B), _ptr(bias), _ptr(Y), _ptr(out), M, N,
                                          K, dtype, _ptr(workspace), workspace_bytes,
                                          int(inter_f32), _stream(stream)),
           "fgemm_unfused_addmm_gate")


# Size of the library's own intermediate array used by fgemm_unfused_bias_relu_noalloc.
NOALLOC_SCRATCH_BYTES = 16 << 20


def fgemm_unfused_bias_relu_noalloc(A, B, bias, out, M, N, K, dtype, inter_f32=0,
                                    stream=None) -> None:
    """Unfused bias + ReLU chain whose intermediate lives in the library's fixed device array
    (for callers that cannot allocate device memory); see include/fgemm.h."""
    _check(lib().fgemm_unfused_bias_relu_noalloc(_ptr(A), _ptr(B), _ptr(bias), _ptr(out), M, N,
                                                 K, dtype, int(inter_f32), _stream(stream)),
           "fgemm_unfused_bias_relu_noalloc")


def fgemm_device_status(stream=None) -> int:
    """Synchronise the stream; return (and clear) the device error word."""
    code = ctypes.c_int(0)
    _check(lib().fgemm_device_status(_stream(stream), ctypes.byref(code)), "fgemm_device_status")
    return code.value


def fgemm_plan(A, B, bias, Y, out, M, N, K, dtype, gate=False, opts=None, epilogue=None) -> dict:
    """Launch plan of a fused call (nothing is launched).  epilogue: EPI_* (default: gate or relu)."""
    info = PlanInfo()
    o = _opts(opts)
    epi = epilogue if epilogue is not None else (EPI_GATE if gate else EPI_RELU)
    _check(lib().fgemm_plan(_ptr(A), _ptr(B), _ptr(bias), _ptr(Y), _ptr(out), M, N, K, dtype,
                            epi, ctypes.byref(o) if o else None, ctypes.byref(info)),
           "fgemm_plan")
    return {name: getattr(info, name) for name, _ in PlanInfo._fields_}


def fgemm_plan_on(A, B, bias, Y, out, M, N, K, dtype, num_sms, resident_pairs, gate=False,
                  opts=None, epilogue=None) -> dict:
    """fgemm_plan for a device with `num_sms` SMs and `resident_pairs` resident CTA pairs,
    computed on the host (no GPU needed); the buffers (ints are fine) are checked for alignment."""
    info = PlanInfo()
    o = _opts(opts)
    epi = epilogue if epilogue is not None else (EPI_GATE if gate else EPI_RELU)
    _check(lib().fgemm_plan_on(_ptr(A), _ptr(B), _ptr(bias), _ptr(Y), _ptr(out), M, N, K, dtype,
                               epi, ctypes.byref(o) if o else None, num_sms, resident_pairs,
                               ctypes.byref(info)),
           "fgemm_plan_on")
    return {name: getattr(info, name) for name, _ in PlanInfo._fields_}


def fgemm_tile_of(t, tiles_m, tiles_n, group) -> tuple[int, int]:
    m, n = ctypes.c_int64(), ctypes.c_int64()
    _check(lib().fgemm_tile_of(t, tiles_m, tiles_n, group, ctypes.byref(m), ctypes.byref(n)),
           "fgemm_tile_of")
    return m.value, n.value


def call_status(name: str, *args) -> int:
    """Raw status of an entry point (for tests of argument validation)."""
    return getattr(lib(), name)(*args)
