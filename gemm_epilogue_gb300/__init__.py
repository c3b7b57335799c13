"""gemm_epilogue_gb300: fused GEMM + epilogue (bias + ReLU, addmm + GLU gate) for sm_103a.

The compute lives in a C-ABI CUDA library (``libfgemm.so``, see ``include/fgemm.h``);
``gemm_epilogue_gb300.binding`` is the thin ctypes binding with the same entry-point
names.  ``gemm_epilogue_gb300.inputs`` draws the seeded synthetic workloads.
"""
__all__ = ["binding", "inputs"]


def __getattr__(name):
    if name in __all__:
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
