"""INT4 block-quantized mixture-of-experts FFN layer for NVIDIA GB300 (sm_103a).

The compute lives in a C-ABI CUDA library (csrc/, header include/qmoe.h);
`binding` is a thin ctypes layer over it with the same entry-point names.
Importing the package does not load the library; the binding does, and it
raises if the library is missing -- there is no CPU fallback.
"""

__all__ = ["binding", "synthetic"]


def __getattr__(name):
    if name in ("qmoe_route", "matmul_nbits", "qmoe_forward", "qmoe_dequant", "qmoe_rmsnorm",
                "qmoe_workspace_size", "qmoe_status_string", "QMoEError", "Workspace"):
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
