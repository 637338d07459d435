"""Fused nested 4-bit weight dequantization for NVIDIA GB300 (sm_103a).

The computation lives in the CUDA library ``libdq4.so`` (C ABI in
``include/dq4.h``); this package is its thin Python binding.  The first use
of the library raises ImportError if it has not been built (see ``build``):
there is no CPU fallback.
"""

from ._binding import (  # noqa: F401
    OUT_BF16,
    OUT_F16,
    OUT_F32,
    Dq4Error,
    dq4,
    dq4_nested,
    dq4_nested_host,
    dq4_nested_transposed,
    dq4_nested_unfused,
    dq4_nested_unfused_static,
    get_lib,
    int8_correction_prep,
    linear,
    out_prod,
    sizes,
)


def __getattr__(name):
    if name == "lib":
        return get_lib()
    raise AttributeError(name)


__all__ = ["dq4_nested", "dq4_nested_host", "dq4_nested_transposed", "dq4",
           "dq4_nested_unfused", "dq4_nested_unfused_static", "Dq4Error", "get_lib", "sizes",
           "int8_correction_prep", "out_prod", "linear", "OUT_F16", "OUT_BF16", "OUT_F32"]
