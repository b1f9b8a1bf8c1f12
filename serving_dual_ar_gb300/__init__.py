"""GB300-native Dual-AR frame decode (Fish Audio S2 shape).

The compute path is libs2.so (hand-written sm_103a CUDA kernels plus a C++
host runtime) behind the C ABI in include/s2.h and include/s2_ops.h;
``binding`` exposes those calls to Python under the same names.  Importing
the binding loads the library and raises if it is missing.
"""

__all__ = ["build", "binding"]


def build(force=False):
    from . import buildlib as _b
    return _b.build(force=force)
