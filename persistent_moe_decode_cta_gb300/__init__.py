"""GB300-native persistent MoE decode megakernel.

The compute path lives in libmk.so (CUDA kernels for sm_103a behind the C ABI of
include/mk.h); `binding` is a thin ctypes layer over it (the library is loaded on
first use and its absence is an error) and `sol` holds the speed-of-light byte
arithmetic used to report bandwidth fractions.
"""
from . import binding, sol  # noqa: F401

__all__ = ["binding", "sol"]
