"""Exact tiled attention for GB300 (sm_103a).

The compute path is the C-ABI library ``lib/libfa.so`` (hand-written CUDA
kernels, declared in ``include/fa.h``); ``fa`` is its ctypes binding, and
``workloads`` draws the seeded synthetic inputs.  Importing the package does
not load the library; the first call into ``fa`` does, and fails loudly if it
was not built.
"""

from .build import LIB_PATH, build_library  # noqa: F401
