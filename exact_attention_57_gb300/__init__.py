"""GB300 (sm_103a) exact-attention forward: a C-ABI CUDA library and its binding.

``fa`` is the ctypes binding of ``libfa.so`` (see include/fa.h); ``workloads``
draws the seeded synthetic inputs; ``build`` compiles the library in-tree.
"""
from . import fa, workloads  # noqa: F401
from .fa import (  # noqa: F401
    FaError,
    attention,
    fa_fwd,
    fa_fwd_host,
    fa_fwd_status,
    fa_set_test_hooks,
    fa_status_string,
    fa_version,
)
