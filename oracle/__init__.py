"""CPU float64 oracle for exact attention (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package.  The product library never does.
"""
from .oracle import (  # noqa: F401
    build,
    attn_fwd,
    attn_rows,
    attn_probs,
    attn_fwd_online,
    attn_bwd,
    lib_path,
)
