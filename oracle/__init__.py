"""Test infrastructure only: the fp64 CPU oracle for exact attention.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package. The product (the CUDA library under
``exact_io_aware_108_b300/`` and its binding) never imports it, and the two
share no code: inputs reach the oracle as plain arrays.

The arithmetic lives in ``attention_ref.c`` (plain C, double precision);
``ref.py`` is the ctypes loader.
"""
from .ref import (  # noqa: F401
    attn_fwd,
    attn_fwd_rows,
    attn_bwd,
    attn_bwd_sampled,
    build,
    library_path,
)
