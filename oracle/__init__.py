"""Float64 CPU oracle for the product-VQ KV cache -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its binding) never does, and the two share no code.

The arithmetic lives in ``vq_oracle.c`` (plain C, float64); this package only
builds it with gcc and marshals numpy arrays through ctypes.
"""
from .oracle import (  # noqa: F401
    build,
    hadamard,
    encode,
    dequant,
    reconstruct,
    attend_rows,
    attend,
    lut_score,
    to_f16,
)
