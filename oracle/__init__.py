"""fp64 CPU oracle for exact attention -- test infrastructure, not the product.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports it and shares no code with it.
"""

from .attention import (  # noqa: F401
    backward,
    backward_head,
    backward_varlen,
    eligible,
    forward,
    forward_head,
    forward_rows,
    forward_varlen,
    score_matrix_payload_bytes,
    scores,
    tensor_payload_bytes,
)
