"""fp64 CPU oracle for exact attention -- TEST INFRASTRUCTURE.

Only tests/, the smoke check and the bench's CPU-baseline leg may import this
package.  The product (the CUDA library and its binding) never does, and the
two share no code.  See attn_oracle.c for the definitions and the passages of
the pages each one follows.

Parity pins: every function here is pinned in tests/test_oracle_pins.py to
values the pages print, closed forms, invariants or library routines.
"""
from .oracle import (  # noqa: F401
    build_oracle,
    attn_fwd,
    attn_fwd_rows,
    attn_decode,
    attn_decode_rows,
    decode_chunk_states,
    decode_chunk_bounds,
    num_threads,
    attn_bwd,
    attn_bwd_kvheads,
)
