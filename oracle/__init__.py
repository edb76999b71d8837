"""fp64 CPU oracle (test infrastructure; never imported by the product path)."""
from .attention_oracle import (  # noqa: F401
    backward,
    backward_batched,
    backward_cols,
    backward_rows,
    bob,
    bob_batched,
    bob_cols,
    bob_rows,
    default_row_block,
    forward,
    forward_batched,
    forward_rows,
)
