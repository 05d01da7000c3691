"""Peak-memory accounting for the fused top-K KL head.

The fused loss keeps no tokens x vocabulary tensor: besides the caller's
inputs and gradients it needs a workspace whose only vocabulary-sized parts are
two chunks of dZ (chunk_tokens x V, bf16), fixed in the number of tokens. The
dense comparison grid that the method avoids costs N x V elements (blog "Why
distillation recovery is expensive": a 4 x 201,088 x 32,768 bf16 teacher grid
is about 50 GB).
"""
from __future__ import annotations


def dense_grid_bytes(n_tokens: int, vocab: int, bytes_per_elem: int) -> int:
    """Bytes of one dense tokens x vocabulary grid."""
    return int(n_tokens) * int(vocab) * int(bytes_per_elem)
