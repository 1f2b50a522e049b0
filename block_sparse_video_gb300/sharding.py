"""Head partition of one attention layer across ranks (host logic only).

"UniServe: serving FastH3 at its fastest", section "The FastH3 workload": the
56 attention heads of a layer are split across the GPUs of a sequence-parallel
group (14 per GPU under 4-way Ulysses). Every (batch, head) slice is
independent through the whole forward (pool, coarse branch, selection, fine
attention, gated combination), so a rank computes its heads with no exchange
inside the path. Each rank gets a contiguous range of heads; the ranges
differ in size by at most one head.
"""
from __future__ import annotations


def head_ranges(num_heads: int, world: int):
    """[(first_head, heads)] for ranks 0 .. world - 1: contiguous, in order,
    covering every head once. The first num_heads % world ranks take one head
    more. Needs 1 <= world <= num_heads (every rank gets a head)."""
    if num_heads < 1 or world < 1 or world > num_heads:
        raise ValueError(f"cannot split {num_heads} heads over {world} ranks")
    base, extra = divmod(num_heads, world)
    out, h0 = [], 0
    for r in range(world):
        n = base + (1 if r < extra else 0)
        out.append((h0, n))
        h0 += n
    return out
