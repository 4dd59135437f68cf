"""Expert-range sharding of a CSF stack across GPUs (one process per GPU).

The codec has no exchange step: experts, and the rows inside them, are
independent.  The page "Load native FP4 experts with optional lossless CSF
scales" notes that tensor-parallel workers compress their own slices
independently; an expert-parallel split is the same idea along the expert
axis.  Each rank owns a contiguous range of experts [e0, e1), prepares the CSF
stack of that sub-stack on its own GPU, and decodes it into a local
workspace.  Routing needs no rebasing: the grouped-routing prefix
`expert_start` (E + 1 entries) marks expert e active when
expert_start[e + 1] > expert_start[e], so the rank's routing view is the
slice expert_start[e0 : e1 + 1] -- the pointer expert_start + e0, no copy --
and its sub-stack decodes exactly the rows that the whole stack's routed
decode writes for those experts.

Host-side marshalling only: every byte of prepare and decode runs in the
library's kernels (csf.prepare, csf.decode).
"""
from __future__ import annotations


def expert_range(E: int, world: int, rank: int) -> tuple[int, int]:
    """Contiguous experts [e0, e1) of `rank` among `world` ranks: sizes differ
    by at most one, the larger ranges first, and the ranges partition [0, E)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside a world of {world}")
    if E < world:
        raise ValueError(f"{E} experts cannot give each of {world} ranks at least one")
    q, r = divmod(E, world)
    e0 = rank * q + min(rank, r)
    return e0, e0 + q + (1 if rank < r else 0)


def shard_dense(dense, e0: int, e1: int):
    """The rank's dense sub-stack: experts [e0, e1) of a [E, R, C] stack (a view)."""
    return dense[e0:e1]


def routing_view(expert_start, e0: int, e1: int):
    """The rank's routing: entries [e0, e1] of the grouped-routing prefix (a
    contiguous view, i.e. the pointer expert_start + e0 with e1 - e0 + 1
    entries).  Its differences are the sub-stack's per-expert token counts."""
    if expert_start.shape[0] < e1 + 1:
        raise ValueError("expert_start is shorter than E + 1 entries")
    return expert_start[e0:e1 + 1]


def prepare_shard(dense, kind: int, world: int, rank: int):
    """Prepare this rank's sub-stack of the whole [E, R, C] uint8 CUDA stack
    `dense` on its GPU.  Returns (stack, e0, e1)."""
    from . import csf
    e0, e1 = expert_range(int(dense.shape[0]), world, rank)
    return csf.prepare(shard_dense(dense, e0, e1).contiguous(), kind), e0, e1
