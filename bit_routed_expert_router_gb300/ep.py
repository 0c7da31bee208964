"""Expert-parallel split of one MoE layer over G ranks (one GPU each).

The layer's work is a set of units whose outputs add up to y:

  - routed unit e (picked expert e): gate_e * FFN_e(x), d values;
  - shared unit c (a contiguous chunk of the shared expert's int4 groups of
    its intermediate dimension): the down projection of GELU(gate) * up over
    that chunk's rows, d values (the shared FFN is the sum over its chunks).

Each unit's output is rounded once onto the 2^-32 grid and the grid values
are summed as int64, which is the clustered decode kernel's combine.  Integer
sums do not depend on their order or grouping, so any partition of the units
over ranks, followed by one integer all-reduce of the d-vector, gives the bits
a single rank gets.  This module holds the partition (which rank owns which
routed expert and which shared chunk) and the all-reduce; the units
themselves run in the decode kernels.

The pages run on one device and describe no multi-device split; this is the
plain expert-parallel reading of the per-layer step ("MoE needed parallel
work, reuse, and coarse overlap": the routed experts of a token are
independent units; the shared expert's rows are too).
"""

from __future__ import annotations

GRID_BITS = 32     # units round onto the 2^-32 grid (as in the clustered decode kernel)


def expert_owner(e: int, world: int) -> int:
    """Rank that holds routed expert e: experts are dealt round-robin, so a run
    of hot neighbouring experts spreads over the ranks."""
    if world < 1 or e < 0:
        raise ValueError("bad expert or world size")
    return e % world


def owned_experts(ids, rank: int, world: int) -> list[tuple[int, int]]:
    """(top-k position, expert) pairs of one token that `rank` computes."""
    return [(j, int(e)) for j, e in enumerate(ids) if expert_owner(int(e), world) == rank]


def shared_chunks(n_groups: int, rank: int, world: int) -> tuple[int, int]:
    """Half-open range of the shared expert's intermediate int4 groups (64 rows
    of gate/up each, 64 columns of down) that `rank` computes: contiguous,
    sizes differing by at most one."""
    if world < 1 or not 0 <= rank < world or n_groups < 0:
        raise ValueError("bad rank, world size or group count")
    base, extra = divmod(n_groups, world)
    g0 = rank * base + min(rank, extra)
    return g0, g0 + base + (1 if rank < extra else 0)


def allreduce_fixed(y_fixed, group=None):
    """Sums the ranks' int64 grid vectors in place (one all-reduce per layer and
    token: d values; 22.5 KB at d = 2816)."""
    import torch
    import torch.distributed as dist

    if y_fixed.dtype != torch.int64:
        raise TypeError("the layer partials are int64 values on the 2^-32 grid")
    dist.all_reduce(y_fixed, op=dist.ReduceOp.SUM, group=group)
    return y_fixed
