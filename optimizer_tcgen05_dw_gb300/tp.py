"""Column-parallel (output-feature) tensor parallelism for the FORGE step.

FORGE explainer ("FORGE: Fused On-Register Gradient Elimination for
Memory-Efficient LLM Training", gist.science), Technical Summary §2
"Distributed Training Compatibility": under tensor parallelism each device
already holds the complete gradient of its own weight shard when the backward
pass reaches the layer, so the fused step stays exact there (data
parallelism, which would first need the gradients of all replicas summed, is
what the method cannot serve).

Layout for P ranks, W [N x K] split by rows (output features):

* rank r owns rows [r N/P, (r+1) N/P) of W and of its optimizer states, the
  same columns of dY (what its share of the forward pass produced) and a
  replica of X;
* its step is ``forge_linear_bwd_step_shard`` on those rows: the weight
  update needs nothing from the other ranks, and stochastic rounding draws
  the bits of the rows' indices in the whole matrix, so P shards reproduce
  the one-device step's weights and states bit for bit;
* the one exchange is the input gradient: each shard yields the partial
  dX_r = dY_r W_r, and dX = sum over r of dX_r, formed by an all-reduce.

This module holds the partition arithmetic and that reduction; the shard's
computation is the library's (or, in CPU tests of the partitioning, a
function the caller passes).
"""

import torch


def shard_rows(N: int, world: int, rank: int, align: int = 8):
    """(first row, row count) of rank `rank`'s equal shard of N rows.  Rows are
    split evenly and each shard's row count must be a multiple of `align` (8:
    the element-index groups of the stochastic rounding stay whole; 64 lets a
    shard use the one-launch step)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} of world {world}")
    if N % world != 0 or (N // world) % align != 0:
        raise ValueError(f"N = {N} rows do not split into {world} shards of a multiple of {align}")
    rows = N // world
    return rank * rows, rows


def shard(t: torch.Tensor, world: int, rank: int, dim: int = 0) -> torch.Tensor:
    """Rank `rank`'s contiguous copy of `t` split evenly along `dim` (rows of W
    and of the states: dim 0; columns of dY: dim 1)."""
    n = t.shape[dim]
    if n % world != 0:
        raise ValueError(f"dimension {dim} of size {n} does not split into {world} shards")
    size = n // world
    return t.narrow(dim, rank * size, size).contiguous()


def reduce_partial_dx(dX: torch.Tensor, group=None) -> torch.Tensor:
    """dX <- the sum over the group's ranks of their partial input gradients.

    The partials are summed in float32 and the sum rounded once to bf16 (to
    nearest even), in place.  Without an initialised process group (one
    rank) dX is left as it is."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size(group) == 1:
        return dX
    acc = dX.float()
    dist.all_reduce(acc, op=dist.ReduceOp.SUM, group=group)
    dX.copy_(acc)
    return dX


def column_parallel_bwd_step(X, dY_shard, W_shard, opt: str, hp: dict, step: int, seed: int,
                             s1=None, s2=None, s1_scale=None, s2_scale=None, dX=None,
                             world: int = 1, rank: int = 0, group=None, step_fn=None):
    """One rank's FORGE step of a column-parallel linear layer.

    W_shard and the states are this rank's equal row shard (rows
    [rank R, rank R + R), R = W_shard.shape[0]), dY_shard the matching
    columns of dY.  Updates them in place; if dX is given it receives the
    layer's whole input gradient (this shard's partial, then the all-reduce
    over `group`).  `step_fn` computes the shard (default: the library's
    forge_linear_bwd_step_shard); it takes the arguments of that binding."""
    if step_fn is None:
        from . import api
        step_fn = api.forge_linear_bwd_step_shard
    row_offset = rank * W_shard.shape[0]
    step_fn(X, dY_shard, W_shard, opt, hp, step, seed, row_offset, s1=s1, s2=s2,
            s1_scale=s1_scale, s2_scale=s2_scale, dX=dX)
    if dX is not None and world > 1:
        reduce_partial_dx(dX, group)
    return row_offset
