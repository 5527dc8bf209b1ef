"""Row-sharded dense matrices: gather each matrix's update to one owner rank,
orthogonalise it there, scatter the result back.

Source: "Training a 1T-Parameter MoE on EU public infrastructure with PyTorch
and TorchTitan", section "FlexShard: Muon without communication".  Expert
matrices are owned whole by one rank and need no communication; the dense
matrices, which FSDP shards, are gathered to an owner rank for Newton-Schulz
and the result is sent back to the ranks that hold the shards (the page
overlaps this with the experts' Newton-Schulz).

Layout.  Matrix j (rows_j x cols_j) is split by rows over the ranks of the
process group the way torch.tensor_split splits: the first rows_j % world ranks
hold one row more.  Rank r holds rows [start_r, stop_r).  Matrix j is owned by
rank j % world.

One step, on every rank:
  1. momentum on the local shards (elementwise, so exactly the full matrix's
     rows);
  2. every update shard is padded to the largest shard and gathered to the
     owner;
  3. the owner runs Newton-Schulz on the full update;
  4. the owner scatters the orthogonalised rows back (padded, trimmed on
     arrival);
  5. the parameter update on the local shards, with the full matrix's shape
     scale.
With one rank there are no collectives.  Steps 1, 3 and 5 are the library's C
calls, so the result equals, bit for bit, the single-process step on the full
matrices given the same fp32 shape scale.  The calls run on the current CUDA stream; to overlap them with the
experts' Newton-Schulz, call this under another stream.

Argument marshalling and torch.distributed plumbing only: the arithmetic runs
in the library's kernels (or, in tests of the data movement alone, in the
operations passed as `ops`).
"""

from __future__ import annotations

import dataclasses
import math
from typing import Callable, Sequence

QUINTIC = (3.4445, -4.7750, 2.0315)


def row_splits(rows: int, world: int) -> list:
    """[(start, stop)] of each rank's rows, as torch.tensor_split splits."""
    if rows < 0 or world < 1:
        raise ValueError("rows >= 0 and world >= 1 required")
    base, extra = divmod(rows, world)
    out, start = [], 0
    for r in range(world):
        n = base + (1 if r < extra else 0)
        out.append((start, start + n))
        start += n
    return out


def owner_of(index: int, world: int) -> int:
    """The rank that orthogonalises matrix `index`."""
    return index % world


def default_scale(rows: int, cols: int) -> float:
    """sqrt(max(1, rows/cols)) of the full matrix (the library's default)."""
    return math.sqrt(max(1.0, rows / cols))


@dataclasses.dataclass
class Ops:
    """The three operations of a step on one matrix (or shard)."""
    momentum: Callable   # (grad, momentum, update_out) -> None, in place
    ns: Callable         # (X) -> None, in place on the full matrix
    apply: Callable      # (param, update, scale) -> None, in place


def library_ops(*, mu: float, nesterov: bool, steps: int, coeffs, eps: float, lr: float,
                weight_decay: float) -> Ops:
    """The library's calls (bf16 parameters and updates, fp32 momentum)."""
    from . import muon_apply_update, muon_momentum_update, muon_ns_batched

    return Ops(
        momentum=lambda g, m, u: muon_momentum_update(g, m, u, mu, nesterov),
        ns=lambda x: muon_ns_batched(x, steps, coeffs, eps),
        apply=lambda p, o, sc: muon_apply_update(p, o, lr, weight_decay, sc),
    )


def dense_step(params: Sequence, grads: Sequence, momenta: Sequence, shapes: Sequence, *, group=None,
               mu: float = 0.95, nesterov: bool = True, steps: int = 5, coeffs=QUINTIC, eps: float = 1e-7,
               lr: float = 0.02, weight_decay: float = 0.1, scale: float = 0.0, ops: Ops | None = None) -> None:
    """One Muon step on row-sharded dense matrices, in place on this rank's shards.

    params, grads, momenta: this rank's shards, one 2-D tensor per matrix
    (its rows of matrix j, all columns); shapes: the full (rows_j, cols_j).
    group: the torch.distributed process group the matrices are sharded over
    (None: the default group if one is initialised, else a single rank).
    scale <= 0 selects sqrt(max(1, rows_j/cols_j)) of the full matrix.
    """
    import torch
    import torch.distributed as dist

    if not (len(params) == len(grads) == len(momenta) == len(shapes)):
        raise ValueError("params, grads, momenta and shapes must have one entry per matrix")
    distributed = dist.is_available() and dist.is_initialized()
    world = dist.get_world_size(group) if distributed else 1
    rank = dist.get_rank(group) if distributed else 0
    if ops is None:
        ops = library_ops(mu=mu, nesterov=nesterov, steps=steps, coeffs=coeffs, eps=eps, lr=lr,
                          weight_decay=weight_decay)

    def global_rank(r):
        return dist.get_global_rank(group, r) if group is not None else r

    for j, ((rows, cols), p, g, m) in enumerate(zip(shapes, params, grads, momenta)):
        splits = row_splits(rows, world)
        lo, hi = splits[rank]
        if tuple(p.shape) != (hi - lo, cols) or p.shape != g.shape or p.shape != m.shape:
            raise ValueError(f"matrix {j}: this rank's shard must be {(hi - lo, cols)}")
    outs = []
    for j, ((rows, cols), g, m) in enumerate(zip(shapes, grads, momenta)):
        splits = row_splits(rows, world)
        lo, hi = splits[rank]
        u = torch.empty_like(g)
        ops.momentum(g, m, u)
        if world == 1:
            ops.ns(u)
            outs.append(u)
            continue
        owner = owner_of(j, world)
        pad = max(b - a for a, b in splits)
        send = torch.zeros((pad, cols), dtype=u.dtype, device=u.device)
        send[: hi - lo] = u
        gathered = [torch.empty_like(send) for _ in range(world)] if rank == owner else None
        dist.gather(send, gathered, dst=global_rank(owner), group=group)
        pieces = None
        if rank == owner:
            full = torch.cat([gathered[r][: b - a] for r, (a, b) in enumerate(splits)]).contiguous()
            ops.ns(full)
            pieces = []
            for a, b in splits:
                piece = torch.zeros_like(send)
                piece[: b - a] = full[a:b]
                pieces.append(piece)
        recv = torch.empty_like(send)
        dist.scatter(recv, pieces, src=global_rank(owner), group=group)
        outs.append(recv[: hi - lo].contiguous())
    for (rows, cols), p, o in zip(shapes, params, outs):
        ops.apply(p, o, scale if scale > 0 else default_scale(rows, cols))
