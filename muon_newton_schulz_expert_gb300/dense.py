"""Row-sharded dense matrices: send each matrix's update to one owner rank,
orthogonalise it there, send the result back.

Source: "Training a 1T-Parameter MoE on EU public infrastructure with PyTorch
and TorchTitan", section "FlexShard: Muon without communication".  Expert
matrices are owned whole by one rank and need no communication; the dense
matrices, which FSDP shards, are gathered to an owner rank for Newton-Schulz
and the result is sent back to the ranks that hold the shards, overlapped
with the experts' Newton-Schulz.

Layout.  Matrix j (rows_j x cols_j) is split by rows over the ranks of the
process group the way torch.tensor_split splits: the first rows_j % world ranks
hold one row more.  Rank r holds rows [start_r, stop_r).  Matrix j is owned by
rank j % world.

One step, on every rank, per group of matrices of one shape:
  1. momentum on the local shards (elementwise, so exactly the full matrix's
     rows);
  2. one all-to-all: every rank sends each owner its shard of every matrix
     that owner holds in the group, padded to the largest shard;
  3. every owner stacks its full matrices of the group and orthogonalises
     them in one batched Newton-Schulz call;
  4. one all-to-all back: every owner returns each rank its rows of those
     matrices;
  5. the parameter update on the local shards, with the full matrix's shape
     scale (the library's default for the full shape, unless given).
With one rank there are no collectives.  Steps 1, 3 and 5 are the library's C
calls, so the result equals, bit for bit, the single-process step on the full
matrices given the same fp32 shape scale.

Streams.  Everything is enqueued on `stream` (default: the current CUDA
stream): the library's launches directly, the collectives through
torch.distributed, which orders them on the current stream.  Running
dense_step on a side stream while the experts' step runs on another lets the
two overlap on the GPU; the call itself returns once the work is enqueued
(the collectives may block the host until their peers join).

Argument marshalling and torch.distributed plumbing only: the arithmetic runs
in the library's kernels (or, in tests of the data movement alone, in the
operations passed as `ops`).
"""

from __future__ import annotations

import contextlib
import dataclasses
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


def shape_groups(shapes: Sequence) -> list:
    """[(shape, [matrix indices])], one entry per distinct shape, in order of first appearance."""
    groups: dict = {}
    for j, s in enumerate(shapes):
        groups.setdefault(tuple(s), []).append(j)
    return list(groups.items())


@dataclasses.dataclass
class Ops:
    """The operations of a step on one matrix (or shard), or one stack of full matrices."""
    momentum: Callable   # (grad, momentum, update_out) -> None, in place
    ns: Callable         # (X of shape (batch, rows, cols)) -> None, in place on full matrices
    apply: Callable      # (param, update, scale) -> None, in place
    scale: Callable      # (rows, cols) -> the default shape scale of a full rows x cols matrix


def library_ops(*, mu: float, nesterov: bool, steps: int, coeffs, eps: float, lr: float,
                weight_decay: float) -> Ops:
    """The library's calls (bf16 parameters and updates, fp32 momentum)."""
    from . import muon_apply_update, muon_default_scale, muon_momentum_update, muon_ns_batched

    return Ops(
        momentum=lambda g, m, u: muon_momentum_update(g, m, u, mu, nesterov),
        ns=lambda x: muon_ns_batched(x, steps, coeffs, eps),
        apply=lambda p, o, sc: muon_apply_update(p, o, lr, weight_decay, sc),
        scale=muon_default_scale,
    )


def dense_step(params: Sequence, grads: Sequence, momenta: Sequence, shapes: Sequence, *, group=None,
               mu: float = 0.95, nesterov: bool = True, steps: int = 5, coeffs=QUINTIC, eps: float = 1e-7,
               lr: float = 0.02, weight_decay: float = 0.1, scale: float = 0.0, ops: Ops | None = None,
               stream=None) -> None:
    """One Muon step on row-sharded dense matrices, in place on this rank's shards.

    params, grads, momenta: this rank's shards, one 2-D tensor per matrix
    (its rows of matrix j, all columns); shapes: the full (rows_j, cols_j).
    group: the torch.distributed process group the matrices are sharded over
    (None: the default group if one is initialised, else a single rank).
    scale <= 0 selects the library's default scale of the full matrix.
    stream: a torch.cuda.Stream to enqueue everything on (None: the current one).
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
    for j, ((rows, cols), p, g, m) in enumerate(zip(shapes, params, grads, momenta)):
        lo, hi = row_splits(rows, world)[rank]
        if tuple(p.shape) != (hi - lo, cols) or p.shape != g.shape or p.shape != m.shape:
            raise ValueError(f"matrix {j}: this rank's shard must be {(hi - lo, cols)}")

    ctx = torch.cuda.stream(stream) if stream is not None else contextlib.nullcontext()
    with ctx:
        outs = [None] * len(shapes)
        for (rows, cols), members in shape_groups(shapes):
            splits = row_splits(rows, world)
            lo, hi = splits[rank]
            upd = {}
            for j in members:
                u = torch.empty_like(grads[j])
                ops.momentum(grads[j], momenta[j], u)
                upd[j] = u
            if not distributed:
                # no process group: this process owns every matrix (an initialised
                # group, even of one rank, goes through the exchange below)
                full = torch.stack([upd[j] for j in members])
                ops.ns(full)
                for k, j in enumerate(members):
                    outs[j] = full[k]
                continue
            # matrices of the group by owner, in index order; every rank computes the same lists
            owned = [[j for j in members if owner_of(j, world) == o] for o in range(world)]
            pad = max(b - a for a, b in splits)
            ref = upd[members[0]]
            # to each owner o: my padded shard of each matrix o owns
            send = torch.zeros((len(members), pad, cols), dtype=ref.dtype, device=ref.device)
            k = 0
            for o in range(world):
                for j in owned[o]:
                    send[k, : hi - lo] = upd[j]
                    k += 1
            mine = owned[rank]
            recv = torch.empty((world * len(mine), pad, cols), dtype=ref.dtype, device=ref.device)
            dist.all_to_all_single(recv.view(-1, cols), send.view(-1, cols),
                                   output_split_sizes=[len(mine) * pad] * world,
                                   input_split_sizes=[len(owned[o]) * pad for o in range(world)], group=group)
            back = torch.zeros((world * len(mine), pad, cols), dtype=ref.dtype, device=ref.device)
            if mine:
                # from rank q: its rows of each of my matrices, in order
                parts = recv.view(world, len(mine), pad, cols)
                full = torch.cat([parts[q, :, : b - a] for q, (a, b) in enumerate(splits)], dim=1).contiguous()
                ops.ns(full)
                bv = back.view(world, len(mine), pad, cols)
                for q, (a, b) in enumerate(splits):
                    bv[q, :, : b - a] = full[:, a:b]
            ret = torch.empty((len(members), pad, cols), dtype=ref.dtype, device=ref.device)
            dist.all_to_all_single(ret.view(-1, cols), back.view(-1, cols),
                                   output_split_sizes=[len(owned[o]) * pad for o in range(world)],
                                   input_split_sizes=[len(mine) * pad] * world, group=group)
            k = 0
            for o in range(world):
                for j in owned[o]:
                    outs[j] = ret[k, : hi - lo]
                    k += 1
        for (rows, cols), p, o in zip(shapes, params, outs):
            ops.apply(p, o.contiguous(), scale if scale > 0 else ops.scale(rows, cols))
