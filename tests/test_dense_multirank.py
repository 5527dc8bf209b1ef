"""Row-sharded dense matrices over two and three gloo ranks (CPU).

The data movement of dense_step (the all-to-all to the owners, the batched
orthogonalisation there, the all-to-all back) is checked with stand-in
operations on fp32 CPU tensors: a momentum, an orthogonalisation stand-in that
mixes every row of each full matrix of a batch and depends on the matrix's
position in the batch only through its own rows (so a row landing on the wrong
rank, in the wrong order or in the wrong matrix changes the result) and an
update.  Each rank's shards must equal the rows of the same operations applied
to the full matrices in one process.  The library's own kernels run in
tests/test_gpu_dense.py.
"""

import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

from muon_newton_schulz_expert_gb300 import dense

# uneven splits; fewer rows than ranks (empty shards); repeated shapes, so that
# owners batch several matrices and some owners hold none of a shape
SHAPES = [(10, 6), (7, 9), (16, 4), (3, 5), (1, 4), (10, 6), (7, 9), (10, 6), (10, 6)]
MU, LR = 0.9, 0.05


def _ops():
    def momentum(g, m, u):
        m.mul_(MU).add_(g)
        u.copy_(g + MU * m)

    def ns(x):   # on each matrix of a (batch, rows, cols) stack: a function of the whole matrix, row order included
        assert x.dim() == 3
        w = torch.arange(1, x.shape[1] + 1, dtype=x.dtype).view(1, -1, 1)
        x.copy_(torch.flip(x, [1]) * 0.5 + (x * w).sum(1, keepdim=True) / x.shape[1])

    def apply(p, o, sc):
        p.mul_(0.99).add_(o, alpha=-LR * sc)

    def scale(r, c):
        return 1.0 + r / (r + c)

    return dense.Ops(momentum, ns, apply, scale)


def _full_inputs(seed=7):
    g = torch.Generator().manual_seed(seed)
    params = [torch.randn(r, c, generator=g) for r, c in SHAPES]
    grads = [torch.randn(r, c, generator=g) for r, c in SHAPES]
    moms = [torch.randn(r, c, generator=g) for r, c in SHAPES]
    return params, grads, moms


def _reference():
    params, grads, moms = _full_inputs()
    ops = _ops()
    for (r, c), p, g, m in zip(SHAPES, params, grads, moms):
        u = torch.empty_like(g)
        ops.momentum(g, m, u)
        ops.ns(u.unsqueeze(0))
        ops.apply(p, u, ops.scale(r, c))
    return params, moms


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "MASTER_ADDR": "127.0.0.1",
                       "MASTER_PORT": str(port)})
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    params, grads, moms = _full_inputs()
    sl = [dense.row_splits(r, world)[rank] for r, _ in SHAPES]
    p_sh = [p[a:b].clone() for p, (a, b) in zip(params, sl)]
    g_sh = [g[a:b].clone() for g, (a, b) in zip(grads, sl)]
    m_sh = [m[a:b].clone() for m, (a, b) in zip(moms, sl)]
    dense.dense_step(p_sh, g_sh, m_sh, SHAPES, ops=_ops())
    out[rank] = ([t.clone() for t in p_sh], [t.clone() for t in m_sh])
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [1, 2, 3, 4])
def test_dense_step_matches_the_full_matrices(world):
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn")
        res = dict(out)
    ref_p, ref_m = _reference()
    for j, (rows, _) in enumerate(SHAPES):
        got_p = torch.cat([res[r][0][j] for r in range(world)])
        got_m = torch.cat([res[r][1][j] for r in range(world)])
        assert torch.equal(got_p, ref_p[j]), j
        assert torch.equal(got_m, ref_m[j]), j


def test_row_splits_and_owners():
    assert dense.row_splits(10, 3) == [(0, 4), (4, 7), (7, 10)]
    assert dense.row_splits(3, 4) == [(0, 1), (1, 2), (2, 3), (3, 3)]
    assert dense.row_splits(6144, 8)[-1] == (5376, 6144)
    for rows in (0, 1, 5, 10, 1792):
        for world in (1, 2, 3, 4, 7):
            got = [b - a for a, b in dense.row_splits(rows, world)]
            assert got == [t.shape[0] for t in torch.tensor_split(torch.empty(rows), world)], (rows, world)
    for rows in (1, 7, 10, 6144):
        for world in (1, 2, 3, 8):
            s = dense.row_splits(rows, world)
            assert s[0][0] == 0 and s[-1][1] == rows
            assert all(a == b for (_, a), (b, _) in zip(s, s[1:]))
            assert max(b - a for a, b in s) - min(b - a for a, b in s) <= 1
    assert [dense.owner_of(j, 3) for j in range(5)] == [0, 1, 2, 0, 1]
    assert dense.shape_groups(SHAPES) == [((10, 6), [0, 5, 7, 8]), ((7, 9), [1, 6]), ((16, 4), [2]), ((3, 5), [3]),
                                          ((1, 4), [4])]


def test_single_rank_runs_without_a_process_group():
    params, grads, moms = _full_inputs()
    dense.dense_step(params, grads, moms, SHAPES, ops=_ops())
    ref_p, ref_m = _reference()
    for j in range(len(SHAPES)):
        assert torch.equal(params[j], ref_p[j]) and torch.equal(moms[j], ref_m[j])


def test_shard_shapes_are_checked():
    params, grads, moms = _full_inputs()
    with pytest.raises(ValueError):
        dense.dense_step(params[:1], grads[:1], moms[:1], [(11, 6)], ops=_ops())
