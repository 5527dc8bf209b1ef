"""dense_step on one GPU with the library's kernels.

With one rank, dense_step stacks the matrices of each shape and runs one
batched Newton-Schulz call per shape between the momentum and update calls.
Its result must match the fp64 oracle (momentum bit for bit, the
orthogonalised update within 2e-2), and equal, bit for bit, the fused step on
the same matrices given the same fp32 shape scale (the dense path hands the
full matrix's scale to the update as an fp32 argument).  With an initialised
one-rank NCCL group the same step runs through the exchange (both
all_to_all_single calls on CUDA tensors) and must give the same bits.  The
all-to-all of more ranks is covered on CPU by tests/test_dense_multirank.py.
"""

import numpy as np
import pytest
import torch

import workloads
from muon_newton_schulz_expert_gb300 import dense
from oracle import muon_oracle as O
from tests._util import bits16, bits32, np32, rel_fro, require_gpu

pytestmark = pytest.mark.gpu

# two matrices of the attention-like square shape, so that one call batches them
SHAPES = [(workloads.HIDDEN, workloads.HIDDEN), (workloads.HIDDEN, 1024), (264, 776), (776, 264),
          (workloads.HIDDEN, workloads.HIDDEN)]


@pytest.fixture(scope="module")
def mk():
    return require_gpu()


def _inputs(seed):
    out = []
    for i, (r, c) in enumerate(SHAPES):
        g = workloads.gradients(1, r, c, seed + 3 * i, device="cuda", kind="normal")[0]
        W = workloads.parameters(1, r, c, seed + 3 * i + 1, device="cuda")[0]
        m = torch.randn(r, c, generator=torch.Generator("cuda").manual_seed(seed + 3 * i + 2), device="cuda") * 0.1
        out.append((W, g, m))
    return out


@pytest.mark.parametrize("scale", [0.0, 0.5])
def test_single_rank_dense_step_equals_fused_step(mk, scale):
    mats = _inputs(4100)
    params = [W.clone() for W, _, _ in mats]
    moms = [m.clone() for _, _, m in mats]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    dense.dense_step(params, [g for _, g, _ in mats], moms, SHAPES, scale=scale, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    assert mk.muon_get_device_status() == 0
    for (r, c), (W, g, m), p2, m2 in zip(SHAPES, mats, params, moms):
        W1, m1 = W.clone().unsqueeze(0), m.clone().unsqueeze(0)
        sc = scale if scale > 0 else mk.muon_default_scale(r, c)
        mk.muon_step_batched(W1, g.unsqueeze(0), m1, scale=sc)
        torch.cuda.synchronize()
        assert not torch.equal(p2, W)
        assert np.array_equal(bits32(m2), bits32(m1[0]))
        assert np.array_equal(bits16(p2), bits16(W1[0]))


def test_single_rank_dense_step_matches_oracle(mk):
    # W = 0, lr = 1, wd = 0, scale = 1: the new parameter is -bf16(O)
    mats = _inputs(4200)
    params = [torch.zeros_like(W) for W, _, _ in mats]
    moms = [m.clone() for _, _, m in mats]
    dense.dense_step(params, [g for _, g, _ in mats], moms, SHAPES, lr=1.0, weight_decay=0.0, scale=1.0)
    torch.cuda.synchronize()
    assert mk.muon_get_device_status() == 0
    for j, ((r, c), (W, g, m), p2, m2) in enumerate(zip(SHAPES, mats, params, moms)):
        ref = O.muon_step(np.zeros((1, r, c)), np32(g)[None], np32(m)[None], mu=float(np.float32(0.95)), lr=1.0,
                          weight_decay=0.0, scale=1.0)
        assert np.array_equal(bits32(m2), ref["buf"][0].view(np.uint32)), j
        err = rel_fro(-np32(p2), ref["O"][0])
        print(f"dense matrix {j} {r}x{c}: rel {err:.3e}")
        assert err < 2e-2, (j, err)


def test_exchange_over_a_one_rank_nccl_group_equals_the_local_path(mk):
    # An initialised process group, even of one rank, sends the update through
    # the exchange: both all_to_all_single calls run on NCCL with CUDA tensors
    # and the library's kernels on the owner, on a side stream.  One rank owns
    # everything, so the result must equal the path without a group bit for bit.
    import socket

    import torch.distributed as dist
    if not dist.is_nccl_available():
        pytest.skip("NCCL backend not available")
    mats = _inputs(4300)
    p_ref = [W.clone() for W, _, _ in mats]
    m_ref = [m.clone() for _, _, m in mats]
    dense.dense_step(p_ref, [g for _, g, _ in mats], m_ref, SHAPES)
    with socket.socket() as s_:
        s_.bind(("127.0.0.1", 0))
        port = s_.getsockname()[1]
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    try:
        params = [W.clone() for W, _, _ in mats]
        moms = [m.clone() for _, _, m in mats]
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        dense.dense_step(params, [g for _, g, _ in mats], moms, SHAPES, stream=side)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
    finally:
        dist.destroy_process_group()
    assert mk.muon_get_device_status() == 0
    for j in range(len(SHAPES)):
        assert np.array_equal(bits16(params[j]), bits16(p_ref[j])), j
        assert np.array_equal(bits32(moms[j]), bits32(m_ref[j])), j
