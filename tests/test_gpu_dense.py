"""dense_step on one GPU with the library's kernels.

With one rank, dense_step runs the momentum, Newton-Schulz and update calls on
each full matrix; its result must equal, bit for bit, the fused step on the
same matrices given the same fp32 shape scale (the dense path hands the full
matrix's scale to the update as an fp32 argument).  The gather/scatter of more
ranks is covered on CPU by tests/test_dense_multirank.py.
"""

import numpy as np
import pytest
import torch

import workloads
from muon_newton_schulz_expert_gb300 import dense
from tests._util import bits16, bits32, require_gpu

pytestmark = pytest.mark.gpu

SHAPES = [(workloads.HIDDEN, workloads.HIDDEN), (workloads.HIDDEN, 1024), (264, 776), (776, 264)]


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
    dense.dense_step(params, [g for _, g, _ in mats], moms, SHAPES, scale=scale)
    torch.cuda.synchronize()
    assert mk.muon_get_device_status() == 0
    for (r, c), (W, g, m), p2, m2 in zip(SHAPES, mats, params, moms):
        W1, m1 = W.clone().unsqueeze(0), m.clone().unsqueeze(0)
        sc = scale if scale > 0 else float(np.float32(dense.default_scale(r, c)))
        mk.muon_step_batched(W1, g.unsqueeze(0), m1, scale=sc)
        torch.cuda.synchronize()
        assert not torch.equal(p2, W)
        assert np.array_equal(bits32(m2), bits32(m1[0]))
        assert np.array_equal(bits16(p2), bits16(W1[0]))
