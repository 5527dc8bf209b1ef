"""The host-resident step equals the device-resident one bit for bit."""

import numpy as np
import pytest
import torch

import workloads
from oracle import muon_oracle as O
from tests._util import np32, rel_fro, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mk():
    return require_gpu()


@pytest.mark.parametrize("count,rows,cols,chunk", [(11, 256, 768, 4), (5, 640, 192, 0), (3, 128, 128, 3)])
def test_host_streamed_step_matches_device_step(mk, count, rows, cols, chunk):
    g = workloads.gradients(count, rows, cols, 700 + rows, device="cuda")
    W = workloads.parameters(count, rows, cols, 701 + rows, device="cuda")
    buf = torch.randn(count, rows, cols, generator=torch.Generator("cuda").manual_seed(702), device="cuda") * 0.1
    # device-resident reference
    Wd, bd, u = W.clone(), buf.clone(), torch.empty_like(g)
    mk.muon_step([Wd], [g], [bd], [u])
    # host-resident
    Wh = W.cpu().pin_memory()
    gh = g.cpu().pin_memory()
    bh = buf.cpu().pin_memory()
    mk.muon_step_host(Wh, gh, bh, chunk=chunk)
    torch.cuda.synchronize()
    assert mk.muon_get_device_status() == 0
    assert torch.equal(Wh, Wd.cpu())
    assert torch.equal(bh, bd.cpu())


def test_host_streamed_step_against_oracle(mk):
    count, rows, cols = 4, 384, 128
    g = workloads.gradients(count, rows, cols, 711, device="cpu").pin_memory()
    W = workloads.parameters(count, rows, cols, 712, device="cpu").pin_memory()
    m = torch.zeros(count, rows, cols).pin_memory()
    W0 = W.float().numpy().copy()
    mk.muon_step_host(W, g, m, chunk=3)
    torch.cuda.synchronize()
    ref = O.muon_step(W0, g.float().numpy(), np.zeros((count, rows, cols), np.float32), mu=float(np.float32(0.95)),
                      lr=float(np.float32(0.02)), weight_decay=float(np.float32(0.1)))
    assert np.array_equal(m.numpy(), ref["buf"])
    assert np.abs(W.float().numpy() - ref["param"]).max() < 1e-3


def test_host_streamed_step_rejects_pageable_memory(mk):
    W = torch.zeros(2, 64, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        mk.muon_step_host(W, W, torch.zeros(2, 64, 64))


def test_grouped_host_step_equals_one_call_per_group(mk):
    # one pipeline over three shapes (and an empty group) gives each group the
    # bits of its own muon_step_host call; chunk 4 makes the slots rotate
    # across group boundaries mid-cycle
    shapes = [(11, 256, 768), (0, 64, 64), (5, 640, 192), (3, 128, 128)]
    groups, singles = [], []
    for i, (b, r, c) in enumerate(shapes):
        g = workloads.gradients(max(b, 1), r, c, 720 + i, device="cpu")[:b].contiguous()
        W = workloads.parameters(max(b, 1), r, c, 730 + i, device="cpu")[:b].contiguous()
        m = (torch.randn(max(b, 1), r, c, generator=torch.Generator().manual_seed(740 + i)) * 0.1)[:b].contiguous()
        scale = 0.5 if i == 2 else 0.0
        groups.append((W.pin_memory(), g.pin_memory(), m.pin_memory(), scale))
        singles.append((W.clone().pin_memory(), g.pin_memory(), m.clone().pin_memory(), scale))
    mk.muon_step_host_grouped(groups, chunk=4)
    for W, g, m, scale in singles:
        if W.shape[0]:
            mk.muon_step_host(W, g, m, chunk=4, scale=scale)
    torch.cuda.synchronize()
    assert mk.muon_get_device_status() == 0
    for (Wg, _, mg, _), (Ws, _, ms, _) in zip(groups, singles):
        assert torch.equal(Wg.view(torch.int16), Ws.view(torch.int16))
        assert torch.equal(mg, ms)
