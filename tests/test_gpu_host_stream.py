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
