"""Host-injected allocation failures, and checkpoint/resume of the step (GPU).

Allocation failure: muon_inject_alloc_failures makes the library's next
device allocation fail on the host, as an exhausted memory pool would.  Every
allocating entry point must then return MUON_ERR_NO_MEMORY having launched
nothing and changed none of its buffers, and the next call must run normally
and give the bits an undisturbed call gives.  No GPU fault is involved.

Checkpoint/resume: the library keeps no state between calls (the caller owns
the fp32 momentum), so three steps in a row must equal two steps, a round
trip of parameters and momentum through host memory (a checkpoint written and
read back), and a third step on fresh device buffers: bit for bit.
"""

import pytest
import torch

import workloads
from tests._util import require_gpu

pytestmark = pytest.mark.gpu

NO_MEMORY = -4


@pytest.fixture(scope="module")
def mk():
    m = require_gpu()
    yield m
    m.muon_inject_alloc_failures(0)


def expect_no_memory(mk, fn):
    launches = mk.muon_launch_count()
    assert mk.muon_inject_alloc_failures(1) == 0
    with pytest.raises(mk.MuonError) as e:
        fn()
    assert e.value.status == NO_MEMORY
    assert mk.muon_inject_alloc_failures(0) == 0       # the injected failure was consumed
    torch.cuda.synchronize()
    assert mk.muon_launch_count() == launches           # nothing launched
    assert mk.muon_get_device_status() == 0


@pytest.mark.parametrize("batch,m,n", [(3, 264, 776), (2, 1792, 640), (4, 64, 256)])
def test_injected_allocation_failure_in_newton_schulz(mk, batch, m, n):
    X0 = workloads.gradients(batch, m, n, 8100 + m, device="cuda")
    X = X0.clone()
    expect_no_memory(mk, lambda: mk.muon_ns_batched(X))
    assert torch.equal(X.view(torch.int16), X0.view(torch.int16))
    mk.muon_ns_batched(X)                               # the next call runs
    ref = X0.clone()
    mk.muon_ns_batched(ref)
    assert torch.equal(X.view(torch.int16), ref.view(torch.int16))
    Xf0 = X0.float()
    Xf = Xf0.clone()
    expect_no_memory(mk, lambda: mk.muon_ns_batched_f32(Xf))
    assert torch.equal(Xf, Xf0)
    expect_no_memory(mk, lambda: mk.muon_ns_batched_schedule(X, [mk.QUINTIC] * 3))
    assert torch.equal(X.view(torch.int16), ref.view(torch.int16))


def test_injected_allocation_failure_in_the_fused_step(mk):
    b, r, c = 3, 768, 256
    g = workloads.gradients(b, r, c, 8200, device="cuda")
    W0 = workloads.parameters(b, r, c, 8201, device="cuda")
    M0 = torch.randn(b, r, c, generator=torch.Generator("cuda").manual_seed(8202), device="cuda") * 0.1
    W, M = W0.clone(), M0.clone()
    expect_no_memory(mk, lambda: mk.muon_step_batched(W, g, M))
    assert torch.equal(W.view(torch.int16), W0.view(torch.int16)) and torch.equal(M, M0)
    mk.muon_step_batched(W, g, M)
    W1, M1 = W0.clone(), M0.clone()
    mk.muon_step_batched(W1, g, M1)
    assert torch.equal(W.view(torch.int16), W1.view(torch.int16)) and torch.equal(M, M1)


def test_injected_allocation_failure_in_the_host_resident_step(mk):
    b, r, c = 5, 256, 384
    g = workloads.gradients(b, r, c, 8300, device="cpu").pin_memory()
    W = workloads.parameters(b, r, c, 8301, device="cpu").pin_memory()
    M = (torch.randn(b, r, c, generator=torch.Generator().manual_seed(8302)) * 0.1).pin_memory()
    W0, M0 = W.clone(), M.clone()
    expect_no_memory(mk, lambda: mk.muon_step_host(W, g, M, chunk=2))
    assert torch.equal(W.view(torch.int16), W0.view(torch.int16)) and torch.equal(M, M0)
    mk.muon_step_host(W, g, M, chunk=2)
    torch.cuda.synchronize()
    Wd, Md = W0.cuda(), M0.cuda()
    mk.muon_step_batched(Wd, g.cuda(), Md)
    assert torch.equal(W.view(torch.int16), Wd.cpu().view(torch.int16)) and torch.equal(M, Md.cpu())


@pytest.mark.parametrize("b,r,c", [(4, 6144, 1792), (6, 264, 776)])
def test_three_steps_equal_two_steps_a_checkpoint_and_one_step(mk, b, r, c):
    grads = [workloads.gradients(b, r, c, 8400 + 10 * k + r, device="cuda") for k in range(3)]
    W0 = workloads.parameters(b, r, c, 8450 + r, device="cuda")
    # straight through
    W, M = W0.clone(), torch.zeros(b, r, c, device="cuda")
    for g in grads:
        mk.muon_step_batched(W, g, M)
    # two steps, checkpoint to host, fresh device buffers, third step
    W2, M2 = W0.clone(), torch.zeros(b, r, c, device="cuda")
    for g in grads[:2]:
        mk.muon_step_batched(W2, g, M2)
    ckpt = {"param": W2.cpu().clone(), "momentum": M2.cpu().clone()}
    del W2, M2
    torch.cuda.empty_cache()
    W3, M3 = ckpt["param"].cuda(), ckpt["momentum"].cuda()
    mk.muon_step_batched(W3, grads[2], M3)
    torch.cuda.synchronize()
    assert mk.muon_get_device_status() == 0
    assert torch.equal(M3, M)
    assert torch.equal(W3.view(torch.int16), W.view(torch.int16))
