"""The largest calls: every expert matrix of the 384-expert model on one GPU.

A rank that owned all 384 experts would hold 768 matrices of 6144 x 1792
(w1, w3) and 384 of 1792 x 6144 (w2).  One batched Newton-Schulz call over the
768, and one fused step over the 384, cross every 32-bit boundary of the
element offsets (8.5e9 elements in one buffer) and run the largest tile
counts.  Each matrix is processed independently of its neighbours in the
batch, so the big call must equal, bit for bit, the same matrices in chunks
of 96 (the bench's per-rank batch); the first, a middle and the last matrix
are also compared with the fp64 oracle.  The test skips when the device has
not the memory to spare (it needs about 105 GB at its peak).
"""

import pytest
import torch

import workloads
from tests._oracle_pool import oracle_errors
from tests._util import np32, require_gpu

pytestmark = pytest.mark.gpu

BF16_TOL = 2e-2
CHUNK = 96


@pytest.fixture(scope="module")
def mk():
    return require_gpu()


def _need(bytes_):
    torch.cuda.empty_cache()
    free, _ = torch.cuda.mem_get_info()
    if free < 1.2 * bytes_:
        pytest.skip(f"needs {bytes_ / 1e9:.0f} GB of free device memory, {free / 1e9:.0f} GB free")


def test_newton_schulz_over_all_768_w1_w3_matrices(mk):
    b, r, c = 768, workloads.HIDDEN, workloads.EXPERT_HIDDEN
    _need(3 * b * r * c * 2 + mk.muon_ns_workspace_bytes(b, r, c))
    X0 = workloads.gradients(b, r, c, 9100, device="cuda")
    X = X0.clone()
    mk.muon_ns_batched(X)
    torch.cuda.synchronize()
    assert mk.muon_get_device_status() == 0
    assert X.numel() > 2 ** 32
    ref = X0.clone()
    for k in range(0, b, CHUNK):
        mk.muon_ns_batched(ref[k:k + CHUNK])
    torch.cuda.synchronize()
    assert torch.equal(X.view(torch.int16), ref.view(torch.int16))
    del ref
    picks = [0, b // 2 + 7, b - 1]
    res = oracle_errors(((np32(X0[i]), np32(X[i])) for i in picks), len(picks))
    errs = [e for e, _ in res]
    print("768 x 6144x1792: rel errors of matrices", picks, ["%.3e" % e for e in errs])
    assert max(errs) < BF16_TOL
    del X, X0
    torch.cuda.empty_cache()


def test_fused_step_over_all_384_w2_matrices(mk):
    b, r, c = 384, workloads.EXPERT_HIDDEN, workloads.HIDDEN
    elems = b * r * c
    _need(elems * 14 + mk.muon_step_workspace_bytes(b, r, c))   # g, W, M and their copies
    g = workloads.gradients(b, r, c, 9200, device="cuda")
    W0 = workloads.parameters(b, r, c, 9201, device="cuda")
    M0 = torch.zeros(b, r, c, device="cuda")
    W, M = W0.clone(), M0.clone()
    mk.muon_step_batched(W, g, M)
    torch.cuda.synchronize()
    assert mk.muon_get_device_status() == 0
    for k in range(0, b, CHUNK):
        mk.muon_step_batched(W0[k:k + CHUNK], g[k:k + CHUNK], M0[k:k + CHUNK])
    torch.cuda.synchronize()
    assert torch.equal(W.view(torch.int16), W0.view(torch.int16))
    assert torch.equal(M, M0)
    assert bool(torch.isfinite(W.float()).all())
    del g, W0, M0, W, M
    torch.cuda.empty_cache()
