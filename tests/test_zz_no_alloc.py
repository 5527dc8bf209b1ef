"""The entry point that allocates nothing, against the allocating one.

muon_ns_batched_static serves callers that cannot allocate device memory (a
host that owns all device memory through its own arena, a runtime with a
fixed budget after start-up, a C caller without an allocator): it runs the
same Newton-Schulz on a scratch array the library reserves statically on the
device.  Two calls in a row, each checked against muon_ns_batched on the same
input, show that the shared scratch left over from one call does not leak
into the next.  This file is collected last so that a failure here comes
after every other test has run.
"""

import ctypes

import pytest
import torch

import workloads
from tests._util import np32, rel_fro, require_gpu

pytestmark = pytest.mark.gpu

BF16_TOL = 2e-2
QUINTIC = (ctypes.c_float * 3)(3.4445, -4.7750, 2.0315)


@pytest.fixture(scope="module")
def mk():
    return require_gpu()


def call_static(mk, X, steps=5):
    b, m, n = X.shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return mk.lib().muon_ns_batched_static(ctypes.c_void_p(X.data_ptr()), b, m, n, steps, QUINTIC, 1e-7, stream)


def test_static_scratch_matches_allocating_entry_point_twice(mk):
    # one w2-shaped and one w1-shaped expert matrix: each needs about 79 MB of
    # workspace, within the 96 MiB scratch; the second call follows the first
    shapes = [(1, workloads.EXPERT_HIDDEN, workloads.HIDDEN), (1, workloads.HIDDEN, workloads.EXPERT_HIDDEN)]
    assert all(mk.muon_ns_workspace_bytes(*s) <= mk.NS_STATIC_SCRATCH_BYTES for s in shapes)
    for k, (b, m, n) in enumerate(shapes):
        X = workloads.gradients(b, m, n, 4242 + k, device="cuda")
        ref = X.clone()
        mk.muon_ns_batched(ref)
        assert call_static(mk, X) == 0
        assert mk.muon_get_device_status() == 0
        assert rel_fro(np32(X), np32(ref)) < BF16_TOL
        assert torch.equal(X, ref)   # same kernels, same order: identical bits


def test_static_scratch_after_a_large_call_on_ragged_and_near_limit_shapes(mk):
    # After a call that fills most of the scratch, calls whose tiles do not
    # divide their shapes (TMA-clipped loads and stores near the end of the
    # regions they use) and a call whose workspace sits just under the limit
    # must still match the allocating entry point bit for bit: nothing a call
    # reads is left over from an earlier one.
    big = (1, workloads.EXPERT_HIDDEN, workloads.HIDDEN)
    ragged = [(2, 520, 776), (3, 776, 264), (2, 8, 8)]
    # the largest batch of 1024 x 3072 matrices whose workspace fits
    near = max(((b, 1024, 3072) for b in range(1, 16)
                if mk.muon_ns_workspace_bytes(b, 1024, 3072) <= mk.NS_STATIC_SCRATCH_BYTES),
               key=lambda s: s[0])
    assert mk.muon_ns_workspace_bytes(*near) > 0.7 * mk.NS_STATIC_SCRATCH_BYTES
    for k, (b, m, n) in enumerate([big] + ragged + [near] + ragged[:1]):
        X = workloads.gradients(b, m, n, 4400 + k, device="cuda")
        ref = X.clone()
        mk.muon_ns_batched(ref)
        assert call_static(mk, X) == 0
        assert mk.muon_get_device_status() == 0
        assert torch.equal(X, ref), (b, m, n)


def test_static_scratch_rejects_sizes_beyond_its_maximum(mk):
    X = workloads.gradients(2, workloads.EXPERT_HIDDEN, workloads.HIDDEN, 4343, device="cuda")
    before = X.clone()
    assert mk.muon_ns_workspace_bytes(2, workloads.EXPERT_HIDDEN, workloads.HIDDEN) > mk.NS_STATIC_SCRATCH_BYTES
    assert call_static(mk, X) == -4          # MUON_ERR_NO_MEMORY, nothing launched
    torch.cuda.synchronize()
    assert torch.equal(X, before)
