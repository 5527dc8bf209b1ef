"""The checked build of the library on the GPU.

libmuon_checked.so is the same source compiled with -DMUON_DEVICE_CHECKS: the
tensor-core kernels test, before every TMA load and store, that the
coordinate's x sits on a 16-element boundary and that no store starts at a
negative coordinate (a broken one would fault the GPU), and report a broken
one as MUON_ERR_DEVICE instead of making the access.  On ragged shapes in
both orientations, both 16-bit storage formats, one to five iterations and
the fused step, the checked build must report nothing and give the normal
build's bits.  Both libraries run in this process on the same device, each
with its own error word.
"""

import ctypes

import pytest
import torch

import workloads
from tests._util import require_gpu

pytestmark = pytest.mark.gpu

SHAPES = [(2, 264, 776), (3, 776, 264), (1, 8, 8), (2, 136, 1032), (1, 1792, 640), (2, 640, 1792), (1, 520, 200)]


@pytest.fixture(scope="module")
def libs():
    mk = require_gpu()
    from muon_newton_schulz_expert_gb300 import build as b
    lib = ctypes.CDLL(b.build(checked=True))
    for name, (res, args) in mk.SIGNATURES.items():
        f = getattr(lib, name)
        f.restype, f.argtypes = res, args
    return mk, lib


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("steps", [5, 1])
@pytest.mark.parametrize("batch,m,n", SHAPES)
def test_checked_newton_schulz_reports_nothing_and_matches(libs, batch, m, n, steps):
    mk, lib = libs
    X0 = workloads.gradients(batch, m, n, 9300 + m + n, device="cuda")
    X = X0.clone()
    co = (ctypes.c_float * 3)(*mk.QUINTIC)
    assert lib.muon_ns_batched(ctypes.c_void_p(X.data_ptr()), batch, m, n, steps, co, 1e-7, _stream()) == 0
    assert lib.muon_get_device_status(_stream()) == 0
    ref = X0.clone()
    mk.muon_ns_batched(ref, steps=steps)
    torch.cuda.synchronize()
    assert torch.equal(X.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("batch,m,n", SHAPES[:4])
def test_checked_fused_step_reports_nothing_and_matches(libs, batch, m, n):
    mk, lib = libs
    g = workloads.gradients(batch, m, n, 9400 + m, device="cuda")
    W0 = workloads.parameters(batch, m, n, 9401 + m, device="cuda")
    M0 = torch.randn(batch, m, n, generator=torch.Generator("cuda").manual_seed(9402 + m), device="cuda") * 0.1
    W, M = W0.clone(), M0.clone()
    co = (ctypes.c_float * 3)(*mk.QUINTIC)
    st = lib.muon_step_batched(ctypes.c_void_p(W.data_ptr()), ctypes.c_void_p(g.data_ptr()),
                               ctypes.c_void_p(M.data_ptr()), batch, m, n, 0.95, 1, 5, co, 1e-7, 0.02, 0.1, 0.0,
                               None, 0, _stream())
    assert st == 0
    assert lib.muon_get_device_status(_stream()) == 0
    W1, M1 = W0.clone(), M0.clone()
    mk.muon_step_batched(W1, g, M1)
    torch.cuda.synchronize()
    assert torch.equal(W.view(torch.int16), W1.view(torch.int16))
    assert torch.equal(M, M1)
