"""Guard bands around every buffer the tensor-core path writes (GPU).

Each caller buffer (X, or the fused step's parameters, gradients and
momentum) and the workspace sit inside a larger allocation whose surrounding
bytes hold a sentinel; inside the workspace, the library leaves an unwritten
gap after every region (the workspace layout: two X buffers, X's low half
(one byte per element, rows padded to 16 bytes), A, B, the norm partials and
two per-matrix factors, each on a 256-byte boundary and followed by 256
bytes).  After each call every byte
outside what the call may write must still hold the sentinel.  The shapes
have ragged tiles in both orientations (TMA-clipped stores, the mirrored
transpose stores, the diagonal element stores), sizes on both sides of the
fp16/bf16 storage switch at 256 rows, and the single-step and multi-step
paths; every case also checks that the guarded call gives the same bits as
an unguarded one.  All accesses stay inside the allocations: a failure here
is a wrong byte, never a fault.
"""

import pytest
import torch

import workloads
from tests._util import require_gpu

pytestmark = pytest.mark.gpu

SENT = 0xA5
GUARD = 4096                  # bytes before and after each buffer (keeps 256-byte alignment)
GAP = 256                     # the library's gap after each workspace region
SHAPES = [(1, 264, 776), (1, 776, 264), (1, 8, 8), (3, 8, 8), (1, 1792, 640), (2, 136, 1032), (1, 640, 1792)]


@pytest.fixture(scope="module")
def mk():
    return require_gpu()


def a256(x):
    return (x + 255) & ~255


def guarded(nbytes):
    buf = torch.full((GUARD + nbytes + GUARD,), SENT, dtype=torch.uint8, device="cuda")
    return buf, buf[GUARD:GUARD + nbytes]


def untouched(t):
    return bool((t == SENT).all().item())


def ws_regions(batch, m, n):
    """[(offset, bytes a call may write, bytes of the region with its padding and gap)]."""
    mm, nn = min(m, n), max(m, n)
    p16 = lambda c: (c + 15) // 16 * 16     # the low half's rows are padded to 16 bytes
    lo = batch * max(mm * p16(nn), nn * p16(mm))
    sizes = [batch * mm * nn * 2] * 2 + [lo] + [batch * mm * mm * 2] * 2 + [batch * 64 * 4, batch * 4, batch * 4]
    out, off = [], 0
    for sz in sizes:
        out.append((off, sz, a256(sz) + GAP))
        off += a256(sz) + GAP
    return out


def check_workspace(ws_buf, need, batch, m, n):
    assert untouched(ws_buf[:GUARD]) and untouched(ws_buf[GUARD + need:])
    regions = ws_regions(batch, m, n)
    assert regions[-1][0] + regions[-1][2] == need
    for off, used, size in regions:
        assert untouched(ws_buf[GUARD + off + used:GUARD + off + size]), (off, used, size)


@pytest.mark.parametrize("steps", [5, 1])
@pytest.mark.parametrize("batch,m,n", SHAPES)
def test_newton_schulz_writes_nothing_outside_its_buffers(mk, batch, m, n, steps):
    X0 = workloads.gradients(batch, m, n, 7000 + m + n, device="cuda")
    nbytes = X0.numel() * 2
    x_buf, x_mid = guarded(nbytes)
    X = x_mid.view(torch.bfloat16).view(batch, m, n)
    X.copy_(X0)
    need = mk.muon_ns_workspace_bytes(batch, m, n)
    ws_buf, ws = guarded(need)
    mk.muon_ns_batched(X, steps=steps, workspace=ws)
    torch.cuda.synchronize()
    assert mk.muon_get_device_status() == 0
    assert untouched(x_buf[:GUARD]) and untouched(x_buf[GUARD + nbytes:])
    check_workspace(ws_buf, need, batch, m, n)
    ref = X0.clone()
    mk.muon_ns_batched(ref, steps=steps)
    assert torch.equal(X.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("batch,m,n", SHAPES)
def test_fused_step_writes_nothing_outside_its_buffers(mk, batch, m, n):
    g0 = workloads.gradients(batch, m, n, 7100 + m, device="cuda")
    W0 = workloads.parameters(batch, m, n, 7200 + m, device="cuda")
    M0 = torch.randn(batch, m, n, generator=torch.Generator("cuda").manual_seed(7300 + m), device="cuda") * 0.1
    bufs = {}
    for name, t in (("param", W0), ("grad", g0), ("mom", M0)):
        nbytes = t.numel() * t.element_size()
        buf, mid = guarded(nbytes)
        view = mid.view(t.dtype).view(t.shape)
        view.copy_(t)
        bufs[name] = (buf, nbytes, view)
    need = mk.muon_step_workspace_bytes(batch, m, n)
    ws_buf, ws = guarded(need)
    mk.muon_step_batched(bufs["param"][2], bufs["grad"][2], bufs["mom"][2], workspace=ws)
    torch.cuda.synchronize()
    assert mk.muon_get_device_status() == 0
    for name, (buf, nbytes, _) in bufs.items():
        assert untouched(buf[:GUARD]) and untouched(buf[GUARD + nbytes:]), name
    check_workspace(ws_buf, need, batch, m, n)
    W1, M1 = W0.clone(), M0.clone()
    mk.muon_step_batched(W1, g0, M1)
    assert torch.equal(bufs["param"][2].view(torch.int16), W1.view(torch.int16))
    assert torch.equal(bufs["mom"][2], M1)


def test_non_finite_input_norm_is_reported_and_cleared(mk):
    X = workloads.gradients(2, 64, 128, 7400, device="cuda")
    X[1, 3, 5] = float("inf")
    mk.muon_ns_batched(X)
    assert mk.muon_get_device_status() == -6        # MUON_ERR_DEVICE
    assert mk.muon_get_device_status() == 0         # read and cleared
    Y = workloads.gradients(2, 64, 128, 7401, device="cuda")
    mk.muon_ns_batched(Y)
    assert mk.muon_get_device_status() == 0
    assert torch.isfinite(Y.float()).all()
