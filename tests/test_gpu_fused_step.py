"""The fused device step against the three separate calls and the oracle.

muon_step_batched fuses the norm's sum of squares into the momentum kernel and
the parameter update into the last Newton-Schulz epilogue.  Its parameters and
momentum must equal, bit for bit, those of muon_momentum_update ->
muon_ns_batched -> muon_apply_update (each of which the parity tests pin to
the oracle), and with W = 0, lr = 1, wd = 0, scale = 1 the new parameters are
exactly -O, which is checked against the oracle's Newton-Schulz directly.
"""

import numpy as np
import pytest
import torch

import workloads
from oracle import muon_oracle as O
from tests._util import bits16, bits32, np32, rel_fro, require_gpu

pytestmark = pytest.mark.gpu

BF16_TOL = 2e-2


@pytest.fixture(scope="module")
def mk():
    return require_gpu()


def _inputs(count, rows, cols, seed):
    g = workloads.gradients(count, rows, cols, seed, device="cuda")
    W = workloads.parameters(count, rows, cols, seed + 1, device="cuda")
    buf = torch.randn(count, rows, cols, generator=torch.Generator("cuda").manual_seed(seed + 2), device="cuda") * 0.1
    return g, W, buf


def _separate(mk, W, g, buf, steps, nesterov, scale, coeffs=O.QUINTIC):
    u = torch.empty_like(g)
    mk.muon_momentum_update(g, buf, u, 0.95, nesterov)
    mk.muon_ns_batched(u, steps, coeffs, 1e-7)
    mk.muon_apply_update(W, u, 0.02, 0.1, scale)


CASES = [
    (3, 256, 768, 5, True, 0.0),     # m < n, whole tiles
    (3, 768, 256, 5, True, 0.0),     # stored as the transpose
    (2, 264, 776, 5, True, 0.0),     # partial tiles in both directions
    (2, 776, 264, 3, False, 0.7),    # partial tiles, transposed, plain momentum, explicit scale
    (4, 128, 128, 1, True, 0.0),     # one iteration: the fused epilogue also applies 1/||X||
    (2, 64, 192, 0, True, 0.0),      # normalisation only
    (2, 8, 8, 2, True, 0.0),         # smallest shape
    (1, 1792, 6144, 5, True, 0.0),   # expert w2
    (2, 6144, 1792, 5, True, 0.0),   # expert w1 / w3
]


@pytest.mark.parametrize("count,rows,cols,steps,nesterov,scale", CASES)
def test_fused_step_equals_separate_calls(mk, count, rows, cols, steps, nesterov, scale):
    g, W, buf = _inputs(count, rows, cols, 900 + rows + cols + steps)
    W1, b1 = W.clone(), buf.clone()
    _separate(mk, W1, g, b1, steps, nesterov, scale)
    W2, b2 = W.clone(), buf.clone()
    mk.muon_step_batched(W2, g, b2, mu=0.95, nesterov=nesterov, steps=steps, lr=0.02, weight_decay=0.1,
                         scale=scale)
    torch.cuda.synchronize()
    assert mk.muon_get_device_status() == 0
    assert not torch.equal(W1, W)                       # the step did move the parameters
    assert np.array_equal(bits32(b2), bits32(b1))
    assert np.array_equal(bits16(W2), bits16(W1))


def test_fused_step_caller_workspace_and_momentum_carry(mk):
    count, rows, cols = 3, 512, 1536
    g, W, _ = _inputs(count, rows, cols, 931)
    g2 = workloads.gradients(count, rows, cols, 934, device="cuda")
    buf = torch.zeros(count, rows, cols, device="cuda")
    W1, b1, W2, b2 = W.clone(), buf.clone(), W.clone(), buf.clone()
    ws = torch.empty(mk.muon_step_workspace_bytes(count, rows, cols), dtype=torch.uint8, device="cuda")
    assert ws.numel() == mk.muon_ns_workspace_bytes(count, rows, cols)
    for grad in (g, g2, g):
        _separate(mk, W1, grad, b1, 5, True, 0.0)
        mk.muon_step_batched(W2, grad, b2, workspace=ws)
    torch.cuda.synchronize()
    assert np.array_equal(bits32(b2), bits32(b1))
    assert np.array_equal(bits16(W2), bits16(W1))
    small = ws[:-256]
    with pytest.raises(mk.MuonError) as e:
        mk.muon_step_batched(W2, g, b2, workspace=small)
    assert e.value.status == -4


@pytest.mark.parametrize("count,rows,cols", [(4, 256, 512), (3, 640, 192), (2, 1792, 6144)])
def test_fused_step_update_against_oracle(mk, count, rows, cols):
    # W = 0, lr = 1, wd = 0, scale = 1: kw = 1, ko = -1, so W' = bf16(0 + (-1) O) = -O exactly
    g, _, buf = _inputs(count, rows, cols, 950 + rows)
    b0 = np32(buf)
    W = torch.zeros(count, rows, cols, dtype=torch.bfloat16, device="cuda")
    mk.muon_step_batched(W, g, buf, mu=0.95, nesterov=True, steps=5, lr=1.0, weight_decay=0.0, scale=1.0)
    torch.cuda.synchronize()
    assert mk.muon_get_device_status() == 0
    nb, u = O.momentum_update(np32(g), b0, float(np.float32(0.95)), True)
    assert np.array_equal(bits32(buf), nb.view(np.uint32))
    want = O.newton_schulz_batched(O.bf16_round(u))
    assert rel_fro(-np32(W), want) < BF16_TOL


def test_fused_step_at_bench_size_equals_separate_calls(mk):
    # the 96-matrix workload the benchmark times, in its launch configuration
    # (one call per shape group), compared on the device element by element
    groups = [(64, workloads.HIDDEN, workloads.EXPERT_HIDDEN), (32, workloads.EXPERT_HIDDEN, workloads.HIDDEN)]
    for i, (count, rows, cols) in enumerate(groups):
        g, W, buf = _inputs(count, rows, cols, 970 + i)
        W1, b1 = W.clone(), buf.clone()
        _separate(mk, W1, g, b1, 5, True, 0.0)
        W2, b2 = W, buf
        mk.muon_step_batched(W2, g, b2)
        torch.cuda.synchronize()
        assert mk.muon_get_device_status() == 0
        assert torch.equal(b2, b1)
        assert torch.equal(W2.view(torch.int16), W1.view(torch.int16))
        del g, W, buf, W1, b1, W2, b2
        torch.cuda.empty_cache()


@pytest.mark.parametrize("count,rows,cols", [(3, 256, 768), (2, 776, 264)])
def test_fused_schedule_equals_separate_calls(mk, count, rows, cols):
    rows_ = [O.QUINTIC, (3.0, -3.2, 1.2), O.QUINTIC, (2.0, -1.5, 0.5)]
    g, W, buf = _inputs(count, rows, cols, 960 + rows)
    W1, b1, u = W.clone(), buf.clone(), torch.empty_like(g)
    mk.muon_momentum_update(g, b1, u, 0.95, True)
    mk.muon_ns_batched_schedule(u, rows_, 1e-7)
    mk.muon_apply_update(W1, u, 0.02, 0.1, 0.0)
    W2, b2 = W.clone(), buf.clone()
    mk.muon_step_batched_schedule(W2, g, b2, rows_)
    torch.cuda.synchronize()
    assert mk.muon_get_device_status() == 0
    assert not torch.equal(W1, W)
    assert np.array_equal(bits32(b2), bits32(b1))
    assert np.array_equal(bits16(W2), bits16(W1))
    # a schedule of equal rows is the constant-coefficient step
    W3, b3, W4, b4 = W.clone(), buf.clone(), W.clone(), buf.clone()
    mk.muon_step_batched_schedule(W3, g, b3, [O.QUINTIC] * 5)
    mk.muon_step_batched(W4, g, b4)
    torch.cuda.synchronize()
    assert np.array_equal(bits16(W3), bits16(W4))


def test_fused_step_launches_its_own_kernels(mk):
    g, W, buf = _inputs(2, 256, 512, 990)
    mk.muon_trace_begin()
    mk.muon_step_batched(W, g, buf, steps=3)
    trace = mk.muon_trace_end()
    assert trace["momentum_norm_bf16"][0] == 1
    assert trace["ns_axpy_tc"][0] == 2 and trace["ns_axpy_apply_tc"][0] == 1
    assert "norm_partial" not in trace and "apply_bf16" not in trace and "momentum_bf16" not in trace


def test_param_free_event_orders_only_the_update(mk):
    # a side stream sleeps, then copies the parameters and records param_free;
    # the step's parameter-writing launch must come after that copy (which
    # therefore sees the old parameters), and the result is unchanged
    g, W, buf = _inputs(3, 512, 1536, 995)
    W0 = W.clone()
    W1, b1 = W.clone(), buf.clone()
    mk.muon_step_batched(W1, g, b1)
    side, snap = torch.cuda.Stream(), torch.empty_like(W)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        torch.cuda._sleep(20_000_000)   # ~10 ms, bounded
        snap.copy_(W)
        ev = side.record_event()
    mk.muon_step_batched(W, g, buf, param_free=ev)
    torch.cuda.synchronize()
    assert mk.muon_get_device_status() == 0
    assert torch.equal(snap.view(torch.int16), W0.view(torch.int16))
    assert np.array_equal(bits16(W), bits16(W1))
    assert np.array_equal(bits32(buf), bits32(b1))
    with pytest.raises(ValueError):
        mk.muon_step_batched(W, g, buf, param_free=torch.cuda.Event())   # never recorded
