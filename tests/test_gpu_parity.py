"""GPU path against the fp64 oracle, through the C ABI (via the ctypes binding).

Tolerances: the momentum and the fp32-formula update are bit-exact; the
tensor-core Newton-Schulz output (bf16 in, bf16 out) is within 2e-2 relative
Frobenius error of the fp64 oracle run on the same bf16 input, at every size,
and the fp32 verification mode within 1e-5.  What the 2e-2 covers: the
iteration stores A, B and X's high half in power-of-two-scaled fp16 (unit
roundoff 2^-11; the first iteration's B in bf16, 2^-9), X carries a bf16 low
half, and the output is rounded to bf16 (2^-9); the quintic's relative
sensitivity reaches ~10 near sigma ~ 0.87.  A CPU model of these rounding
points (tests/test_rounding_model.py) puts the error near 2e-3 on large
matrices and at most ~1.5e-2 on 8 x 8 ones.
"""

import numpy as np
import pytest
import torch

import workloads
from oracle import muon_oracle as O
from tests._util import bits16, bits32, np32, rel_fro, require_gpu

pytestmark = pytest.mark.gpu

BF16_TOL = 2e-2
F32_TOL = 1e-5


@pytest.fixture(scope="module")
def mk():
    return require_gpu()


def f32(x):
    return float(np.float32(x))


# ----------------------------------------------------------------------------- momentum
@pytest.mark.parametrize("numel,offset", [(1000003, 0), (4096, 0), (77, 1), (8 * 12345 + 5, 3)])
def test_momentum_bf16_bit_exact(mk, numel, offset):
    dev = "cuda"
    g_all = workloads.gradients(1, 1, numel + offset, 11, device=dev, kind="lognormal_rows")[0, 0]
    b_all = torch.randn(numel + offset, generator=torch.Generator(dev).manual_seed(12), device=dev)
    u_all = torch.empty(numel + offset, dtype=torch.bfloat16, device=dev)
    g, b, u = g_all[offset:], b_all[offset:], u_all[offset:]
    b0 = np32(b)
    mk.muon_momentum_update(g, b, u, mu=0.95, nesterov=True)
    torch.cuda.synchronize()
    nb, uu = O.momentum_update(np32(g), b0, f32(0.95), True)
    assert np.array_equal(bits32(b), nb.view(np.uint32))
    assert np.array_equal(bits16(u), O.bf16_bits(uu))
    # nesterov off: u = buf
    mk.muon_momentum_update(g, b, u, mu=0.9, nesterov=False)
    nb2, uu2 = O.momentum_update(np32(g), nb, f32(0.9), False)
    assert np.array_equal(bits32(b), nb2.view(np.uint32))
    assert np.array_equal(bits16(u), O.bf16_bits(uu2))


def test_momentum_f32_bit_exact(mk):
    gen = torch.Generator("cuda").manual_seed(13)
    g = torch.randn(100003, generator=gen, device="cuda")
    b = torch.randn(100003, generator=gen, device="cuda")
    u = torch.empty_like(g)
    b0 = np32(b)
    mk.muon_momentum_update_f32(g, b, u, mu=0.95)
    nb, uu = O.momentum_update(np32(g), b0, f32(0.95), True)
    assert np.array_equal(bits32(b), nb.view(np.uint32))
    assert np.array_equal(bits32(u), uu.view(np.uint32))


# ----------------------------------------------------------------------------- update
@pytest.mark.parametrize("shape", [(3, 640, 192), (2, 192, 640), (1, 37, 41)])
def test_apply_update_bf16_bit_exact(mk, shape):
    gen = torch.Generator("cuda").manual_seed(14)
    W = (torch.randn(shape, generator=gen, device="cuda") * 0.02).to(torch.bfloat16)
    Ob = (torch.randn(shape, generator=gen, device="cuda") * 0.03).to(torch.bfloat16)
    W0 = np32(W)
    lr, wd = f32(0.02), f32(0.1)
    mk.muon_apply_update(W, Ob, lr=lr, weight_decay=wd, scale=0.0)
    sc = O.default_scale(shape[1], shape[2])
    want = O.apply_update_fp32(W0, np32(Ob), lr, wd, sc)
    assert np.array_equal(bits16(W), O.bf16_bits(want))
    f64 = O.bf16_bits(O.apply_update(W0, np32(Ob), lr, wd, sc).astype(np.float32))
    assert np.max(np.abs(bits16(W).astype(np.int32) - f64.astype(np.int32))) <= 1


def test_apply_update_explicit_scale_and_f32(mk):
    gen = torch.Generator("cuda").manual_seed(15)
    W = torch.randn(2, 64, 96, generator=gen, device="cuda")
    Ob = torch.randn(2, 64, 96, generator=gen, device="cuda")
    W0 = np32(W)
    mk.muon_apply_update_f32(W, Ob, lr=f32(0.05), weight_decay=f32(0.01), scale=f32(0.2 * 96 ** 0.5))
    want = O.apply_update_fp32(W0, np32(Ob), f32(0.05), f32(0.01), f32(0.2 * 96 ** 0.5), to_bf16=False)
    assert np.array_equal(bits32(W), want.view(np.uint32))


# ----------------------------------------------------------------------------- Newton-Schulz, fp32 mode
@pytest.mark.parametrize("count,m,n", [(8, 64, 256), (4, 16, 48), (3, 37, 53), (2, 53, 37), (2, 70, 70), (1, 1, 9)])
def test_ns_f32_matches_oracle(mk, count, m, n):
    gen = torch.Generator("cuda").manual_seed(1000 + m * n)
    X = torch.randn(count, m, n, generator=gen, device="cuda")
    want = O.newton_schulz_batched(np32(X))
    mk.muon_ns_batched_f32(X)
    assert rel_fro(np32(X), want) < F32_TOL


def test_tiny_f32_step(mk):
    cfg = workloads.WORKLOADS["tiny_f32_8x64x256"]
    grp = cfg.groups[0]
    dev = "cuda"
    W = workloads.parameters(grp.count, grp.rows, grp.cols, workloads.seed_for(cfg.index, 0, 0, 1), device=dev,
                             dtype=torch.float32)
    buf = torch.zeros_like(W)
    u = torch.empty_like(W)
    for step in range(cfg.steps):
        g = workloads.gradients(grp.count, grp.rows, grp.cols, workloads.seed_for(cfg.index, step, 0, 0), device=dev,
                                kind="normal", dtype=torch.float32)
        ref = O.muon_step(np32(W), np32(g), np32(buf), mu=f32(0.95), lr=f32(0.02), weight_decay=f32(0.1), bf16=False)
        mk.muon_momentum_update_f32(g, buf, u, mu=0.95)
        assert np.array_equal(bits32(buf), ref["buf"].view(np.uint32))
        assert np.array_equal(bits32(u), ref["u"].view(np.uint32))
        mk.muon_ns_batched_f32(u)
        assert rel_fro(np32(u), ref["O"]) < F32_TOL
        W_prev = np32(W)
        mk.muon_apply_update_f32(W, u, lr=0.02, weight_decay=0.1)
        want = O.apply_update_fp32(W_prev, np32(u), f32(0.02), f32(0.1), O.default_scale(grp.rows, grp.cols),
                                   to_bf16=False)
        assert np.array_equal(bits32(W), want.view(np.uint32))
        assert rel_fro(np32(W), ref["param"]) < 1e-6


# ----------------------------------------------------------------------------- Newton-Schulz, bf16 tensor cores
def run_bf16_ns(mk, X, steps=5, coeffs=O.QUINTIC, eps=1e-7):
    x_in = np32(X)
    mk.muon_ns_batched(X, steps=steps, coeffs=coeffs, eps=eps)
    assert mk.muon_get_device_status() == 0
    want = O.newton_schulz_batched(x_in, steps, coeffs, eps)
    return np32(X), want


@pytest.mark.parametrize("coeffs,name", [((0.0, 1.0, 0.0), "syrk+axpy"), ((0.0, 0.0, 1.0), "poly"),
                                         ((1.0, 0.0, 0.0), "epilogue-only"), ((3.4445, -4.775, 2.0315), "quintic")])
def test_ns_bf16_one_step_isolates_kernels(mk, coeffs, name):
    # (0,1,0): X1 = s^3 X X^T X (A from syrk, B = A, X-operand MN-major in axpy)
    # (0,0,1): X1 = s^5 (X X^T)^2 X (exercises the A A product)
    gen = torch.Generator("cuda").manual_seed(21)
    X = torch.randn(2, 256, 512, generator=gen, device="cuda").to(torch.bfloat16)
    got, want = run_bf16_ns(mk, X, steps=1, coeffs=coeffs)
    assert rel_fro(got, want) < BF16_TOL, name


@pytest.mark.parametrize("count,m,n", [(2, 200, 520), (3, 128, 256), (1, 64, 64), (2, 520, 200), (1, 8, 8),
                                       (4, 136, 1032), (2, 384, 384), (1, 1792, 640), (1, 8, 4096)])
def test_ns_bf16_matches_oracle_small(mk, count, m, n):
    X = workloads.gradients(count, m, n, 3000 + m + n, device="cuda", kind="lognormal_rows")
    got, want = run_bf16_ns(mk, X)
    err = rel_fro(got, want)
    print(f"{count}x{m}x{n}: rel {err:.3e}")
    assert err < BF16_TOL


def test_ns_bf16_steps_zero_is_normalisation(mk):
    X = workloads.gradients(3, 96, 160, 31, device="cuda")
    got, want = run_bf16_ns(mk, X, steps=0)
    assert rel_fro(got, want) < 4e-3


def test_ns_bf16_zero_matrix_and_batch_zero(mk):
    X = torch.zeros(2, 64, 128, dtype=torch.bfloat16, device="cuda")
    mk.muon_ns_batched(X)
    assert torch.all(X == 0).item()
    E = torch.empty(0, 64, 128, dtype=torch.bfloat16, device="cuda")
    mk.muon_ns_batched(E)


def test_ns_bf16_with_caller_workspace(mk):
    X = workloads.gradients(3, 256, 768, 41, device="cuda")
    X2 = X.clone()
    ws = torch.empty(mk.muon_ns_workspace_bytes(3, 256, 768), dtype=torch.uint8, device="cuda")
    mk.muon_ns_batched(X, workspace=ws)
    mk.muon_ns_batched(X2)
    assert torch.equal(X, X2)


def test_ns_bf16_unsupported_shapes_are_rejected(mk):
    X = torch.zeros(1, 12, 30, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mk.MuonError) as e:
        mk.muon_ns_batched(X)
    assert e.value.status == -2


def test_wait_timeout_is_reported_and_context_survives(mk):
    mk.muon_selftest_wait_timeout(2_000_000)  # 2 ms, nothing completes the barrier
    assert mk.muon_get_device_status() == -5
    assert mk.muon_get_device_status() == 0   # cleared
    X = workloads.gradients(1, 128, 256, 51, device="cuda")
    got, want = run_bf16_ns(mk, X)
    assert rel_fro(got, want) < BF16_TOL


def test_trace_counts_launches(mk):
    X = workloads.gradients(2, 128, 512, 61, device="cuda")
    n0 = mk.muon_launch_count()
    mk.muon_trace_begin()
    mk.muon_ns_batched(X)
    tr = mk.muon_trace_end()
    assert tr["ns_syrk_tc"][0] == 5 and tr["ns_poly_tc"][0] == 5 and tr["ns_axpy_tc"][0] == 5
    assert all(ms > 0 for _, ms in tr.values())
    assert mk.muon_launch_count() - n0 >= 17


@pytest.mark.parametrize("index", [0, 3])
def test_ns_bf16_low_rank_and_ill_conditioned(mk, index):
    # spectra down to 1e-6 (index 3) and rank 16 (index 0): the small singular
    # values are multiplied by up to 3.4445 per step, so this fails if X is
    # rounded to bf16 between the steps instead of kept as hi + lo
    U, s, V = workloads.spectrum_factors(256, 768, index, device="cuda", dtype=torch.float32, low_rank=16)
    X = ((U * s.unsqueeze(0)) @ V.T).to(torch.bfloat16).unsqueeze(0).contiguous()
    got, want = run_bf16_ns(mk, X)
    assert rel_fro(got, want) < BF16_TOL


# ----------------------------------------------------------------------------- coefficient schedules
# Schedules whose composite scalar map stays positive and well conditioned on
# (0, 1] (relative sensitivity <= ~10): a schedule whose map crosses zero has
# unbounded relative sensitivity there, and no bf16 computation can meet a
# relative tolerance on it.
SCHEDULES = {
    "quintic_then_cubic": [O.QUINTIC] * 5 + [O.CUBIC] * 3,
    "varied": [O.QUINTIC, (3.0, -3.2, 1.2), O.QUINTIC, (2.0, -1.5, 0.5)],
}


@pytest.mark.parametrize("name", sorted(SCHEDULES))
@pytest.mark.parametrize("count,m,n", [(3, 256, 768), (2, 640, 200)])
def test_ns_schedule_bf16_matches_oracle(mk, name, count, m, n):
    rows = SCHEDULES[name]
    X = workloads.gradients(count, m, n, 5000 + m, device="cuda")
    x_in = np32(X)
    mk.muon_ns_batched_schedule(X, rows)
    assert mk.muon_get_device_status() == 0
    want = O.newton_schulz_batched(x_in, len(rows), rows)
    assert rel_fro(np32(X), want) < BF16_TOL


@pytest.mark.parametrize("name", sorted(SCHEDULES))
def test_ns_schedule_f32_matches_oracle(mk, name):
    rows = SCHEDULES[name]
    gen = torch.Generator("cuda").manual_seed(77)
    X = torch.randn(4, 48, 96, generator=gen, device="cuda")
    want = O.newton_schulz_batched(np32(X), len(rows), rows)
    mk.muon_ns_batched_schedule_f32(X, rows)
    assert rel_fro(np32(X), want) < F32_TOL


def test_ns_schedule_of_equal_rows_is_the_constant_call(mk):
    X = workloads.gradients(2, 128, 512, 91, device="cuda")
    Y = X.clone()
    mk.muon_ns_batched(X, steps=5)
    mk.muon_ns_batched_schedule(Y, [O.QUINTIC] * 5)
    assert torch.equal(X, Y)
