"""Pins of the fp64 oracle against what the mathematics fixes (CPU only).

Newton-Schulz with coefficients (a, b, c) maps X = U S V^T to
U (a S + b S^3 + c S^5) V^T, because A = X X^T = U S^2 U^T and
B X = U (b S^2 + c S^4) S V^T.  After the Frobenius normalisation
X0 = G / (||G||_F + eps), k iterations therefore give U p^k(S0) V^T with
S0 = S / (||G||_F + eps).  ("Training a 1T-Parameter MoE on EU public
infrastructure with PyTorch and TorchTitan", section "FlexShard: Muon without
communication": a few Newton-Schulz iterations on the whole matrix.)
Every check below uses a route that does not go through the oracle's own
code: numpy's SVD, exact rational arithmetic, orthogonal factors built by QR,
torch's bf16 conversion, or hand-derived values.
"""

import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import workloads
from oracle import muon_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rel_fro(x, y):
    x = np.asarray(x, np.float64)
    y = np.asarray(y, np.float64)
    return float(np.linalg.norm(x - y) / max(np.linalg.norm(y), 1e-300))


def scalar_map(s, coeffs, k):
    a, b, c = coeffs
    s = np.asarray(s, np.float64)
    for _ in range(k):
        s = a * s + b * s ** 3 + c * s ** 5
    return s


def closed_form(G, steps, coeffs, eps):
    """U p^k(S / (||G||_F + eps)) V^T from numpy's SVD."""
    U, S, Vt = np.linalg.svd(np.asarray(G, np.float64), full_matrices=False)
    fro = math.sqrt(float(np.sum(S * S)))
    return (U * scalar_map(S / (fro + eps), coeffs, steps)) @ Vt


def haar(n, rng):
    q, r = np.linalg.qr(rng.standard_normal((n, n)))
    return q * np.sign(np.diag(r))


# --------------------------------------------------------------------------
# bf16 rounding
# --------------------------------------------------------------------------
def test_bf16_golden_cases():
    rows = []
    with open(os.path.join(GOLDEN, "bf16_rne_cases.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                src, dst = line.split()[:2]
                rows.append((int(src, 16), int(dst, 16)))
    assert len(rows) >= 15
    src = np.array([r[0] for r in rows], dtype=np.uint32).view(np.float32)
    want = np.array([r[1] for r in rows], dtype=np.uint16)
    got = O.bf16_bits(src)
    assert np.array_equal(got, want), [(hex(a), hex(b), hex(c)) for a, b, c in zip(src.view(np.uint32), want, got) if b != c]


def test_bf16_matches_torch_conversion():
    rng = np.random.default_rng(7)
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-60, 60, 200000))).astype(np.float32)
    x[:16] = [0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, 3e38, -3e38, 1e-40, -1e-40, 1e-45, 65504.0, 0.5, 2.0, 1.00390625, 1.01171875]
    ours = O.bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = O.bf16_from_bits(ours)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


# --------------------------------------------------------------------------
# momentum
# --------------------------------------------------------------------------
def test_momentum_exact_rational_sequence():
    # mu = 1/2 and small dyadic values keep every intermediate exact in fp32,
    # so the fp32 result must equal exact rational arithmetic.
    rng = np.random.default_rng(1)
    g_steps = [rng.integers(-64, 64, size=32).astype(np.float32) / 4 for _ in range(4)]
    buf = (rng.integers(-32, 32, size=32).astype(np.float32) / 8)
    fb = [Fraction(float(v)) for v in buf]
    mu = Fraction(1, 2)
    for g in g_steps:
        for nesterov in (True, False):
            nb, u = O.momentum_update(g, buf, 0.5, nesterov)
            want_b = [mu * b + Fraction(float(x)) for b, x in zip(fb, g)]
            want_u = [Fraction(float(x)) + mu * b for b, x in zip(want_b, g)] if nesterov else want_b
            assert [Fraction(float(v)) for v in nb] == want_b
            assert [Fraction(float(v)) for v in u] == want_u
        buf = nb
        fb = want_b


def test_momentum_uses_new_buffer_for_nesterov():
    g = np.array([1.0], np.float32)
    b0 = np.array([4.0], np.float32)
    nb, u = O.momentum_update(g, b0, 0.5, True)
    assert nb[0] == 3.0          # 0.5*4 + 1
    assert u[0] == 2.5           # 1 + 0.5*3 (new buffer); the old buffer would give 3.0


def test_momentum_constant_gradient_geometric_series():
    rng = np.random.default_rng(2)
    g = rng.standard_normal(1000).astype(np.float32)
    buf = np.zeros_like(g)
    mu = 0.95
    for k in range(1, 31):
        buf, u = O.momentum_update(g, buf, mu, True)
        geo = g.astype(np.float64) * (1 - mu ** k) / (1 - mu)
        assert rel_fro(buf, geo) < 2e-6
        nest = g.astype(np.float64) + mu * geo
        assert rel_fro(u, nest) < 2e-6


def test_momentum_special_cases():
    rng = np.random.default_rng(3)
    g = rng.standard_normal(257).astype(np.float32)
    b = rng.standard_normal(257).astype(np.float32)
    nb, u = O.momentum_update(g, b, 0.0, True)
    assert np.array_equal(nb, g) and np.array_equal(u, g)
    nb, u = O.momentum_update(g, b, 0.9, False)
    assert np.array_equal(u, nb)


def test_momentum_ema_form_is_proportional():
    # EMA form buf <- mu buf + (1-mu) g, u <- (1-mu) g + mu buf equals (1-mu) times
    # the SGD form from a zero start, so the normalised NS input is the same.
    rng = np.random.default_rng(4)
    mu = 0.95
    buf = np.zeros((16, 48), np.float32)
    ema = np.zeros((16, 48), np.float64)
    for _ in range(4):
        g = rng.standard_normal((16, 48)).astype(np.float32)
        buf, u = O.momentum_update(g, buf, mu, True)
        ema = mu * ema + (1 - mu) * g
        u_ema = (1 - mu) * g + mu * ema
        assert rel_fro(u_ema, (1 - mu) * u.astype(np.float64)) < 1e-6
    ns_sgd = O.newton_schulz(u, eps=0.0)
    ns_ema = O.newton_schulz(u_ema, eps=0.0)
    assert rel_fro(ns_ema, ns_sgd) < 1e-5


# --------------------------------------------------------------------------
# Newton-Schulz
# --------------------------------------------------------------------------
@pytest.mark.parametrize("count,m,n", [(4, 16, 48), (8, 64, 256), (2, 48, 16), (2, 32, 32), (1, 40, 200)])
def test_ns_matches_svd_closed_form(count, m, n):
    rng = np.random.default_rng(100 + m + n)
    for _ in range(count):
        G = rng.standard_normal((m, n))
        got = O.newton_schulz(G, 5, O.QUINTIC, 1e-7)
        assert rel_fro(got, closed_form(G, 5, O.QUINTIC, 1e-7)) < 1e-10


def test_ns_closed_form_with_other_steps_and_coeffs():
    rng = np.random.default_rng(11)
    G = rng.standard_normal((24, 40)) * np.exp(rng.standard_normal((24, 1)))
    for steps, coeffs in [(1, O.QUINTIC), (3, (2.0, -1.5, 0.5)), (7, O.QUINTIC), (4, O.CUBIC)]:
        got = O.newton_schulz(G, steps, coeffs, 1e-7)
        assert rel_fro(got, closed_form(G, steps, coeffs, 1e-7)) < 1e-10


def test_ns_constructed_spectrum_and_null_space():
    m, n = 64, 256
    for index in (0, 3):          # index 0 is rank-64 -> full rank here; use rank 20 below
        U, s, V = workloads.spectrum_factors(m, n, index, dtype=torch.float64, low=1e-6, rank_every=10, low_rank=20)
        U, s, V = U.numpy(), s.numpy(), V.numpy()
        G = (U * s) @ V.T
        Ons = O.newton_schulz(G, 5, O.QUINTIC, 1e-7)
        core = U.T @ Ons @ V
        want = scalar_map(s / (math.sqrt(float(np.sum(s * s))) + 1e-7), O.QUINTIC, 5)
        assert np.max(np.abs(np.diag(core) - want)) < 1e-10
        assert np.max(np.abs(core - np.diag(np.diag(core)))) < 1e-10
        if index == 0:
            assert np.all(s[20:] == 0)
            # directions outside the row space map to zero
            rest = V[:, 20:]
            assert np.max(np.abs(Ons @ rest)) < 1e-12


@pytest.mark.slow
def test_ns_constructed_spectrum_full_expert_shape():
    # one 1792 x 6144 expert-shaped matrix with a known spectrum (no SVD needed)
    U, s, V = workloads.spectrum_factors(1792, 6144, 3, dtype=torch.float64)
    U, s, V = U.numpy(), s.numpy(), V.numpy()
    G = (U * s) @ V.T
    Ons = O.newton_schulz(G)
    core = U.T @ Ons @ V
    want = scalar_map(s / (math.sqrt(float(np.sum(s * s))) + 1e-7), O.QUINTIC, 5)
    assert np.max(np.abs(np.diag(core) - want)) < 1e-9
    assert np.max(np.abs(core - np.diag(np.diag(core)))) < 1e-9
    # the transposed (w1/w3-like) orientation gives the transposed result
    OT = O.newton_schulz(G.T)
    assert np.array_equal(OT, Ons.T)


def test_ns_cubic_converges_to_polar_factor():
    rng = np.random.default_rng(12)
    for m, n in [(16, 48), (48, 16), (20, 20)]:
        k = min(m, n)
        U = haar(m, rng)[:, :k]
        V = haar(n, rng)[:, :k]
        s = np.exp(rng.uniform(math.log(1e-2), 0, k))
        G = (U * s) @ V.T
        got = O.newton_schulz(G, 50, O.CUBIC, 1e-7)
        assert rel_fro(got, U @ V.T) < 1e-10


def test_ns_orthogonal_equivariance():
    rng = np.random.default_rng(13)
    G = rng.standard_normal((16, 48))
    Q = haar(16, rng)
    R = haar(48, rng)
    lhs = O.newton_schulz(Q @ G @ R)
    rhs = Q @ O.newton_schulz(G) @ R
    assert rel_fro(lhs, rhs) < 1e-12


def test_ns_scale_invariance():
    rng = np.random.default_rng(14)
    G = rng.standard_normal((32, 96))
    for alpha in (1e-3, 37.5, 1e6):
        assert rel_fro(O.newton_schulz(alpha * G, eps=0.0), O.newton_schulz(G, eps=0.0)) < 1e-13


def test_ns_transpose_symmetry_exact():
    rng = np.random.default_rng(15)
    G = rng.standard_normal((24, 72))
    assert np.array_equal(O.newton_schulz(G.T), O.newton_schulz(G).T)


def test_ns_diagonal_against_exact_rationals():
    # G = diag(3, 4) * 0.25 padded to 4 x 8, with eps: s0 = s / (||s|| + eps) and
    # the quintic is evaluated in exact rational arithmetic.
    eps = 1e-7
    G = np.zeros((4, 8))
    G[0, 0], G[1, 1] = 0.75, 1.0
    got = O.newton_schulz(G, 5, O.QUINTIC, eps)
    a, b, c = (Fraction(str(v)) for v in O.QUINTIC)
    # ||s|| = 1.25 exactly
    denom = Fraction(5, 4) + Fraction(eps)
    want = []
    for sv in (Fraction(3, 4), Fraction(1)):
        x = sv / denom
        for _ in range(5):
            x = a * x + b * x ** 3 + c * x ** 5
        want.append(float(x))
    assert abs(got[0, 0] - want[0]) < 1e-13 and abs(got[1, 1] - want[1]) < 1e-13
    mask = np.ones_like(got, bool)
    mask[0, 0] = mask[1, 1] = False
    assert np.all(got[mask] == 0.0)


def test_ns_zero_matrix_gives_zero():
    out = O.newton_schulz(np.zeros((8, 24)))
    assert np.all(out == 0.0) and np.all(np.isfinite(out))


def test_ns_eps_placement_near_eps_scale():
    # ||G|| comparable to eps: the closed form with eps added to the norm must hold
    rng = np.random.default_rng(16)
    G = rng.standard_normal((12, 20))
    G *= 5e-8 / np.linalg.norm(G)
    got = O.newton_schulz(G, 5, O.QUINTIC, 1e-7)
    assert rel_fro(got, closed_form(G, 5, O.QUINTIC, 1e-7)) < 1e-10
    # and differs clearly from the eps-free result
    assert rel_fro(got, closed_form(G, 5, O.QUINTIC, 0.0)) > 1e-2


def test_ns_zero_steps_is_normalisation():
    rng = np.random.default_rng(17)
    G = rng.standard_normal((10, 30))
    got = O.newton_schulz(G, 0, O.QUINTIC, 1e-7)
    assert rel_fro(got, G / (np.linalg.norm(G) + 1e-7)) < 1e-15


def test_quintic_facts():
    # fixed points and growth of the scalar map used throughout
    assert abs(scalar_map(1e-6, O.QUINTIC, 5) - 3.4445 ** 5 * 1e-6) / (3.4445 ** 5 * 1e-6) < 1e-6
    xs = np.exp(np.linspace(math.log(1e-2), 0, 2000))
    ys = scalar_map(xs, O.QUINTIC, 5)
    assert 0.6 < ys.min() and ys.max() < 1.2


PLANTED = {
    "square_dropped": ("poly", lambda A, b, c: b * A + c * A),
    "sign_flipped": ("poly", lambda A, b, c: b * A - c * (A @ A)),
    "update_sign": ("axpy_update", lambda X, B, a: a * X - B @ X),
    "update_missing_aX": ("axpy_update", lambda X, B, a: B @ X),
    "gram_halved": ("gram", lambda X: 0.5 * (X @ X.T)),
    "maxabs_norm": ("frobenius_normalise", lambda X, eps: np.asarray(X, np.float64) / (np.abs(X).max() + eps)),
    "squared_norm_eps": ("frobenius_normalise",
                         lambda X, eps: np.asarray(X, np.float64) / math.sqrt(float(np.sum(np.asarray(X) ** 2)) + eps)),
}


@pytest.mark.parametrize("name", sorted(PLANTED))
def test_planted_mistakes_are_caught(monkeypatch, name):
    attr, bad = PLANTED[name]
    monkeypatch.setattr(O, attr, bad)
    rng = np.random.default_rng(18)
    caught = False
    for G in (rng.standard_normal((16, 48)), 1e-8 * rng.standard_normal((16, 48)) / 7):
        got = O.newton_schulz(G, 5, O.QUINTIC, 1e-7)
        if not np.all(np.isfinite(got)) or rel_fro(got, closed_form(G, 5, O.QUINTIC, 1e-7)) > 1e-6:
            caught = True
    assert caught, name


def test_planted_coefficient_order_is_caught():
    rng = np.random.default_rng(19)
    G = rng.standard_normal((16, 48))
    a, b, c = O.QUINTIC
    got = O.newton_schulz(G, 5, (a, c, b), 1e-7)
    assert rel_fro(got, closed_form(G, 5, O.QUINTIC, 1e-7)) > 1e-3


# --------------------------------------------------------------------------
# update
# --------------------------------------------------------------------------
def test_default_scale_values():
    assert O.default_scale(6144, 1792) == math.sqrt(24 / 7)
    assert abs(O.default_scale(6144, 1792) - 1.8516401995451028) < 1e-15
    assert O.default_scale(1792, 6144) == 1.0
    assert O.default_scale(6144, 6144) == 1.0
    assert O.default_scale(6144, 1024) == math.sqrt(6.0)


def test_apply_update_closed_forms():
    rng = np.random.default_rng(20)
    W = rng.integers(-100, 100, (8, 16)).astype(np.float64) / 64
    Ob = rng.integers(-100, 100, (8, 16)).astype(np.float64) / 64
    assert np.array_equal(O.apply_update(W, Ob, 0.0, 0.1, 2.0), W)
    assert np.array_equal(O.apply_update(W, Ob, 0.5, 0.0, 1.0), W - 0.5 * Ob)
    assert np.array_equal(O.apply_update(W, Ob, 0.25, 2.0, 2.0), 0.5 * W - 0.5 * Ob)
    # fp32 statement agrees with the fp64 one exactly on dyadic data
    assert np.array_equal(O.apply_update_fp32(W, Ob, 0.25, 2.0, 2.0, to_bf16=False), 0.5 * W - 0.5 * Ob)


def test_apply_update_fp32_within_one_bf16_ulp_of_fp64():
    rng = np.random.default_rng(21)
    W = O.bf16_round((rng.standard_normal(100000) * 0.02).astype(np.float32))
    Ob = O.bf16_round((rng.standard_normal(100000) * 0.02).astype(np.float32))
    f32 = O.apply_update_fp32(W, Ob, 0.02, 0.1, 1.8516401995451028)
    f64 = O.bf16_round(O.apply_update(W, Ob, 0.02, 0.1, 1.8516401995451028).astype(np.float32))
    diff = np.abs(f32.view(np.uint32).astype(np.int64) - f64.view(np.uint32).astype(np.int64)) >> 16
    assert diff.max() <= 1


def test_step_resume_is_bit_exact(tmp_path):
    # 3 steps straight == 2 steps, save/reload momentum, 1 step
    rng = np.random.default_rng(22)
    shape = (2, 16, 40)
    grads = [O.bf16_round(rng.standard_normal(shape).astype(np.float32)) for _ in range(3)]
    W0 = O.bf16_round((0.02 * rng.standard_normal(shape)).astype(np.float32))
    buf = np.zeros(shape, np.float32)
    W = W0
    outs = []
    for g in grads:
        r = O.muon_step(W, g, buf)
        buf, W = r["buf"], O.bf16_round(r["param"].astype(np.float32))
        outs.append((buf, W))
    buf2 = np.zeros(shape, np.float32)
    W2 = W0
    for g in grads[:2]:
        r = O.muon_step(W2, g, buf2)
        buf2, W2 = r["buf"], O.bf16_round(r["param"].astype(np.float32))
    np.save(tmp_path / "m.npy", buf2)
    buf2 = np.load(tmp_path / "m.npy")
    r = O.muon_step(W2, grads[2], buf2)
    assert np.array_equal(r["buf"], outs[2][0])
    assert np.array_equal(O.bf16_round(r["param"].astype(np.float32)), outs[2][1])


def test_workload_shapes_follow_the_pages():
    facts = {}
    with open(os.path.join(GOLDEN, "pages_expert_shapes.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, v = line.split()
                facts[k] = int(v)
    assert workloads.HIDDEN == facts["hidden"]
    assert workloads.EXPERT_HIDDEN == facts["expert_hidden"]
    assert workloads.ROUTED_EXPERTS == facts["routed_experts"]
    batch = workloads.WORKLOADS["rank_expert_batch_96"]
    shapes = {(g.rows, g.cols) for g in batch.groups}
    assert shapes == {(facts["hidden"], facts["expert_hidden"]), (facts["expert_hidden"], facts["hidden"])}
    assert sum(g.count for g in batch.groups) == 96   # 32 experts x (w1, w3, w2)


# --------------------------------------------------------------------------
# coefficient schedules (one (a, b, c) per step)
# --------------------------------------------------------------------------
def schedule_map(s, rows):
    s = np.asarray(s, np.float64)
    for a, b, c in rows:
        s = a * s + b * s ** 3 + c * s ** 5
    return s


def test_schedule_matches_svd_closed_form():
    rng = np.random.default_rng(30)
    rows = [(4.0, -5.0, 2.0), (3.4445, -4.7750, 2.0315), (2.0, -1.5, 0.5), (1.5, -0.5, 0.0)]
    for m, n in [(16, 48), (48, 16), (24, 24)]:
        G = rng.standard_normal((m, n))
        got = O.newton_schulz(G, len(rows), rows, 1e-7)
        U, S, Vt = np.linalg.svd(G, full_matrices=False)
        want = (U * schedule_map(S / (math.sqrt(float(np.sum(S * S))) + 1e-7), rows)) @ Vt
        assert rel_fro(got, want) < 1e-10


def test_schedule_of_identical_rows_equals_constant_coefficients():
    rng = np.random.default_rng(31)
    G = rng.standard_normal((20, 60))
    assert np.array_equal(O.newton_schulz(G, 5, [O.QUINTIC] * 5), O.newton_schulz(G, 5, O.QUINTIC))


def test_schedule_order_matters():
    # the step maps do not commute in general: reversing the schedule changes the result
    rng = np.random.default_rng(32)
    G = rng.standard_normal((16, 40))
    rows = [(3.4445, -4.7750, 2.0315), (1.5, -0.5, 0.0), (2.0, -1.5, 0.5)]
    assert rel_fro(O.newton_schulz(G, 3, rows), O.newton_schulz(G, 3, rows[::-1])) > 1e-3


def test_quintic_then_cubic_reaches_polar_factor():
    rng = np.random.default_rng(33)
    U = haar(16, rng)
    V = haar(48, rng)[:, :16]
    s = np.exp(rng.uniform(math.log(1e-2), 0, 16))
    G = (U * s) @ V.T
    rows = [O.QUINTIC] * 5 + [O.CUBIC] * 12
    assert rel_fro(O.newton_schulz(G, len(rows), rows), U @ V.T) < 1e-10


def test_schedule_shape_is_checked():
    with pytest.raises(ValueError):
        O.newton_schulz(np.ones((4, 8)), 3, [O.QUINTIC] * 2)


# --------------------------------------------------------------------------
# the whole step: momentum -> bf16(u) -> Newton-Schulz -> update
# --------------------------------------------------------------------------
# Each pin below reaches the step's result through a route that does not use
# the oracle's composition: torch's own bf16 conversion, numpy's SVD, exact
# dyadic arithmetic.  The planted mistakes are the plausible ones of the
# composition (FlexShard section: one fp32 state per parameter; Newton-Schulz
# on each whole matrix; the update with its shape scale).
def torch_bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).float().numpy()


def step_pins(shape=(2, 16, 40), seed=30):
    """Runs the pins on one stack; returns the list of pins that failed."""
    rng = np.random.default_rng(seed)
    bad = []
    # fp32 gradients that are not bf16 values, so rounding u to bf16 matters
    g = (rng.standard_normal(shape) * (1 + rng.random(shape) / 64)).astype(np.float32)
    zero = np.zeros(shape, np.float32)
    W0 = np.zeros(shape, np.float64)
    # (1) mu = 0 from a zero buffer: u = g exactly, the Newton-Schulz input is
    # bf16(g); with W = 0, lr = 1, wd = 0 and scale 1 the new parameter is -O.
    r = O.muon_step(W0, g, zero, mu=0.0, lr=1.0, weight_decay=0.0, scale=1.0)
    want = np.stack([closed_form(torch_bf16(g[i]), 5, O.QUINTIC, 1e-7) for i in range(shape[0])])
    if not (rel_fro(r["O"], want) < 1e-10 and rel_fro(r["param"], -want) < 1e-10):
        bad.append("ns_input_is_bf16_of_u")
    # (2) lr = 0 leaves the parameters as they were
    W = O.bf16_round((0.02 * rng.standard_normal(shape)).astype(np.float32)).astype(np.float64)
    r = O.muon_step(W, g, zero, lr=0.0, weight_decay=0.1)
    if not np.array_equal(r["param"], W):
        bad.append("lr_zero_is_identity")
    # (3) a zero gradient from a zero buffer gives O = 0: pure decoupled decay,
    # exact on dyadic data (1 - 0.5 * 0.5 = 3/4)
    Wd = rng.integers(-64, 64, shape).astype(np.float64) / 16
    r = O.muon_step(Wd, zero, zero, lr=0.5, weight_decay=0.5)
    if not (np.array_equal(r["O"], np.zeros(shape)) and np.array_equal(r["param"], 0.75 * Wd)):
        bad.append("decay_alone")
    # (4) two momentum steps with mu = 1/2 on dyadic gradients: u2 = g2 + (g1/2 + g2)/2
    # exactly (fp32 and bf16 represent it), O2 = closed form of u2; decay and
    # update combined: W' = (1 - lr wd) W - lr O with dyadic lr, wd
    g1 = rng.integers(-8, 9, shape).astype(np.float32) / 8
    g2 = rng.integers(-8, 9, shape).astype(np.float32) / 8
    r1 = O.muon_step(Wd, g1, zero, mu=0.5, lr=0.25, weight_decay=0.5, scale=1.0)
    r2 = O.muon_step(Wd, g2, r1["buf"], mu=0.5, lr=0.25, weight_decay=0.5, scale=1.0)
    u2 = g2.astype(np.float64) + 0.5 * (0.5 * g1.astype(np.float64) + g2)
    want2 = np.stack([closed_form(u2[i], 5, O.QUINTIC, 1e-7) for i in range(shape[0])])
    if not (np.array_equal(r1["buf"], g1) and np.array_equal(r2["buf"], 0.5 * g1 + g2)
            and rel_fro(r2["O"], want2) < 1e-10
            and rel_fro(r2["param"], 0.875 * Wd - 0.25 * want2) < 1e-12):
        bad.append("nesterov_composition")
    return bad


def scale_pins():
    """The default shape scale on the stored shape, at the pages' expert shapes
    (steps = 0: O is u / (||u|| + eps), cheap at full size)."""
    bad = []
    for (rows, cols), s in (((6144, 1792), math.sqrt(6144 / 1792)), ((1792, 6144), 1.0)):
        g = workloads.gradients(1, rows, cols, 41).float().numpy()
        r = O.muon_step(np.zeros((1, rows, cols)), g, np.zeros((1, rows, cols), np.float32), steps=0,
                        lr=1.0, weight_decay=0.0)
        u = g.astype(np.float64) * (1 + 0.95)          # mu = 0.95 from zero: u = g + 0.95 g
        u = torch_bf16(u.astype(np.float32)).astype(np.float64)
        O0 = u / (math.sqrt(float(np.sum(u * u))) + 1e-7)
        if not rel_fro(r["param"], -s * O0) < 1e-12:
            bad.append(f"scale_{rows}x{cols}")
    return bad


def test_step_composition_pins_hold():
    assert step_pins() == []
    assert step_pins(shape=(1, 40, 16), seed=31) == []


@pytest.mark.slow
def test_step_scale_pins_hold_at_expert_shapes():
    assert scale_pins() == []


PLANTED_STEP = {
    # Newton-Schulz fed the fp32 u instead of bf16(u)
    "u_not_rounded": ("bf16_round", lambda x: np.asarray(x, np.float32), "ns_input_is_bf16_of_u"),
    # Nesterov dropped: the step orthogonalises the buffer
    "buffer_not_u": ("momentum_update",
                     lambda g, b, mu, nesterov=True: (lambda nb: (nb, nb.copy()))(
                         np.add(np.multiply(np.float32(mu), np.asarray(b, np.float32), dtype=np.float32),
                                np.asarray(g, np.float32), dtype=np.float32)),
                     "nesterov_composition"),
    # decay applied to the update instead of the parameter
    "decay_on_update": ("apply_update",
                        lambda W, Ob, lr, wd, s: np.asarray(W, np.float64) - lr * s * (1 - lr * wd) * np.asarray(Ob),
                        "decay_alone"),
}


@pytest.mark.parametrize("name", sorted(PLANTED_STEP))
def test_planted_step_mistakes_are_caught(monkeypatch, name):
    attr, bad_fn, pin = PLANTED_STEP[name]
    monkeypatch.setattr(O, attr, bad_fn)
    assert pin in step_pins()


@pytest.mark.slow
def test_planted_canonical_shape_scale_is_caught(monkeypatch):
    # the scale taken on the m <= n orientation instead of the stored shape
    monkeypatch.setattr(O, "default_scale", lambda r, c: math.sqrt(max(1.0, min(r, c) / max(r, c))))
    assert "scale_6144x1792" in scale_pins()
