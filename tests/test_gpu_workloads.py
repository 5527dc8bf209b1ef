"""Full-size workloads on the GPU, in the launch configuration bench.py times.

Every matrix of a shape group goes through one batched call; the fp64 oracle
then recomputes every matrix of the workload (same bf16 inputs), on all host
cores (tests/_oracle_pool.py).  Momentum is compared bit for bit, the
Newton-Schulz output within 2e-2 relative Frobenius error, the updated
parameters against the update formula applied to the GPU's own orthogonalised
update (bit-exact) and against the fp64 chain (within one bf16 ulp plus
lr*scale times the update difference).  The largest error of each workload is
printed.
"""

import numpy as np
import pytest
import torch

import workloads
from oracle import muon_oracle as O
from tests._oracle_pool import oracle_errors
from tests._util import bits16, bits32, np32, rel_fro, require_gpu

pytestmark = pytest.mark.gpu

BF16_TOL = 2e-2
LR, WD, MU = float(np.float32(0.02)), float(np.float32(0.1)), float(np.float32(0.95))


@pytest.fixture(scope="module")
def mk():
    return require_gpu()


def step_groups(mk, wl, groups, W, buf, u, step):
    grads = []
    for gi, grp in enumerate(groups):
        g = workloads.gradients(grp.count, grp.rows, grp.cols, workloads.seed_for(wl.index, step, gi, 0),
                                device="cuda", kind=wl.grad_kind)
        grads.append(g)
    snap = [(np32(w), np32(b)) for w, b in zip(W, buf)]
    for gi in range(len(groups)):
        mk.muon_momentum_update(grads[gi], buf[gi], u[gi], mu=MU)
    u_in = [u_.clone() for u_ in u]
    for gi in range(len(groups)):
        mk.muon_ns_batched(u[gi])
    for gi in range(len(groups)):
        mk.muon_apply_update(W[gi], u[gi], lr=LR, weight_decay=WD)
    assert mk.muon_get_device_status() == 0
    return grads, snap, u_in


def check_matrix(g, W_prev, b_prev, buf_new, u_in, O_gpu, W_new, rows, cols):
    nb, uu = O.momentum_update(np32(g), b_prev, MU, True)
    assert np.array_equal(bits32(buf_new), nb.view(np.uint32))
    assert np.array_equal(bits16(u_in), O.bf16_bits(uu))
    want = O.newton_schulz(O.bf16_round(uu))
    Og = np32(O_gpu)
    err = rel_fro(Og, want)
    assert err < BF16_TOL, err
    sc = O.default_scale(rows, cols)
    exact = O.apply_update_fp32(W_prev, Og, LR, WD, sc)
    assert np.array_equal(bits16(W_new), O.bf16_bits(exact))
    # fp64 chain: one bf16 ulp of the result plus what the update difference moves
    chain = O.apply_update(W_prev, want, LR, WD, sc)
    Wn = np32(W_new)
    mag = np.maximum(np.abs(Wn), np.abs(chain))
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(mag, 2.0 ** -126))) - 7)
    assert np.all(np.abs(Wn - chain) <= ulp + LR * sc * np.abs(Og - want) * (1 + 1e-6) + 1e-12)
    return err


def test_one_expert_three_steps(mk):
    cfg = workloads.WORKLOADS["one_expert_w1w3w2"]
    groups = cfg.groups
    W = [workloads.parameters(g.count, g.rows, g.cols, workloads.seed_for(cfg.index, 0, gi, 1), device="cuda")
         for gi, g in enumerate(groups)]
    buf = [torch.zeros(g.count, g.rows, g.cols, device="cuda") for g in groups]
    u = [torch.empty(g.count, g.rows, g.cols, dtype=torch.bfloat16, device="cuda") for g in groups]
    errs = []
    for step in range(cfg.steps):
        grads, snap, u_in = step_groups(mk, cfg, groups, W, buf, u, step)
        for gi, grp in enumerate(groups):
            for i in range(grp.count):
                errs.append(check_matrix(grads[gi][i], snap[gi][0][i], snap[gi][1][i], buf[gi][i], u_in[gi][i],
                                         u[gi][i], W[gi][i], grp.rows, grp.cols))
    print("one_expert_w1w3w2 rel errors", ["%.3e" % e for e in errs])


def check_momentum_and_update(g, W_prev, b_prev, buf_new, u_in, O_gpu, W_new, rows, cols):
    """The step's elementwise parts for one matrix; the Newton-Schulz output is
    compared with the oracle separately (oracle_errors)."""
    nb, uu = O.momentum_update(np32(g), b_prev, MU, True)
    assert np.array_equal(bits32(buf_new), nb.view(np.uint32))
    assert np.array_equal(bits16(u_in), O.bf16_bits(uu))
    sc = O.default_scale(rows, cols)
    exact = O.apply_update_fp32(W_prev, np32(O_gpu), LR, WD, sc)
    assert np.array_equal(bits16(W_new), O.bf16_bits(exact))


def test_rank_expert_batch_96_every_matrix(mk):
    cfg = workloads.WORKLOADS["rank_expert_batch_96"]
    groups = cfg.groups
    W = [workloads.parameters(g.count, g.rows, g.cols, workloads.seed_for(cfg.index, 0, gi, 1), device="cuda")
         for gi, g in enumerate(groups)]
    buf = [torch.zeros(g.count, g.rows, g.cols, device="cuda") for g in groups]
    u = [torch.empty(g.count, g.rows, g.cols, dtype=torch.bfloat16, device="cuda") for g in groups]
    grads, snap, u_in = step_groups(mk, cfg, groups, W, buf, u, 0)
    pairs = [(gi, i) for gi, grp in enumerate(groups) for i in range(grp.count)]
    for gi, i in pairs:
        grp = groups[gi]
        check_momentum_and_update(grads[gi][i], snap[gi][0][i], snap[gi][1][i], buf[gi][i], u_in[gi][i], u[gi][i],
                                  W[gi][i], grp.rows, grp.cols)
    res = oracle_errors(((np32(u_in[gi][i]), np32(u[gi][i])) for gi, i in pairs), len(pairs))
    errs = np.array([e for e, _ in res])
    print(f"rank_expert_batch_96: {len(errs)} matrices vs the oracle, rel max {errs.max():.3e} mean {errs.mean():.3e}")
    assert len(errs) == 96 and errs.max() < BF16_TOL


def test_dense_projections_every_matrix(mk):
    cfg = workloads.WORKLOADS["dense_projections"]
    groups = cfg.groups
    X = [workloads.gradients(g.count, g.rows, g.cols, workloads.seed_for(cfg.index, 0, gi, 0), device="cuda", kind="normal")
         for gi, g in enumerate(groups)]
    X_in = [x.clone() for x in X]
    for x in X:
        mk.muon_ns_batched(x)
    assert mk.muon_get_device_status() == 0
    pairs = [(gi, i) for gi, grp in enumerate(groups) for i in range(grp.count)]
    res = oracle_errors(((np32(X_in[gi][i]), np32(X[gi][i])) for gi, i in pairs), len(pairs))
    errs = np.array([e for e, _ in res])
    print(f"dense_projections: {len(errs)} matrices vs the oracle, rel max {errs.max():.3e} mean {errs.mean():.3e}")
    assert len(errs) == 12 and errs.max() < BF16_TOL


def test_conditioning_stress_128_every_matrix(mk):
    cfg = workloads.WORKLOADS["conditioning_stress_128"]
    grp = cfg.groups[0]
    m, n = grp.rows, grp.cols
    G = workloads.spectrum_batch(grp.count, m, n, device="cuda", dtype=torch.float32)
    G_in = G.clone()
    mk.muon_ns_batched(G)
    assert mk.muon_get_device_status() == 0
    assert torch.isfinite(G.float()).all()

    def jobs():
        for i in range(grp.count):
            U, s, V = workloads.spectrum_factors(m, n, i, device="cuda", dtype=torch.float32)
            if i % 10 == 0:
                assert torch.all(s[64:] == 0).item()      # rank-64 matrices: the error check only
                yield np32(G_in[i]), np32(G[i])
            else:                                         # full rank: also the spectrum along U, V
                yield np32(G_in[i]), np32(G[i]), np32(U), np32(s), np32(V)

    res = oracle_errors(jobs(), grp.count)
    errs = np.array([e for e, _ in res])
    devs = np.array([d for _, d in res if d is not None])
    print(f"conditioning_stress_128: {len(errs)} matrices vs the oracle, rel max {errs.max():.3e} "
          f"mean {errs.mean():.3e}; {len(devs)} full-rank spectra, max |diag(U^T O V) - p^5(s)| {devs.max():.3e}")
    assert len(errs) == 128 and errs.max() < BF16_TOL
    assert len(devs) == 115 and devs.max() < 5e-2
