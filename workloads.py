"""Seeded synthetic inputs for the Muon step (shared by tests and bench.py).

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no momentum, normalisation, Newton-Schulz or update).
Shapes follow the model-configuration table of "Training a 1T-Parameter MoE on
EU public infrastructure with PyTorch and TorchTitan": hidden size 6144, expert
hidden size 1792, 384 routed experts.  An expert holds w1 and w3 stored as
6144 x 1792 and w2 stored as 1792 x 6144.

Recipe (all seeded, torch's own generators; device chosen by the caller):
* gradients: N(0,1) times a per-stored-row log-normal factor exp(N(0,1)),
  rounded to bf16 (configs 2 and 3), or plain N(0,1) (configs 1 and 4);
* parameters: N(0, 0.02), bf16 (fp32 for config 1);
* momentum: zero at the first step;
* spectrum matrices (config 5): U diag(s) V^T with U Haar on O(m), V the
  thin Haar factor of an n x m Gaussian (QR with the sign of R's diagonal
  folded in), s log-uniform in [1e-6, 1]; every tenth matrix keeps only its
  64 largest singular values.
Seeds: 1234 + 1000*config + 100000*step + 10*group + kind, with kind 0 for
gradients and 1 for parameters; config-5 matrix i uses 1234 + 5000 + 7 + 13*i.
"""

from __future__ import annotations

import dataclasses
import math

import torch

HIDDEN = 6144
EXPERT_HIDDEN = 1792
ROUTED_EXPERTS = 384


@dataclasses.dataclass(frozen=True)
class Group:
    count: int
    rows: int
    cols: int


@dataclasses.dataclass(frozen=True)
class Workload:
    index: int          # enters the seeds (seed_for)
    name: str
    groups: tuple
    dtype: str          # "bf16" or "f32"
    grad_kind: str      # "lognormal_rows", "normal" or "spectrum"
    steps: int          # optimizer steps the workload is run for


WORKLOADS = {w.name: w for w in (
    Workload(1, "tiny_f32_8x64x256", (Group(8, 64, 256),), "f32", "normal", 3),
    Workload(2, "one_expert_w1w3w2", (Group(2, HIDDEN, EXPERT_HIDDEN), Group(1, EXPERT_HIDDEN, HIDDEN)),
             "bf16", "lognormal_rows", 3),
    Workload(3, "rank_expert_batch_96", (Group(64, HIDDEN, EXPERT_HIDDEN), Group(32, EXPERT_HIDDEN, HIDDEN)),
             "bf16", "lognormal_rows", 1),
    Workload(4, "dense_projections", (Group(8, HIDDEN, HIDDEN), Group(4, HIDDEN, 1024)), "bf16", "normal", 1),
    Workload(5, "conditioning_stress_128", (Group(128, EXPERT_HIDDEN, HIDDEN),), "bf16", "spectrum", 1),
)}

TINY_SVD_GROUP = Group(4, 16, 48)


def seed_for(index: int, step: int = 0, group: int = 0, kind: int = 0) -> int:
    return 1234 + 1000 * index + 100000 * step + 10 * group + kind


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def gradients(count: int, rows: int, cols: int, seed: int, device="cpu", kind: str = "lognormal_rows",
              dtype=torch.bfloat16) -> torch.Tensor:
    """A (count, rows, cols) stack of synthetic gradients."""
    g = _gen(device, seed)
    z = torch.randn(count, rows, cols, generator=g, device=device, dtype=torch.float32)
    if kind == "lognormal_rows":
        row = torch.randn(count, rows, 1, generator=g, device=device, dtype=torch.float32)
        z.mul_(torch.exp(row))
    elif kind != "normal":
        raise ValueError(kind)
    return z.to(dtype)


def parameters(count: int, rows: int, cols: int, seed: int, device="cpu", dtype=torch.bfloat16,
               std: float = 0.02) -> torch.Tensor:
    g = _gen(device, seed)
    return (torch.randn(count, rows, cols, generator=g, device=device, dtype=torch.float32) * std).to(dtype)


def spectrum_seed(index: int) -> int:
    return 1234 + 5000 + 7 + 13 * index


def spectrum_factors(m: int, n: int, index: int, device="cpu", dtype=torch.float64, low: float = 1e-6,
                     rank_every: int = 10, low_rank: int = 64):
    """(U, s, V) with U m x m, V n x m orthonormal columns, s log-uniform, for matrix ``index``."""
    g = _gen(device, spectrum_seed(index))
    gu = torch.randn(m, m, generator=g, device=device, dtype=dtype)
    gv = torch.randn(n, m, generator=g, device=device, dtype=dtype)
    u01 = torch.rand(m, generator=g, device=device, dtype=dtype)
    qu, ru = torch.linalg.qr(gu)
    U = qu * torch.sign(torch.diagonal(ru)).unsqueeze(0)
    qv, rv = torch.linalg.qr(gv)
    V = qv * torch.sign(torch.diagonal(rv)).unsqueeze(0)
    s = torch.exp(math.log(low) * u01)                  # log-uniform in [low, 1]
    s, _ = torch.sort(s, descending=True)
    if rank_every and index % rank_every == 0:
        s[low_rank:] = 0
    return U, s, V


def spectrum_matrix(m: int, n: int, index: int, device="cpu", dtype=torch.float64, out_dtype=torch.bfloat16):
    """G = U diag(s) V^T (m x n) and its factors, G rounded to ``out_dtype``."""
    U, s, V = spectrum_factors(m, n, index, device=device, dtype=dtype)
    G = (U * s.unsqueeze(0)) @ V.T
    return G.to(out_dtype), (U, s, V)


def spectrum_batch(count: int, m: int, n: int, device="cpu", dtype=torch.float32, out_dtype=torch.bfloat16,
                   first: int = 0) -> torch.Tensor:
    out = torch.empty(count, m, n, device=device, dtype=out_dtype)
    for i in range(count):
        out[i] = spectrum_matrix(m, n, first + i, device=device, dtype=dtype, out_dtype=out_dtype)[0]
    return out
