"""A CPU model of where the tensor-core Newton-Schulz rounds, against the oracle.

This is not a pin of the oracle and shares no code with the CUDA path: it
restates, in numpy, the storage formats the CUDA iteration uses, to show what
error they cost against the exact iteration ("Training a 1T-Parameter MoE on
EU public infrastructure with PyTorch and TorchTitan", section "FlexShard:
Muon without communication": a few Newton-Schulz iterations on each whole
matrix) and why the formats were chosen.  The products themselves are taken
exact (the tensor cores accumulate in fp32); what is modelled is the rounding
of what each step stores:

* bf16 scheme: A, B and X's high half in bf16 (what the library does for
  matrices of more than 256 rows);
* fp16 scheme (matrices of up to 256 rows): A, B and X's high half in fp16
  after scaling by a power of two that puts the largest possible entry near
  2^14, except the first step's B in bf16 (it meets the bf16 input in one
  product).
In both, X's low half is kept as an 8-bit e5m2 times a power of two chosen
from the bound on the high half's rounding unit, and the last step's input
carries no low half, as in the library.
The output is rounded to bf16 in both.  On 8 x 8 inputs the bf16 scheme
exceeds the 2e-2 relative Frobenius tolerance on some inputs, while the fp16
scheme stays well inside it; above a few dozen rows the bf16 scheme's error
settles near 1%.
"""

import math

import numpy as np
import torch

from oracle import muon_oracle as O


def rnd_bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).double().numpy()


def rnd_f16(x, sigma):
    return (np.asarray(x, np.float64) * sigma).astype(np.float16).astype(np.float64) / sigma


def max_abs_on(f, hi):
    # dense sampling of |f| on [0, hi] (a model: the library solves for the stationary points)
    xs = np.linspace(0.0, hi, 20001)
    return float(np.max(np.abs(f(xs))))


def sigma_for(bound):
    return 2.0 ** (14 - math.ceil(math.log2(bound * 1.01))) if bound > 1e-30 else 1.0


def rnd_e5m2(x, bound):
    # e5m2(x * S) / S with S the power of two that puts `bound` at or below 2^13
    S = 2.0 ** (13 - math.ceil(math.log2(bound * 1.01)))
    t = torch.from_numpy(np.asarray(x * S, np.float32)).to(torch.float8_e5m2)
    return t.to(torch.float32).double().numpy() / S


def model(G, scheme, steps=5, coeffs=O.QUINTIC, eps=1e-7):
    X0 = np.asarray(G, np.float64)
    tr = X0.shape[0] > X0.shape[1]
    if tr:
        X0 = X0.T
    s = 1.0 / (math.sqrt(float(np.sum(X0 * X0))) + eps)
    a, b, c = coeffs
    hi, lo = X0, np.zeros_like(X0)
    bx = 1.0
    for it in range(steps):
        first, last = it == 0, it == steps - 1
        ba = bx * bx
        bb = max_abs_on(lambda l: b * l + c * l * l, ba)
        bx = max_abs_on(lambda x: a * x + b * x ** 3 + c * x ** 5, bx)
        A = (s * s if first else 1.0) * (hi @ hi.T)
        A = rnd_bf16(A) if scheme == "bf16" else rnd_f16(A, sigma_for(ba))
        B = b * A + c * (A @ A)
        B = rnd_bf16(B) if (scheme == "bf16" or first) else rnd_f16(B, sigma_for(bb))
        Xn = (s if first else 1.0) * (a * (hi + lo) + B @ hi)
        if last:
            out = rnd_bf16(Xn)
            return out.T if tr else out
        hi = rnd_bf16(Xn) if scheme == "bf16" else rnd_f16(Xn, sigma_for(bx))
        unit = 2.0 ** -8 if scheme == "bf16" else 2.0 ** -11
        lo = rnd_e5m2(Xn - hi, unit * bx) if it + 2 < steps else np.zeros_like(hi)


def rel(x, y):
    return float(np.linalg.norm(x - y) / np.linalg.norm(y))


def lognormal_rows(m, n, seed):
    g = torch.Generator().manual_seed(seed)
    z = torch.randn(m, n, generator=g) * torch.exp(torch.randn(m, 1, generator=g))
    return z.to(torch.bfloat16).double().numpy()


def errors(m, n, seeds, scheme):
    out = []
    for sd in seeds:
        G = lognormal_rows(m, n, sd)
        out.append(rel(model(G, scheme), O.newton_schulz(G)))
    return np.array(out)


def test_fp16_scheme_meets_the_tolerance_at_8x8_where_bf16_does_not():
    seeds = range(200)
    e16 = errors(8, 8, seeds, "fp16")
    ebf = errors(8, 8, seeds, "bf16")
    assert e16.max() < 2e-2 * 0.9, e16.max()
    assert ebf.max() > 2e-2, ebf.max()          # storing A, B, X in bf16 fails some 8 x 8 inputs
    assert e16.mean() < ebf.mean() / 3


def test_fp16_scheme_on_larger_and_rank_deficient_inputs_and_bf16_above_256_rows():
    e16 = errors(64, 192, range(4), "fp16")
    ebf = errors(64, 192, range(4), "bf16")
    assert e16.max() < 4e-3 and e16.max() < ebf.min() / 2
    # above 256 rows the library stores bf16: the error settles near 1%, well inside 2e-2
    ebig = errors(264, 776, range(2), "bf16")
    assert ebig.max() < 1.5e-2
    # rank 8 with a spectrum down to 1e-6: the low half of X keeps the null space quiet
    rng = np.random.default_rng(5)
    U, _ = np.linalg.qr(rng.standard_normal((64, 64)))
    V, _ = np.linalg.qr(rng.standard_normal((192, 64)))
    s = np.exp(np.linspace(0.0, math.log(1e-6), 64))
    s[8:] = 0.0
    G = rnd_bf16((U * s) @ V.T)
    assert rel(model(G, "fp16"), O.newton_schulz(G)) < 4e-3
