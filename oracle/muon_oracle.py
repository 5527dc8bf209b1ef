"""Plain fp64 CPU oracle for the Muon optimizer step on whole weight matrices.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or run
this module.  The CUDA library never calls it and shares no code with it: the
two sides agree only through the seeded inputs of ``workloads.py``.

Source of the method: "Training a 1T-Parameter MoE on EU public infrastructure
with PyTorch and TorchTitan" (PyTorch blog; Chinese translation), section
"FlexShard: Muon without communication" and the model-configuration table.
That section fixes: Muon on every weight matrix but routers and embeddings,
one fp32 state per parameter, and an update orthogonalised by a few
Newton-Schulz iterations acting on the whole matrix, each rank owning whole
expert matrices so no communication is needed.  It does not print the
iteration, its coefficients, the momentum form, eps, the learning rate, the
weight decay or the shape scale; the readings taken here are:

* momentum (SGD/Nesterov form, fp32, each operation rounded to fp32):
  buf <- mu*buf + g ; u <- g + mu*buf (new buf) when Nesterov, else u <- buf.
* Newton-Schulz: orient to rows <= cols (X = G^T when rows > cols),
  X <- G / (||G||_F + eps), then ``steps`` times
  A = X X^T ; B = b A + c A A ; X = a X + B X ; then orient back.
  Quintic coefficients (a, b, c) = (3.4445, -4.7750, 2.0315), 5 steps.
* update with decoupled weight decay:
  W <- (1 - lr*wd) W - lr*scale*O, scale = sqrt(max(1, rows/cols)) by default.

Arithmetic: fp64 throughout for the matrix work (numpy matmul is the only
library step); the momentum is fp32 by definition (one fp32 state per
parameter) and bf16 conversions are round-to-nearest-even.

Parity pins (tests/test_oracle.py): SVD closed form U p^k(S) V^T on tiny
inputs, constructed spectra U diag(s) V^T, the cubic converging to the polar
factor, orthogonal equivariance, scale invariance, transpose symmetry,
diagonal inputs against exact rational arithmetic, the zero matrix, planted
mistakes that the pins must catch, exact-arithmetic momentum sequences, the
EMA/SGD proportionality, hand-derived bf16 rounding cases and torch's own
bf16 conversion.  No function here is "parity unpinned".
"""

from __future__ import annotations

import math

import numpy as np

QUINTIC = (3.4445, -4.7750, 2.0315)
CUBIC = (1.5, -0.5, 0.0)
DEFAULT_STEPS = 5
DEFAULT_EPS = 1e-7


# --------------------------------------------------------------------------
# bf16 (round to nearest, ties to even) on float32 bit patterns
# --------------------------------------------------------------------------
def bf16_round(x) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even).

    bfloat16 keeps the sign, the 8 exponent bits and the top 7 fraction bits
    of an IEEE binary32 value.  Rounding adds 0x7FFF plus the lowest kept bit
    to the 32-bit pattern before truncating the low 16 bits; a carry moves into
    the exponent (and to infinity past the largest finite bf16).  NaNs stay
    NaN (quiet).  Returns float32 values that are exactly bf16-representable.
    """
    x32 = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    bits = x32.view(np.uint32).astype(np.uint64)
    keep_lsb = (bits >> np.uint64(16)) & np.uint64(1)
    rounded = ((bits + np.uint64(0x7FFF) + keep_lsb) >> np.uint64(16)) << np.uint64(16)
    out = rounded.astype(np.uint32)
    nan = np.isnan(x32)
    if nan.any():
        out[nan] = (bits[nan].astype(np.uint32) | np.uint32(0x00400000)) & np.uint32(0xFFFF0000)
    return out.view(np.float32)


def bf16_bits(x) -> np.ndarray:
    """The 16-bit bfloat16 patterns of ``bf16_round(x)``."""
    return (bf16_round(x).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def bf16_from_bits(bits) -> np.ndarray:
    """float32 values of 16-bit bfloat16 patterns (exact widening)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


# --------------------------------------------------------------------------
# momentum: the single fp32 state per parameter
# --------------------------------------------------------------------------
def momentum_update(grad, buf, mu: float, nesterov: bool = True):
    """One fp32 momentum step; returns ``(new_buf, u)``.

    FlexShard section: Muon keeps one fp32 state per parameter.  SGD form with
    every multiply and add rounded to fp32 separately:
    buf' = fp32(fp32(mu*buf) + g);  u = fp32(g + fp32(mu*buf')) if Nesterov,
    else u = buf'.  ``grad`` is widened exactly to fp32 first.
    """
    g = np.asarray(grad, dtype=np.float32)
    b = np.asarray(buf, dtype=np.float32)
    mu32 = np.float32(mu)
    new_buf = np.add(np.multiply(mu32, b, dtype=np.float32), g, dtype=np.float32)
    if nesterov:
        u = np.add(g, np.multiply(mu32, new_buf, dtype=np.float32), dtype=np.float32)
    else:
        u = new_buf.copy()
    return new_buf, u


# --------------------------------------------------------------------------
# Newton-Schulz, split into the steps named by the method so that each one can
# be read against its definition (and replaced by a planted mistake in tests)
# --------------------------------------------------------------------------
def frobenius_normalise(X: np.ndarray, eps: float) -> np.ndarray:
    """X / (||X||_F + eps) with ||X||_F = sqrt(sum of squares), fp64."""
    X = np.asarray(X, dtype=np.float64)
    return X / (math.sqrt(float(np.sum(X * X))) + eps)


def gram(X: np.ndarray) -> np.ndarray:
    """A = X X^T (m x m for an m x n X)."""
    return X @ X.T


def poly(A: np.ndarray, b: float, c: float) -> np.ndarray:
    """B = b A + c A A."""
    return b * A + c * (A @ A)


def axpy_update(X: np.ndarray, B: np.ndarray, a: float) -> np.ndarray:
    """X' = a X + B X."""
    return a * X + B @ X


def coefficient_rows(steps: int, coeffs):
    """The (a, b, c) of each step: one triple for every step, or one row per step."""
    arr = np.asarray(coeffs, dtype=np.float64)
    if arr.shape == (3,):
        return [tuple(arr)] * int(steps)
    if arr.shape != (int(steps), 3):
        raise ValueError("coeffs must be (a, b, c) or one (a, b, c) row per step")
    return [tuple(r) for r in arr]


def newton_schulz(G, steps: int = DEFAULT_STEPS, coeffs=QUINTIC, eps: float = DEFAULT_EPS) -> np.ndarray:
    """Orthogonalise one matrix G (rows x cols); returns fp64 in G's layout.

    FlexShard section: a few Newton-Schulz iterations act on the whole matrix
    (each rank owns complete expert matrices).  Orientation: work on G^T when
    rows > cols, so that A = X X^T is the smaller Gram matrix.  ``coeffs`` is
    one (a, b, c) for every step or a schedule of one row per step.
    """
    G = np.asarray(G, dtype=np.float64)
    if G.ndim != 2:
        raise ValueError("newton_schulz takes one 2-D matrix")
    rows = coefficient_rows(steps, coeffs)
    transposed = G.shape[0] > G.shape[1]
    X = G.T if transposed else G
    X = frobenius_normalise(X, eps)
    for a, b, c in rows:
        A = gram(X)
        B = poly(A, b, c)
        X = axpy_update(X, B, a)
    return X.T if transposed else X


def newton_schulz_batched(G, steps: int = DEFAULT_STEPS, coeffs=QUINTIC, eps: float = DEFAULT_EPS) -> np.ndarray:
    """``newton_schulz`` on each matrix of a (batch, rows, cols) stack."""
    G = np.asarray(G)
    return np.stack([newton_schulz(G[i], steps, coeffs, eps) for i in range(G.shape[0])]) \
        if G.shape[0] else np.zeros(G.shape, dtype=np.float64)


# --------------------------------------------------------------------------
# parameter update
# --------------------------------------------------------------------------
def default_scale(rows: int, cols: int) -> float:
    """Shape scale sqrt(max(1, rows/cols)) on the stored shape."""
    return math.sqrt(max(1.0, rows / cols))


def apply_update(param, update, lr: float, weight_decay: float, scale: float) -> np.ndarray:
    """W' = (1 - lr*wd) W - lr*scale*O in fp64 (decoupled weight decay)."""
    W = np.asarray(param, dtype=np.float64)
    O = np.asarray(update, dtype=np.float64)
    return (1.0 - lr * weight_decay) * W - lr * scale * O


def apply_update_fp32(param, update, lr: float, weight_decay: float, scale: float, to_bf16: bool = True):
    """The same update as ``apply_update`` written in fp32 with a fixed order.

    The two constants are formed in fp64 and rounded once to fp32:
    k_w = fp32(1 - lr*wd), k_o = fp32(-lr*scale).  Then
    W' = fp32(fp32(k_w*W) + fp32(k_o*O)), rounded to bf16 (RNE) when the
    parameter is bf16.  This is the exact-rounding statement of the update
    that a bf16 parameter can be compared against bit for bit; it differs from
    the fp64 form by at most a few fp32 ulps before the final rounding.
    """
    kw = np.float32(1.0 - lr * weight_decay)
    ko = np.float32(-lr * scale)
    W = np.asarray(param, dtype=np.float32)
    O = np.asarray(update, dtype=np.float32)
    out = np.add(np.multiply(kw, W, dtype=np.float32), np.multiply(ko, O, dtype=np.float32), dtype=np.float32)
    return bf16_round(out) if to_bf16 else out


# --------------------------------------------------------------------------
# the whole step on a stack of same-shape matrices
# --------------------------------------------------------------------------
def muon_step(param, grad, buf, *, mu: float = 0.95, nesterov: bool = True, steps: int = DEFAULT_STEPS,
              coeffs=QUINTIC, eps: float = DEFAULT_EPS, lr: float = 0.02, weight_decay: float = 0.1,
              scale: float | None = None, bf16: bool = True):
    """Momentum -> (bf16 u) -> Newton-Schulz -> update, per matrix of a stack.

    ``param``/``grad``/``buf`` are (batch, rows, cols).  With ``bf16`` the
    Newton-Schulz input is u rounded to bf16 (the NS input of a bf16 path);
    otherwise u stays fp32.  Returns a dict with the new momentum (fp32), u,
    the orthogonalised update O (fp64) and the new parameter (fp64).
    """
    grad = np.asarray(grad, dtype=np.float32)
    new_buf, u = momentum_update(grad, buf, mu, nesterov)
    ns_in = bf16_round(u) if bf16 else u
    O = newton_schulz_batched(ns_in, steps, coeffs, eps)
    rows, cols = grad.shape[-2], grad.shape[-1]
    s = default_scale(rows, cols) if scale is None or scale <= 0 else float(scale)
    W = apply_update(param, O, lr, weight_decay, s)
    return {"buf": new_buf, "u": ns_in, "O": O, "param": W, "scale": s}
