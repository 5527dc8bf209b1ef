"""AdamW oracle (test infrastructure only; same rules as muon_oracle).

Source: "Training a 1T-Parameter MoE on EU public infrastructure with PyTorch
and TorchTitan", section "FlexShard: Muon without communication": routers and
embeddings (the parameters Muon does not take) use AdamW, which keeps two
fp32 states per parameter where Muon keeps one.  The page prints no formula;
the reading taken is AdamW with decoupled weight decay and bias correction:

  m <- b1 m + (1 - b1) g ;  v <- b2 v + (1 - b2) g^2
  W <- (1 - lr wd) W - lr * (m / (1 - b1^t)) / (sqrt(v / (1 - b2^t)) + eps)

``adamw_step`` is that definition in fp64; ``adamw_step_fp32`` states the same
update with every fp32 operation rounded separately in a fixed order (the
statement a GPU kernel can match bit for bit).  Pins: tests/test_adamw_oracle.py
(first-step and constant-gradient closed forms, zero gradient, fp32 statement
within a few ulps of fp64).
"""

from __future__ import annotations

import numpy as np

from .muon_oracle import bf16_round


def adamw_step(param, grad, exp_avg, exp_avg_sq, *, lr, beta1, beta2, eps, weight_decay, step):
    """One AdamW step in fp64; returns (param, exp_avg, exp_avg_sq)."""
    W = np.asarray(param, np.float64)
    g = np.asarray(grad, np.float64)
    m = beta1 * np.asarray(exp_avg, np.float64) + (1.0 - beta1) * g
    v = beta2 * np.asarray(exp_avg_sq, np.float64) + (1.0 - beta2) * g * g
    m_hat = m / (1.0 - beta1 ** step)
    v_hat = v / (1.0 - beta2 ** step)
    W = (1.0 - lr * weight_decay) * W - lr * m_hat / (np.sqrt(v_hat) + eps)
    return W, m, v


def adamw_constants(lr, beta1, beta2, eps, weight_decay, step):
    """The fp32 constants of the fixed-order statement, formed in fp64 and rounded once."""
    f = np.float32
    return {
        "b1": f(beta1), "c1": f(1.0 - beta1), "b2": f(beta2), "c2": f(1.0 - beta2),
        "bc2": f(1.0 - beta2 ** step), "step_size": f(lr / (1.0 - beta1 ** step)),
        "kw": f(1.0 - lr * weight_decay), "eps": f(eps),
    }


def adamw_step_fp32(param, grad, exp_avg, exp_avg_sq, *, lr, beta1, beta2, eps, weight_decay, step,
                    to_bf16=False):
    """The same step with each fp32 operation rounded separately:

    m' = (b1 m) + (c1 g);  v' = (b2 v) + (c2 (g g));
    d = sqrt(v' / bc2) + eps;  u = m' / d;  W' = (kw W) - (step_size u)
    with c1 = fp32(1 - b1), c2 = fp32(1 - b2), bc2 = fp32(1 - b2^t),
    step_size = fp32(lr / (1 - b1^t)), kw = fp32(1 - lr wd).  W' is rounded to
    bf16 when the parameter is bf16.
    """
    k = adamw_constants(lr, beta1, beta2, eps, weight_decay, step)
    f32 = np.float32
    W = np.asarray(param, f32)
    g = np.asarray(grad, f32)
    m = np.asarray(exp_avg, f32)
    v = np.asarray(exp_avg_sq, f32)
    m = np.add(np.multiply(k["b1"], m, dtype=f32), np.multiply(k["c1"], g, dtype=f32), dtype=f32)
    gg = np.multiply(g, g, dtype=f32)
    v = np.add(np.multiply(k["b2"], v, dtype=f32), np.multiply(k["c2"], gg, dtype=f32), dtype=f32)
    d = np.add(np.sqrt(np.divide(v, k["bc2"], dtype=f32), dtype=f32), k["eps"], dtype=f32)
    u = np.divide(m, d, dtype=f32)
    W = np.subtract(np.multiply(k["kw"], W, dtype=f32), np.multiply(k["step_size"], u, dtype=f32), dtype=f32)
    return (bf16_round(W) if to_bf16 else W), m, v
