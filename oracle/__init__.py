"""fp64 CPU oracle of the Muon step (test infrastructure; see muon_oracle)."""

from .muon_oracle import (  # noqa: F401
    CUBIC,
    DEFAULT_EPS,
    DEFAULT_STEPS,
    QUINTIC,
    apply_update,
    apply_update_fp32,
    axpy_update,
    bf16_bits,
    bf16_from_bits,
    bf16_round,
    coefficient_rows,
    default_scale,
    frobenius_normalise,
    gram,
    momentum_update,
    muon_step,
    newton_schulz,
    newton_schulz_batched,
    poly,
)
