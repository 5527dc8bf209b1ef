"""Helpers shared by the tests (no method arithmetic here)."""

import numpy as np
import pytest
import torch


def rel_fro(x, y):
    x = np.asarray(x, np.float64)
    y = np.asarray(y, np.float64)
    return float(np.linalg.norm(x - y) / max(np.linalg.norm(y), 1e-300))


def np32(t):
    """A torch tensor (any float dtype, any device) as a numpy float32 array (exact for bf16)."""
    return t.detach().to("cpu", torch.float32).numpy()


def bits16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bits32(t):
    return t.detach().cpu().contiguous().view(torch.int32).numpy().view(np.uint32)


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import muon_newton_schulz_expert_gb300.build as b
    import muon_newton_schulz_expert_gb300 as mk
    b.build(checked=mk.CHECKED)
    mk.lib()
    return mk
