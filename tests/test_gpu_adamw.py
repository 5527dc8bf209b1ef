"""AdamW kernels against the oracle's fixed-order fp32 statement: bit for bit."""

import numpy as np
import pytest
import torch

from oracle import adamw_oracle as A
from tests._util import bits16, bits32, np32, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mk():
    return require_gpu()


def f32(x):
    return float(np.float32(x))


HP = dict(lr=f32(1e-3), beta1=f32(0.9), beta2=f32(0.95), eps=f32(1e-8), weight_decay=f32(0.1))


@pytest.mark.parametrize("numel,offset", [(1 << 20, 0), (1000003, 0), (77, 3)])
def test_adamw_bf16_bit_exact_over_steps(mk, numel, offset):
    gen = torch.Generator("cuda").manual_seed(500 + numel)
    n = numel + offset
    W = (torch.randn(n, generator=gen, device="cuda") * 0.02).to(torch.bfloat16)[offset:]
    m = torch.zeros(n, device="cuda")[offset:]
    v = torch.zeros(n, device="cuda")[offset:]
    Wr, mr, vr = np32(W), np.zeros(numel, np.float32), np.zeros(numel, np.float32)
    for t in range(1, 4):
        g = (torch.randn(n, generator=gen, device="cuda") * 1e-2).to(torch.bfloat16)[offset:]
        mk.muon_adamw_update(W, g, m, v, step=t, **HP)
        Wr, mr, vr = A.adamw_step_fp32(Wr, np32(g), mr, vr, step=t, to_bf16=True, **HP)
        assert np.array_equal(bits32(m), mr.view(np.uint32))
        assert np.array_equal(bits32(v), vr.view(np.uint32))
        assert np.array_equal(bits16(W), (Wr.view(np.uint32) >> 16).astype(np.uint16))


def test_adamw_f32_bit_exact(mk):
    gen = torch.Generator("cuda").manual_seed(601)
    W = torch.randn(65537, generator=gen, device="cuda") * 0.02
    m = torch.randn(65537, generator=gen, device="cuda") * 1e-3
    v = torch.rand(65537, generator=gen, device="cuda") * 1e-5
    g = torch.randn(65537, generator=gen, device="cuda") * 1e-2
    want = A.adamw_step_fp32(np32(W), np32(g), np32(m), np32(v), step=9, **HP)
    mk.muon_adamw_update_f32(W, g, m, v, step=9, **HP)
    for got, ref in zip((W, m, v), want):
        assert np.array_equal(bits32(got), ref.view(np.uint32))


def test_adamw_rejects_bad_arguments(mk):
    W = torch.zeros(8, dtype=torch.bfloat16, device="cuda")
    m = torch.zeros(8, device="cuda")
    with pytest.raises(mk.MuonError):
        mk.muon_adamw_update(W, W, m, m, step=0)
    with pytest.raises(mk.MuonError):
        mk.muon_adamw_update(W, W, m, m, step=1, beta1=1.0)
