"""The algorithmic work bench.py divides by measured time (CPU).

Per 1792 x 6144 matrix and quintic iteration, with the symmetric products
counted once per computed triangle: X X^T takes m^2 n multiply-adds' worth of
flops (half of the dense 2 m^2 n), A A takes m^3 (half of 2 m^3), and aX + BX
takes the dense 2 m^2 n.  Five iterations give 3.247e11 flops per matrix and
4.52e11 dense-equivalent; the 96-matrix workload is 3.117e13.  The elementwise
kernels' bytes are the bytes each element moves once.
"""

import pytest

import bench


def test_flops_per_matrix():
    m, n = bench.M_EXP, bench.N_EXP
    assert (m, n) == (1792, 6144)
    dense = {"syrk": 2 * m * n * m, "poly": 2 * m * m * m, "axpy": 2 * m * m * n}   # 2 x multiply-adds of each GEMM
    assert bench.FLOPS_SYRK * 2 == dense["syrk"]
    assert bench.FLOPS_POLY * 2 == dense["poly"]
    assert bench.FLOPS_AXPY == dense["axpy"]
    assert bench.FLOPS_NS == 5 * (bench.FLOPS_SYRK + bench.FLOPS_POLY + bench.FLOPS_AXPY)
    assert bench.FLOPS_NS == pytest.approx(3.247e11, rel=1e-3)
    assert bench.FLOPS_NS_DENSE == 5 * sum(dense.values())
    assert bench.FLOPS_NS_DENSE == pytest.approx(4.52e11, rel=1e-3)
    assert 96 * bench.FLOPS_NS == pytest.approx(3.117e13, rel=1e-3)
    # the update-fused last iteration does the work of one aX + BX
    assert bench.KERNEL_FLOPS["ns_axpy_apply_tc"] == bench.FLOPS_AXPY


def test_elementwise_bytes_per_element():
    bf16, f32 = 2, 4
    assert bench.KERNEL_BYTES["momentum_bf16"] == bf16 + f32 + f32 + bf16          # g in, buf in/out, u out
    assert bench.KERNEL_BYTES["momentum_norm_bf16"] == bench.KERNEL_BYTES["momentum_bf16"]  # squares in registers
    assert bench.KERNEL_BYTES["apply_bf16"] == bf16 + bf16 + bf16                  # W in/out, O in
    assert bench.KERNEL_BYTES["norm_partial"] == bf16                              # X read once
    assert bench.PER_MATRIX_ELEMS == 1792 * 6144
