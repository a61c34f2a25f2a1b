"""Seeded random shapes for the FSDP unit: the forward with the gather fused into the GEMM's
loads (shard rows a multiple of 128) or through a scratch buffer (any shard rows), the
backward on both its in-place and its transposed path, and the MLP unit; each checked
against the oracle by the same bounds as the fixed-shape tests."""
import numpy as np
import pytest
import torch

import test_fsdp_parity as F  # the fixed-shape checks, called with random shapes
from test_fsdp_parity import z  # noqa: F401  (fixture)

pytestmark = pytest.mark.gpu


def forward_case(i):
    rng = np.random.default_rng(2000 + i)
    n = int(rng.choice([1, 2, 3, 4, 8]))
    k = 8 * int(rng.integers(1, 130))
    m = int(rng.integers(1, 700))
    if i % 2 == 0:  # fused gather: shard rows a multiple of 128
        return "fused", m, n * 128 * int(rng.integers(1, 6)), k, n
    return "scratch", m, n * int(rng.integers(1, 300)), k, n


def backward_case(i):
    rng = np.random.default_rng(3000 + i)
    n = int(rng.choice([1, 2, 3, 4, 5, 8, 16]))
    if i % 2 == 0:  # in place: R / N, K and M multiples of 64
        return n, n * 64 * int(rng.integers(1, 6)), 64 * int(rng.integers(1, 9)), 64 * int(rng.integers(1, 5))
    rows = n * 8 * int(rng.integers(1, 40))
    k = 8 * int(rng.integers(1, 70))
    m = int(rng.integers(1, 300))
    while (n * m) % 8:  # the GEMMs' 16-byte rows
        m += 1
    return n, rows, k, m


@pytest.mark.parametrize("i", range(10))
def test_random_forward(z, i):
    path, m, rows, k, n = forward_case(i)
    if path == "fused":
        F.test_gemm_fused_gather_vs_oracle(z, m, rows, k, n)
    else:
        F.test_gemm_scratch_gather_vs_oracle(z, m, rows, k, n)


@pytest.mark.parametrize("i", range(10))
def test_random_backward(z, i):
    n, rows, k, m = backward_case(i)
    F.test_backward_vs_oracle(z, n, rows, k, m)
    if rows * k <= 1 << 20 and n * m * max(rows, k) <= 1 << 22:
        F.test_backward_integer_values_exact(z, n, rows, k, m)


@pytest.mark.parametrize("i", range(4))
def test_random_mlp_unit(z, i):
    rng = np.random.default_rng(4000 + i)
    n = int(rng.choice([1, 2, 4]))
    scratch = bool(i % 2)
    d = n * 128 * int(rng.integers(1, 5)) if not scratch else n * 8 * int(rng.integers(1, 64))
    f = n * 128 * int(rng.integers(1, 4))
    m = int(rng.integers(1, 400))
    F.test_mlp_unit_vs_oracle(z, n, d, f, m, scratch)


@pytest.mark.parametrize("i", range(6))
def test_random_backward_both_kernels_bit_identical(z, i):
    """Random backward shapes on the one-CTA kernel (zero_set_gemm_kernel(1)) against the
    default CTA-pair kernel, on the in-place path's MN-major GEMMs and the transposed path's
    K-major ones: the same bits."""
    n, rows, k, m = backward_case(100 + i)
    outs = []
    try:
        for kernel in (0, 1):
            z.zero_set_gemm_kernel(kernel)
            _, _, _, dX, dW = F.run_backward(z, n, rows, k, m, key=rows + 7 * i)
            outs.append(([x.view(torch.int32).clone() for x in dX], dW.view(torch.int32).clone()))
    finally:
        z.zero_set_gemm_kernel(0)
    for q in range(n):
        assert torch.equal(outs[0][0][q], outs[1][0][q]), f"dX of rank {q}: n={n} rows={rows} k={k} m={m}"
    assert torch.equal(outs[0][1], outs[1][1]), f"dW: n={n} rows={rows} k={k} m={m}"


def zero3_case(i):
    """A random stack of linear units for fsdp_zero3_step: N, unit count, chained shapes
    (rows_out / N and k_in multiples of 64), tokens per rank (N M a multiple of 8, ragged K
    blocks in dW), flags."""
    rng = np.random.default_rng(5000 + i)
    n = int(rng.choice([1, 2, 3, 4, 8]))
    flags = int(rng.choice([0, 1, 2, 3, 4, 6, 7]))
    fused_rows = n * 128 * int(rng.integers(1, 4))  # shards that tile the fused gather
    shapes, k = [], 64 * int(rng.integers(1, 9))
    for _ in range(int(rng.integers(1, 4))):
        r = fused_rows if not flags & 1 or rng.random() < 0.5 else 64 * n * int(rng.integers(1, 5))
        shapes.append((r, k))
        k = r
    m = int(rng.integers(8, 200))
    while (n * m) % 8:
        m += 1
    return n, shapes, m, flags


@pytest.mark.parametrize("i", range(6))
def test_random_zero3_step(z, i):
    import test_fsdp_zero3 as Z3
    n, shapes, m, flags = zero3_case(i)
    units = Z3.make_units(z, n, shapes, m, key=50 + i)
    for t in (1, 2):
        before = Z3.snapshot(units)
        y, dx = Z3.run_step(z, units, m, t, flags, prefetch=bool(flags & 6))
        Z3.check_step(z, n, m, before, units, y, dx, t)


@pytest.mark.parametrize("i", range(4))
def test_random_zero3_mlp_step(z, i):
    import test_fsdp_zero3_mlp as ZM
    rng = np.random.default_rng(6000 + i)
    n = int(rng.choice([1, 2, 4]))
    d = n * 128 * int(rng.integers(1, 4))
    f = n * 128 * int(rng.integers(1, 4))
    m = int(rng.integers(8, 120))
    while (n * m) % 8:
        m += 1
    units = ZM.make_units(z, n, d, f, int(rng.integers(1, 3)), m, key=60 + i)
    for t in (1, 2):
        before = ZM.snapshot(units)
        y, dx = ZM.run_step(z, units, m, t)
        ZM.check_step(n, m, before, units, y, dx, t)
