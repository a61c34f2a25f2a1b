"""GPU parity of the FSDP GEMMs where their persistent tile walk runs in several bands.

Both GEMM kernels walk output tiles in bands of rows: 12 pairs of 256 rows on the
CTA-pair kernel, 24 blocks of 128 rows on the one-CTA kernel, i.e. 3,072 output rows per
band. Shapes below that height degenerate to whole columns, so these cases use M above
it, with a ragged last band and several column tiles, and compare EVERY output with the
oracle:
  - the forward (fused gather on both kernels, and the scratch gather) against the
    oracle's float64 product under the fp32 summation bound
        |Y - Y_exact| <= (K + 1) 2^-23 sum_k |a_k w_k|;
  - the backward's all-rank row-split dX (N M rows) and its dW (R rows), each above one
    band, against the oracle's dX_q = dY_q W and (1/N) sum_q dY_q^T X_q under their bounds;
  - the full Mistral-7B MLP shapes (8192 tokens; W_up 14336 x 4096 and W_down 4096 x 14336
    in 8 row shards) with every input a small integer in {-2..2}: every product and
    partial sum is an integer below 2^24, so any fp32 summation order is exact and every
    one of the 117,440,512 outputs must equal the oracle's product exactly.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle.zero_oracle as O
import synth
from _util import bits16, f32, from_bits16

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def z():
    import __graft_entry__ as g
    g.build()
    import fsdp_sharded_optimizer_zero_gb300 as z
    yield z
    z.zero_set_gemm_kernel(0)


@pytest.fixture(autouse=True)
def _default_gemm_kernel(z):
    z.zero_set_gemm_kernel(0)
    yield
    z.zero_set_gemm_kernel(0)


def check_forward(y_gpu, a_bits, shard_bits, what):
    y64, _, _ = O.fsdp_linear_forward(a_bits, shard_bits)
    a64 = np.abs(O.bf16_to_f32(a_bits).astype(np.float64))
    w64 = np.abs(O.bf16_to_f32(O.gather_rows(shard_bits)).astype(np.float64))
    bound = (a64.shape[1] + 1) * 2.0 ** -23 * (a64 @ w64.T)
    err = np.abs(y_gpu.astype(np.float64) - y64)
    bad = err > bound
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outputs outside the bound, first at " \
                          f"{np.unravel_index(np.argmax(bad), bad.shape)}"


# M = 4352: 17 pair rows (bands 12 + 5) / 34 one-CTA row blocks (24 + 10); M = 4429 adds a
# ragged row tile; R = 1024 / 1280 gives 4 / 5 column tiles of 256
@pytest.mark.parametrize("kernel", [0, 1])
@pytest.mark.parametrize("m,rows,k,n", [(4352, 1024, 136, 4), (4429, 1280, 200, 5), (6400, 2048, 64, 8)])
def test_forward_banded_walk_every_output(z, kernel, m, rows, k, n):
    if kernel == 1 and (rows // n) % 256:
        pytest.skip("the one-CTA kernel's fused gather needs 256-row shards")
    z.zero_set_gemm_kernel(kernel)
    shards = synth.weight_shards(rows, k, n, device=DEV, seed_key=m + kernel)
    A = synth.activations(m, k, device=DEV, seed_key=rows)
    Y = torch.full((m, rows), float("nan"), device=DEV)
    z.fsdp_unit_forward(shards, A, Y)
    z.zero_device_status()
    check_forward(f32(Y), bits16(A), [bits16(s) for s in shards], f"kernel {kernel} m={m} rows={rows} k={k}")


@pytest.mark.parametrize("m,rows,k,n", [(4352, 1000, 136, 5), (3333, 768, 72, 3)])
def test_forward_banded_walk_scratch_gather(z, m, rows, k, n):
    shards = synth.weight_shards(rows, k, n, device=DEV, seed_key=rows)
    A = synth.activations(m, k, device=DEV, seed_key=m)
    Y = torch.full((m, rows), float("nan"), device=DEV)
    scratch = torch.empty(rows, k, dtype=torch.bfloat16, device=DEV)
    z.fsdp_unit_forward(shards, A, Y, scratch_w=scratch)
    z.zero_device_status()
    check_forward(f32(Y), bits16(A), [bits16(s) for s in shards], f"scratch m={m} rows={rows}")


def run_backward(z, n, rows, k, m, key, ints):
    if ints:
        rng = np.random.default_rng(key)
        mk = lambda shape: from_bits16(O.f32_to_bf16(rng.integers(-2, 3, shape).astype(np.float32)), DEV)
        shards = [mk((rows // n, k)) for _ in range(n)]
        A = [mk((m, k)) for _ in range(n)]
        dY = [mk((m, rows)) for _ in range(n)]
    else:
        shards = synth.weight_shards(rows, k, n, device=DEV, seed_key=key)
        A = [synth.activations(m, k, device=DEV, seed_key=100 * key + q) for q in range(n)]
        dY = [synth.upstream_grad(m, rows, device=DEV, seed_key=100 * key + q) for q in range(n)]
    dX = [torch.full((m, k), float("nan"), device=DEV) for _ in range(n)]
    dW = torch.full((rows, k), float("nan"), device=DEV)
    ws = torch.empty(z.fsdp_unit_backward_workspace(n, rows, k, m), dtype=torch.uint8, device=DEV)
    z.fsdp_unit_backward(shards, A, dY, dX, dW, ws)
    z.zero_device_status()
    return shards, A, dY, dX, dW


# dX over all ranks is one row-split GEMM of N M = 4096 rows (32 blocks of 128: bands 24 + 8);
# dW has R = 3584 rows (28 blocks: 24 + 4); every operand in place (R/N, M, K multiples of
# 64), on the CTA-pair kernel (the default) and on the one-CTA kernel.
# (4, 3200, 200, 896): K not a multiple of 64, so the transposed path's K-major GEMMs run
# the same walk.
@pytest.mark.parametrize("kernel", [0, 1])
@pytest.mark.parametrize("n,rows,k,m", [(8, 3584, 128, 512), (4, 3200, 200, 896)])
def test_backward_banded_walk_every_output(z, kernel, n, rows, k, m):
    z.zero_set_gemm_kernel(kernel)
    shards, A, dY, dX, dW = run_backward(z, n, rows, k, m, key=rows + kernel, ints=False)
    sb = [bits16(s) for s in shards]
    w_abs = np.abs(O.bf16_to_f32(O.gather_rows(sb)).astype(np.float64))
    exact_dw = np.zeros((rows, k))
    bound_dw = np.zeros((rows, k))
    for q in range(n):
        dx64, dw64 = O.fsdp_linear_backward(bits16(A[q]), sb, bits16(dY[q]), n)
        dy_abs = np.abs(O.bf16_to_f32(bits16(dY[q])).astype(np.float64))
        a_abs = np.abs(O.bf16_to_f32(bits16(A[q])).astype(np.float64))
        bound_dx = (rows + 1) * 2.0 ** -23 * (dy_abs @ w_abs)
        bad = np.abs(f32(dX[q]) - dx64) > bound_dx
        assert not bad.any(), f"dX of rank {q}: {bad.sum()} entries outside the bound"
        exact_dw += dw64
        bound_dw += dy_abs.T @ a_abs
    exact_dw /= n
    bound = (n * m + 1) * 2.0 ** -23 * bound_dw / n + 2.0 ** -24 * np.abs(exact_dw)
    bad = np.abs(f32(dW) - exact_dw) > bound
    assert not bad.any(), f"dW: {bad.sum()} entries outside the bound"


@pytest.mark.parametrize("n,rows,k,m", [(8, 3584, 128, 512)])
def test_backward_banded_walk_integers_exact(z, n, rows, k, m):
    shards, A, dY, dX, dW = run_backward(z, n, rows, k, m, key=11, ints=True)
    w = O.bf16_to_f32(O.gather_rows([bits16(s) for s in shards])).astype(np.float64)
    acc = np.zeros((rows, k))
    for q in range(n):
        a = O.bf16_to_f32(bits16(A[q])).astype(np.float64)
        dy = O.bf16_to_f32(bits16(dY[q])).astype(np.float64)
        assert np.array_equal(f32(dX[q]).astype(np.float64), dy @ w), f"dX of rank {q}"
        acc += dy.T @ a
    assert np.array_equal(f32(dW), acc.astype(np.float32) * np.float32(1.0 / n)), "dW"


def small_ints(rng, shape):
    return O.f32_to_bf16(rng.integers(-2, 3, shape).astype(np.float32))


@pytest.mark.parametrize("which,rows,k", [("up", 14336, 4096), ("down", 4096, 14336)])
def test_mistral_shape_integers_exact_everywhere(z, which, rows, k):
    """Every output of the full-size Mistral GEMM, fused gather of 8 row shards, in the
    launch configuration the bench times (CTA-pair kernel, fp32 output)."""
    m, n = 8192, 8
    rng = np.random.default_rng(rows)
    a_bits = small_ints(rng, (m, k))
    w_bits = small_ints(rng, (rows, k))
    rs = rows // n
    shard_bits = [w_bits[r * rs:(r + 1) * rs] for r in range(n)]
    A = from_bits16(a_bits, DEV)
    shards = [from_bits16(s, DEV) for s in shard_bits]
    Y = torch.full((m, rows), float("nan"), device=DEV)
    z.fsdp_unit_forward(shards, A, Y)
    z.zero_device_status()
    y = f32(Y)
    del Y, A, shards
    y64, _, _ = O.fsdp_linear_forward(a_bits, shard_bits)
    assert np.abs(y64).max() < 2 ** 24
    bad = y != y64.astype(np.float32)
    assert not bad.any(), f"W_{which}: {bad.sum()} of {bad.size} outputs differ from the integer product, " \
                          f"first at {np.unravel_index(np.argmax(bad), bad.shape)}"
