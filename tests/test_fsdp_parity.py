"""GPU parity of the FSDP unit (row-shard gather + tcgen05 GEMM) against the CPU oracle.

The gather is a bit copy: compared bit for bit. The GEMM sums exact bf16 x bf16 products
in fp32 in an order the tensor cores choose, so it is compared with the oracle's float64
result under the rounding bound of any fp32 summation order:
    |Y - Y_exact| <= (K + 1) * 2^-23 * sum_k |a_k w_k|
(first-order bound of recursive summation with unit roundoff 2^-23, which also covers
round-toward-zero accumulation). The bf16 output must be the round-to-nearest-even of the
kernel's own fp32 output, bit for bit. The fused-gather path and the scratch-gather path
load identical tiles, so their outputs must agree bit for bit.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle.zero_oracle as O
import synth
from _util import assert_bf16_identical, bits16, f32

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


def gemm_bound(a64, w64, K):
    return (K + 1) * 2.0 ** -23 * (np.abs(a64) @ np.abs(w64).T)


def check_gemm(y_gpu, a_bits, shards_bits, what):
    y64, _, _ = O.fsdp_linear_forward(a_bits, shards_bits)
    a64 = O.bf16_to_f32(a_bits).astype(np.float64)
    w64 = O.bf16_to_f32(O.gather_rows(shards_bits)).astype(np.float64)
    bound = gemm_bound(a64, w64, a64.shape[1])
    err = np.abs(y_gpu.astype(np.float64) - y64)
    bad = err > bound + 1e-30
    assert not bad.any(), f"{what}: {bad.sum()} outputs outside the bound; worst err {err.max()} at {np.unravel_index(err.argmax(), err.shape)}"


@pytest.mark.parametrize("rows,k,n", [(2048, 1024, 8), (77 * 8, 520, 8), (999, 40, 3), (64, 8, 64), (5, 3, 5)])
def test_gather_rows_bit_exact(z, rows, k, n):
    shards = synth.weight_shards(rows, k, n, device=DEV)
    full = torch.empty(rows, k, dtype=torch.bfloat16, device=DEV)
    z.fsdp_gather_rows(shards, full)
    z.zero_device_status()
    assert_bf16_identical(bits16(full), O.gather_rows([bits16(s) for s in shards]), "gather")


def test_gather_rows_misaligned_scalar_path(z):
    rows, k, n = 12, 7, 4
    base = torch.zeros(rows * k + 1, dtype=torch.bfloat16, device=DEV)
    full = base[1:].view(rows, k)
    shards = synth.weight_shards(rows, k, n, device=DEV)
    z.fsdp_gather_rows(shards, full)
    z.zero_device_status()
    assert_bf16_identical(bits16(full), O.gather_rows([bits16(s) for s in shards]), "gather misaligned")


@pytest.mark.parametrize("m,rows,k,n", [(128, 256, 64, 1), (256, 2048, 512, 8), (200, 2048, 520, 8),
                                        (384, 512, 1024, 2), (1, 256, 8, 1), (130, 4096, 136, 16),
                                        # shard rows a multiple of 128 but not of 256: the CTA pair's halves
                                        (300, 384, 136, 3), (257, 1152, 72, 9), (1, 128, 8, 1), (513, 640, 200, 5)])
def test_gemm_fused_gather_vs_oracle(z, m, rows, k, n):
    shards = synth.weight_shards(rows, k, n, device=DEV, seed_key=m)
    A = synth.activations(m, k, device=DEV, seed_key=k)
    Y = torch.full((m, rows), float("nan"), device=DEV)
    Yb = torch.zeros(m, rows, dtype=torch.bfloat16, device=DEV)
    z.fsdp_unit_forward(shards, A, Y, Y_bf16=Yb)
    z.zero_device_status()
    y = f32(Y)
    check_gemm(y, bits16(A), [bits16(s) for s in shards], f"fused m={m} rows={rows} k={k} n={n}")
    assert_bf16_identical(bits16(Yb), O.f32_to_bf16(y), "bf16 output = RNE(fp32 output)")


@pytest.mark.parametrize("m,rows,k,n", [(300, 1024, 264, 8), (129, 300, 72, 3), (256, 2048, 512, 8)])
def test_gemm_scratch_gather_vs_oracle(z, m, rows, k, n):
    shards = synth.weight_shards(rows, k, n, device=DEV, seed_key=rows)
    A = synth.activations(m, k, device=DEV, seed_key=m)
    Y = torch.full((m, rows), float("nan"), device=DEV)
    scratch = torch.empty(rows, k, dtype=torch.bfloat16, device=DEV)
    z.fsdp_unit_forward(shards, A, Y, scratch_w=scratch)
    z.zero_device_status()
    check_gemm(f32(Y), bits16(A), [bits16(s) for s in shards], f"scratch m={m} rows={rows} k={k}")
    assert_bf16_identical(bits16(scratch), O.gather_rows([bits16(s) for s in shards]), "scratch holds gathered W")
    if (rows // n) % 128 == 0:
        Y2 = torch.empty_like(Y)
        z.fsdp_unit_forward(shards, A, Y2)
        z.zero_device_status()
        assert torch.equal(Y.view(torch.int32), Y2.view(torch.int32)), "fused and scratch gathers disagree"


@pytest.mark.parametrize("m,rows,k,n,scratch", [(300, 2048, 264, 8, False), (129, 512, 72, 2, False),
                                                 (200, 1000, 136, 5, True), (1, 256, 8, 1, False)])
def test_gemm_bf16_only_output_equals_rounded_fp32(z, m, rows, k, n, scratch):
    """With Y = NULL the kernel writes only bf16 Y (TMA stores of 64-column chunks); it must
    equal, bit for bit, the round-to-nearest-even of the fp32 result of the same GEMM."""
    shards = synth.weight_shards(rows, k, n, device=DEV, seed_key=rows + k)
    A = synth.activations(m, k, device=DEV, seed_key=m)
    sw = (lambda: torch.empty(rows, k, dtype=torch.bfloat16, device=DEV)) if scratch else (lambda: None)
    Y = torch.empty(m, rows, device=DEV)
    z.fsdp_unit_forward(shards, A, Y, scratch_w=sw())
    Yb = torch.full((m, rows), float("nan"), dtype=torch.bfloat16, device=DEV)
    z.fsdp_unit_forward(shards, A, None, Y_bf16=Yb, scratch_w=sw())
    z.zero_device_status()
    assert_bf16_identical(bits16(Yb), O.f32_to_bf16(f32(Y)), "bf16-only output")


def test_gemm_integer_values_exact(z):
    """Small integers: every product and partial sum is exact in fp32, so any summation
    order gives the exact result; checks orientation (Y = A W^T) and shard order."""
    m, rows, k, n = 128, 512, 128, 2
    rng = np.random.default_rng(0)
    a = rng.integers(-3, 4, (m, k)).astype(np.float32)
    w = rng.integers(-3, 4, (rows, k)).astype(np.float32)
    A = torch.from_numpy(O.f32_to_bf16(a).view(np.int16)).view(torch.bfloat16).to(DEV)
    wb = O.f32_to_bf16(w)
    shards = [torch.from_numpy(wb[r * 256:(r + 1) * 256].view(np.int16).copy()).view(torch.bfloat16).to(DEV)
              for r in range(n)]
    Y = torch.empty(m, rows, device=DEV)
    z.fsdp_unit_forward(shards, A, Y)
    z.zero_device_status()
    assert np.array_equal(f32(Y), a @ w.T)


@pytest.mark.parametrize("shard_rows,kernel,ok", [(192, 0, False), (192, 1, False), (128, 0, True), (128, 1, False),
                                                   (256, 1, True)])
def test_gemm_needs_scratch_when_shards_do_not_tile(z, shard_rows, kernel, ok):
    """Without a scratch buffer the fused gather needs each B tile to lie in one shard: shard
    rows a multiple of 128 for the CTA-pair kernel (128-row halves), of 256 for the one-CTA
    kernel (whole 256-row tiles); otherwise the call is ZERO_ERR_UNSUPPORTED (-4)."""
    z.zero_set_gemm_kernel(kernel)
    shards = synth.weight_shards(8 * shard_rows, 64, 8, device=DEV)
    A = synth.activations(128, 64, device=DEV)
    Y = torch.empty(128, 8 * shard_rows, device=DEV)
    if ok:
        z.fsdp_unit_forward(shards, A, Y)
        z.zero_device_status()
        check_gemm(f32(Y), bits16(A), [bits16(s) for s in shards], f"shard rows {shard_rows}")
        return
    with pytest.raises(z.ZeroError) as e:
        z.fsdp_unit_forward(shards, A, Y)
    assert e.value.code == -4


@pytest.mark.parametrize("m,rows,k,n,mode", [(128, 256, 64, 1, "fused"), (300, 2048, 520, 8, "fused"),
                                             (1, 256, 8, 1, "fused"), (257, 512, 136, 2, "fused"),
                                             (640, 4096, 1024, 16, "fused"), (300, 1024, 264, 8, "scratch"),
                                             (129, 300, 72, 3, "scratch"), (200, 2048, 72, 4, "bf16"),
                                             (130, 1000, 136, 5, "bf16_scratch")])
def test_pair_and_one_cta_kernels_bit_identical(z, m, rows, k, n, mode):
    """The CTA-pair kernel (the default) and the one-CTA kernel feed each output the same
    K = 16 products in the same order, so they must give the same bits; with the pair
    kernel checked against the oracle above, this carries the check to the other one."""
    shards = synth.weight_shards(rows, k, n, device=DEV, seed_key=rows + m)
    A = synth.activations(m, k, device=DEV, seed_key=k + m)
    outs = []
    for kernel in (0, 1):
        z.zero_set_gemm_kernel(kernel)
        sw = torch.empty(rows, k, dtype=torch.bfloat16, device=DEV) if mode.endswith("scratch") else None
        if mode.startswith("bf16"):
            out = torch.full((m, rows), float("nan"), dtype=torch.bfloat16, device=DEV)
            z.fsdp_unit_forward(shards, A, None, Y_bf16=out, scratch_w=sw)
        else:
            out = torch.full((m, rows), float("nan"), device=DEV)
            z.fsdp_unit_forward(shards, A, out, scratch_w=sw)
        z.zero_device_status()
        outs.append(out.view(torch.int16 if mode.startswith("bf16") else torch.int32).clone())
    assert torch.equal(outs[0], outs[1]), f"pair and one-CTA kernels differ: {mode} m={m} rows={rows} k={k} n={n}"


def test_mistral_mlp_unit_sampled(z):
    """Mistral-7B MLP unit, N = 8 row shards: W_up / W_gate [14336, 4096] with X [8192,
    4096] and W_down [4096, 14336] with H [8192, 14336]; gather fused into the loads. 4096
    sampled outputs per matrix plus every output column at the shard seams for a few rows,
    each against the float64 oracle under the fp32 summation bound. Memory stays at the
    shards plus activations and output: no gathered W is ever allocated."""
    n, M = 8, 8192
    rng = np.random.default_rng(42)
    X = synth.activations(M, 4096, device=DEV)
    H = synth.activations(M, 14336, device=DEV, seed_key=1)
    for name, R, K, A, key in (("up", 14336, 4096, X, 11), ("gate", 14336, 4096, X, 12), ("down", 4096, 14336, H, 13)):
        shards = synth.weight_shards(R, K, n, device=DEV, seed_key=key)
        Y = torch.empty(M, R, device=DEV)
        torch.cuda.synchronize()
        before = torch.cuda.memory_allocated()
        torch.cuda.reset_peak_memory_stats()
        z.fsdp_unit_forward(shards, A, Y)
        z.zero_device_status()
        assert torch.cuda.max_memory_allocated() <= before, "the fused gather allocated memory"
        rs = R // n
        rows = rng.integers(0, M, 4096)
        cols = rng.integers(0, R, 4096)
        seam_cols = np.array([c for r in range(1, n) for c in (r * rs - 1, r * rs)] + [0, R - 1])
        seam_rows = rng.integers(0, M, 8)
        rows = np.concatenate([rows, np.repeat(seam_rows, seam_cols.size)])
        cols = np.concatenate([cols, np.tile(seam_cols, seam_rows.size)])
        a64 = O.bf16_to_f32(bits16(A[torch.from_numpy(rows).to(DEV)])).astype(np.float64)
        w_full = torch.cat(shards, 0)
        w64 = O.bf16_to_f32(bits16(w_full[torch.from_numpy(cols).to(DEV)])).astype(np.float64)
        exact = np.einsum("ik,ik->i", a64, w64)
        bound = (K + 1) * 2.0 ** -23 * np.einsum("ik,ik->i", np.abs(a64), np.abs(w64))
        got = f32(Y[torch.from_numpy(rows).to(DEV), torch.from_numpy(cols).to(DEV)]).astype(np.float64)
        bad = np.abs(got - exact) > bound
        assert not bad.any(), f"{name}: {bad.sum()} sampled outputs outside the bound"
        del shards, Y, w_full


# aligned (16-byte rows, the pipelined kernel): whole tiles; tiles straddling ranks with
# ragged edges in both dimensions (3 x 40 rows, 72 columns; 5 x 200, 136; 16 x 8, 8); many
# tiles per persistent CTA (X^T of 8 ranks x 2048 tokens x 4096: 16384 tiles).
# unaligned (the element kernel): odd columns, misaligned destination, tiny, rows % 8 != 0
@pytest.mark.parametrize("n,rows,cols,misalign", [(8, 1792, 512, False), (3, 40, 72, False), (5, 200, 136, False),
                                                  (16, 8, 8, False), (8, 2048, 4096, False), (3, 70, 130, False),
                                                  (2, 64, 64, True), (1, 1, 9, False), (4, 129, 8, False)])
def test_transpose_cat_bit_exact(z, n, rows, cols, misalign):
    srcs = synth.weight_shards(n * rows, cols, n, device=DEV, seed_key=rows)
    if misalign:
        dst = torch.zeros(cols * n * rows + 1, dtype=torch.bfloat16, device=DEV)[1:].view(cols, n * rows)
    else:
        dst = torch.zeros(cols, n * rows, dtype=torch.bfloat16, device=DEV)
    z.fsdp_transpose_cat(srcs, dst)
    z.zero_device_status()
    assert_bf16_identical(bits16(dst), O.transpose_cat([bits16(s) for s in srcs]), "transpose_cat")


# ---------------------------------------------------------------------------------------
# FSDP unit backward: dX_q = dY_q W for every rank, dW = (1/N) sum_q dY_q^T X_q
# ---------------------------------------------------------------------------------------

def run_backward(z, n, rows, k, m, key=0, ints=False):
    if ints:
        rng = np.random.default_rng(key)
        mk = lambda shape: torch.from_numpy(O.f32_to_bf16(rng.integers(-2, 3, shape).astype(np.float32))
                                            .view(np.int16)).view(torch.bfloat16).to(DEV)
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


def test_backward_workspace_sizes(z):
    # W, dY and X are read in place when R/N, M and K are multiples of 64 (and N <= 16): no
    # workspace; otherwise W^T, dY^T and X^T
    assert z.fsdp_unit_backward_workspace(8, 14336, 4096, 2048) == 0
    assert z.fsdp_unit_backward_workspace(5, 320, 192, 192) == 0
    assert z.fsdp_unit_backward_workspace(5, 320, 200, 192) > 2 * 200 * 5 * 192
    assert z.fsdp_unit_backward_workspace(4, 512, 256, 40) > 2 * 256 * 4 * 40
    assert z.fsdp_unit_backward_workspace(8, 2048, 512, 96) > 2 * 512 * 8 * 96


# in place: one dX launch over all ranks (M % 128 == 0), per-rank dX launches (M % 128 ==
# 64), ragged output tiles in both GEMMs (R = 320, K = 192: zero-filled column chunks);
# transposed: M = 40, K = 200
@pytest.mark.parametrize("n,rows,k,m", [(4, 512, 256, 128), (5, 320, 192, 192), (5, 320, 200, 192), (3, 120, 72, 40)])
def test_backward_integer_values_exact(z, n, rows, k, m):
    shards, A, dY, dX, dW = run_backward(z, n, rows, k, m, key=3, ints=True)
    w = O.bf16_to_f32(O.gather_rows([bits16(s) for s in shards])).astype(np.float64)
    acc = np.zeros((rows, k))
    for q in range(n):
        a = O.bf16_to_f32(bits16(A[q])).astype(np.float64)
        dy = O.bf16_to_f32(bits16(dY[q])).astype(np.float64)
        assert np.array_equal(f32(dX[q]).astype(np.float64), dy @ w)
        acc += dy.T @ a
    # the sum of small integers is exact in fp32; the 1/N scale is f32(1/N) applied with one
    # fp32 rounding, exact only for N a power of two
    expect = acc.astype(np.float32) * (np.float32(1.0) / np.float32(n))
    assert np.array_equal(f32(dW), expect)


@pytest.mark.parametrize("n,rows,k,m", [(4, 512, 256, 128), (3, 120, 72, 40), (8, 2048, 512, 96), (1, 256, 64, 200),
                                        (2, 256, 64, 64), (5, 320, 192, 192), (1, 128, 64, 64), (16, 1024, 192, 128),
                                        (5, 320, 200, 192),
                                        # transposed path with M % 128 == 0: dX as one row-split GEMM
                                        (2, 200, 72, 128), (3, 192, 40, 256)])
def test_backward_vs_oracle(z, n, rows, k, m):
    shards, A, dY, dX, dW = run_backward(z, n, rows, k, m, key=rows)
    sb = [bits16(s) for s in shards]
    w64 = O.bf16_to_f32(O.gather_rows(sb)).astype(np.float64)
    exact_dw = np.zeros((rows, k))
    bound_dw = np.zeros((rows, k))
    for q in range(n):
        dx64, dw64 = O.fsdp_linear_backward(bits16(A[q]), sb, bits16(dY[q]), n)
        dy_abs = np.abs(O.bf16_to_f32(bits16(dY[q])).astype(np.float64))
        a_abs = np.abs(O.bf16_to_f32(bits16(A[q])).astype(np.float64))
        bound_dx = (rows + 1) * 2.0 ** -23 * (dy_abs @ np.abs(w64))
        assert np.all(np.abs(f32(dX[q]) - dx64) <= bound_dx), f"dX of rank {q}"
        exact_dw += dw64
        bound_dw += dy_abs.T @ a_abs
    exact_dw /= n
    bound = (n * m + 1) * 2.0 ** -23 * bound_dw / n + 2.0 ** -24 * np.abs(exact_dw)
    assert np.all(np.abs(f32(dW) - exact_dw) <= bound), "reduce-scattered dW"
    # each rank's shard of the reduced gradient equals the oracle's per-rank reduce-scatter
    # of the fp32 per-rank dW (both within the same bound of the exact sum)
    rs = rows // n
    dws32 = [O.fsdp_linear_backward(bits16(A[q]), sb, bits16(dY[q]), n)[1].astype(np.float32) for q in range(n)]
    for r in range(n):
        ref = O.reduce_rows(dws32, n, r).astype(np.float64)
        assert np.all(np.abs(f32(dW)[r * rs:(r + 1) * rs] - ref) <= 2 * bound[r * rs:(r + 1) * rs] + 1e-30)


def test_backward_mistral_up_sampled(z):
    """W_up [14336, 4096] in 8 row shards, 2048 tokens per rank: sampled dX and dW entries
    against float64 dot products under the bounds."""
    n, rows, k, m = 8, 14336, 4096, 2048
    shards, A, dY, dX, dW = run_backward(z, n, rows, k, m, key=7)
    rng = np.random.default_rng(1)
    w_full = torch.cat(shards, 0)
    for q in (0, n - 1):
        i = rng.integers(0, m, 512)
        c = rng.integers(0, k, 512)
        dy = O.bf16_to_f32(bits16(dY[q][torch.from_numpy(i).to(DEV)])).astype(np.float64)
        wc = O.bf16_to_f32(bits16(w_full[:, torch.from_numpy(c).to(DEV)].t().contiguous())).astype(np.float64)
        exact = np.einsum("ir,ir->i", dy, wc)
        bound = (rows + 1) * 2.0 ** -23 * np.einsum("ir,ir->i", np.abs(dy), np.abs(wc))
        got = f32(dX[q][torch.from_numpy(i).to(DEV), torch.from_numpy(c).to(DEV)]).astype(np.float64)
        assert np.all(np.abs(got - exact) <= bound), f"dX rank {q}"
    rr = rng.integers(0, rows, 256)
    cc = rng.integers(0, k, 256)
    ex = np.zeros(256)
    bd = np.zeros(256)
    for q in range(n):
        dyc = O.bf16_to_f32(bits16(dY[q][:, torch.from_numpy(rr).to(DEV)].t().contiguous())).astype(np.float64)
        ac = O.bf16_to_f32(bits16(A[q][:, torch.from_numpy(cc).to(DEV)].t().contiguous())).astype(np.float64)
        ex += np.einsum("im,im->i", dyc, ac)
        bd += np.einsum("im,im->i", np.abs(dyc), np.abs(ac))
    ex /= n
    bound = (n * m + 1) * 2.0 ** -23 * bd / n + 2.0 ** -24 * np.abs(ex)
    got = f32(dW[torch.from_numpy(rr).to(DEV), torch.from_numpy(cc).to(DEV)]).astype(np.float64)
    assert np.all(np.abs(got - ex) <= bound), "dW"


def test_backward_mistral_down_sampled(z):
    """W_down [4096, 14336] in 8 row shards of 512 rows (read in place by the dX GEMM),
    1024 tokens per rank: sampled dX and dW entries against float64 dot products under the
    bounds."""
    n, rows, k, m = 8, 4096, 14336, 1024
    assert z.fsdp_unit_backward_workspace(n, rows, k, m) == 0  # every operand read in place
    shards, A, dY, dX, dW = run_backward(z, n, rows, k, m, key=9)
    rng = np.random.default_rng(2)
    w_full = torch.cat(shards, 0)
    for q in (0, 3, n - 1):
        i = torch.from_numpy(rng.integers(0, m, 384)).to(DEV)
        c = torch.from_numpy(rng.integers(0, k, 384)).to(DEV)
        dy = O.bf16_to_f32(bits16(dY[q][i])).astype(np.float64)
        wc = O.bf16_to_f32(bits16(w_full[:, c].t().contiguous())).astype(np.float64)
        exact = np.einsum("ir,ir->i", dy, wc)
        bound = (rows + 1) * 2.0 ** -23 * np.einsum("ir,ir->i", np.abs(dy), np.abs(wc))
        assert np.all(np.abs(f32(dX[q][i, c]).astype(np.float64) - exact) <= bound), f"dX rank {q}"
    # dW rows on both sides of every shard seam, random columns
    rr = np.concatenate([np.arange(1, n) * (rows // n) + d for d in (-1, 0)] + [rng.integers(0, rows, 128)])
    cc = rng.integers(0, k, rr.size)
    ex = np.zeros(rr.size)
    bd = np.zeros(rr.size)
    for q in range(n):
        dyc = O.bf16_to_f32(bits16(dY[q][:, torch.from_numpy(rr).to(DEV)].t().contiguous())).astype(np.float64)
        ac = O.bf16_to_f32(bits16(A[q][:, torch.from_numpy(cc).to(DEV)].t().contiguous())).astype(np.float64)
        ex += np.einsum("im,im->i", dyc, ac)
        bd += np.einsum("im,im->i", np.abs(dyc), np.abs(ac))
    ex /= n
    bound = (n * m + 1) * 2.0 ** -23 * bd / n + 2.0 ** -24 * np.abs(ex)
    got = f32(dW[torch.from_numpy(rr).to(DEV), torch.from_numpy(cc).to(DEV)]).astype(np.float64)
    assert np.all(np.abs(got - ex) <= bound), "dW"


@pytest.mark.parametrize("n,rows,k,m", [(4, 512, 256, 128), (5, 320, 192, 192), (8, 2048, 512, 64),
                                        (8, 3584, 128, 512), (4, 256, 1024, 128), (8, 512, 2048, 64)])
def test_backward_in_place_same_bits_on_both_kernels(z, n, rows, k, m):
    """The in-place backward (W's shards, dY and X all read as MN-major operands, no
    workspace: None is accepted, and a workspace passed anyway is not touched) gives the
    same dX and dW bits on the CTA-pair kernel as on the one-CTA kernel, whose layouts
    and K loops are compiled separately."""
    assert z.fsdp_unit_backward_workspace(n, rows, k, m) == 0
    shards = synth.weight_shards(rows, k, n, device=DEV, seed_key=5)
    A = [synth.activations(m, k, device=DEV, seed_key=q) for q in range(n)]
    dY = [synth.upstream_grad(m, rows, device=DEV, seed_key=q) for q in range(n)]
    out = []
    spare = torch.full((1 << 16,), 0x5A, dtype=torch.uint8, device=DEV)
    try:
        for kernel, ws in ((0, None), (1, spare)):
            z.zero_set_gemm_kernel(kernel)
            dX = [torch.full((m, k), float("nan"), device=DEV) for _ in range(n)]
            dW = torch.full((rows, k), float("nan"), device=DEV)
            z.fsdp_unit_backward(shards, A, dY, dX, dW, ws)
            z.zero_device_status()
            out.append((dX, dW))
    finally:
        z.zero_set_gemm_kernel(0)
    (dXa, dWa), (dXb, dWb) = out
    assert torch.equal(dWa.view(torch.int32), dWb.view(torch.int32))
    for a, b in zip(dXa, dXb):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert bool((spare == 0x5A).all())


@pytest.mark.parametrize("n,rows,k,m", [(8, 512, 2048, 128), (4, 1024, 256, 192)])
def test_backward_dw_equals_k_major_product_of_transposes(z, n, rows, k, m):
    """dW does not depend on the operands' layout: fsdp_unit_backward's dW (dY and X both
    read in place as MN-major operands) equals, bit for bit, the K-major product dY^T
    (X^T)^T of both transposes through fsdp_unit_forward, scaled by 1/N (exact for N a
    power of two)."""
    shards = synth.weight_shards(rows, k, n, device=DEV, seed_key=8)
    A = [synth.activations(m, k, device=DEV, seed_key=q) for q in range(n)]
    dY = [synth.upstream_grad(m, rows, device=DEV, seed_key=q) for q in range(n)]
    dX = [torch.empty(m, k, device=DEV) for _ in range(n)]
    dW = torch.empty(rows, k, device=DEV)
    ws = torch.empty(z.fsdp_unit_backward_workspace(n, rows, k, m), dtype=torch.uint8, device=DEV)
    z.fsdp_unit_backward(shards, A, dY, dX, dW, ws)
    dyt = torch.empty(rows, n * m, dtype=torch.bfloat16, device=DEV)
    xt = torch.empty(k, n * m, dtype=torch.bfloat16, device=DEV)
    z.fsdp_transpose_cat(dY, dyt)
    z.fsdp_transpose_cat(A, xt)
    ref = torch.empty(rows, k, device=DEV)
    z.fsdp_unit_forward([xt], dyt, ref)
    z.zero_device_status()
    assert torch.equal(dW.view(torch.int32), (ref * (1.0 / n)).view(torch.int32))


def test_backward_rejects_small_workspace(z):
    n, rows, k, m = 2, 512, 64, 40
    shards = synth.weight_shards(rows, k, n, device=DEV)
    A = [synth.activations(m, k, device=DEV) for _ in range(n)]
    dY = [synth.upstream_grad(m, rows, device=DEV) for _ in range(n)]
    dX = [torch.empty(m, k, device=DEV) for _ in range(n)]
    dW = torch.empty(rows, k, device=DEV)
    ws = torch.empty(z.fsdp_unit_backward_workspace(n, rows, k, m) - 256, dtype=torch.uint8, device=DEV)
    with pytest.raises(z.ZeroError) as e:
        z.fsdp_unit_backward(shards, A, dY, dX, dW, ws)
    assert e.value.code == -1


# ---------------------------------------------------------------------------------------
# full MLP unit: H = silu(X Wg^T) * (X Wu^T) in one kernel, then Y = H Wd^T
# ---------------------------------------------------------------------------------------

def h_bound(g64, u64, bg, bu, h_gpu):
    """|H_gpu - H_exact| for H = silu(G) U from fp32 G, U within bg, bu of exact:
    |silu'| <= 1.1, a few fp32 roundings in silu and the product, one bf16 rounding."""
    sil = np.abs(O.silu(g64))
    return (1.1 * bg * np.abs(u64) + sil * bu + 1.1 * bg * bu + 16 * 2.0 ** -24 * sil * np.abs(u64)
            + 2.0 ** -8 * 1.01 * np.abs(h_gpu) + 1e-38)


def make_mlp(n, d, f, m, key):
    gate = synth.weight_shards(f, d, n, device=DEV, seed_key=10 * key + 1)
    up = synth.weight_shards(f, d, n, device=DEV, seed_key=10 * key + 2)
    down = synth.weight_shards(d, f, n, device=DEV, seed_key=10 * key + 3)
    X = synth.activations(m, d, device=DEV, seed_key=key)
    return gate, up, down, X


@pytest.mark.parametrize("n,d,f,m,scratch", [(2, 512, 512, 200, False), (2, 256, 512, 200, True),
                                             (4, 1024, 1024, 130, False), (8, 2048, 1024, 64, True),
                                             (1, 256, 256, 1, False), (3, 384, 384, 100, False),
                                             # pair-tile edges: M around 256, ragged d_model via scratch
                                             (2, 256, 256, 257, False), (1, 136, 128, 255, True),
                                             (4, 512, 512, 1, False)])
def test_mlp_unit_vs_oracle(z, n, d, f, m, scratch):
    gate, up, down, X = make_mlp(n, d, f, m, key=d + f)
    H = torch.zeros(m, f, dtype=torch.bfloat16, device=DEV)
    Y = torch.full((m, d), float("nan"), device=DEV)
    sd = torch.empty(d, f, dtype=torch.bfloat16, device=DEV) if scratch else None
    side = torch.cuda.Stream() if scratch else None
    z.fsdp_mlp_forward(gate, up, down, X, H, Y, scratch_down=sd, prefetch_stream=side)
    z.zero_device_status()
    gb, ub, db, xb = [bits16(s) for s in gate], [bits16(s) for s in up], [bits16(s) for s in down], bits16(X)
    hb = bits16(H)
    g64, u64, h64, y64 = O.mlp_unit_forward(xb, gb, ub, db, h_bf16=hb)
    xa = np.abs(O.bf16_to_f32(xb).astype(np.float64))
    bg = (d + 1) * 2.0 ** -23 * (xa @ np.abs(O.bf16_to_f32(O.gather_rows(gb)).astype(np.float64)).T)
    bu = (d + 1) * 2.0 ** -23 * (xa @ np.abs(O.bf16_to_f32(O.gather_rows(ub)).astype(np.float64)).T)
    h_gpu = O.bf16_to_f32(hb).astype(np.float64)
    assert np.all(np.abs(h_gpu - h64) <= h_bound(g64, u64, bg, bu, h_gpu)), "H"
    by = (f + 1) * 2.0 ** -23 * (np.abs(h_gpu) @ np.abs(O.bf16_to_f32(O.gather_rows(db)).astype(np.float64)).T)
    assert np.all(np.abs(f32(Y) - y64) <= by + 1e-30), "Y"
    if scratch:
        assert_bf16_identical(bits16(sd), O.gather_rows(db), "W_down gathered into scratch")
    if (d // n) % 128 == 0:
        Y2 = torch.empty_like(Y)
        H2 = torch.empty_like(H)
        z.fsdp_mlp_forward(gate, up, down, X, H2, Y2,
                           scratch_down=torch.empty(d, f, dtype=torch.bfloat16, device=DEV), prefetch_stream=None)
        z.zero_device_status()
        assert torch.equal(H2.view(torch.int16), H.view(torch.int16))
        assert torch.equal(Y2.view(torch.int32), Y.view(torch.int32)), "fused and scratch W_down disagree"


def test_mlp_unit_mistral_sampled(z):
    """Mistral-7B MLP unit, N = 8 shards, 8192 tokens: 4096 sampled H entries against the
    float64 oracle, 4096 sampled Y entries against float64 dot products of the kernel's H."""
    n, d, f, m = 8, 4096, 14336, 8192
    gate, up, down, X = make_mlp(n, d, f, m, key=5)
    H = torch.empty(m, f, dtype=torch.bfloat16, device=DEV)
    Y = torch.empty(m, d, device=DEV)
    z.fsdp_mlp_forward(gate, up, down, X, H, Y)
    z.zero_device_status()
    rng = np.random.default_rng(3)
    i = torch.from_numpy(rng.integers(0, m, 4096)).to(DEV)
    j = torch.from_numpy(rng.integers(0, f, 4096)).to(DEV)
    xi = O.bf16_to_f32(bits16(X[i])).astype(np.float64)
    wg = O.bf16_to_f32(bits16(torch.cat(gate)[j])).astype(np.float64)
    wu = O.bf16_to_f32(bits16(torch.cat(up)[j])).astype(np.float64)
    g64, u64 = np.einsum("ik,ik->i", xi, wg), np.einsum("ik,ik->i", xi, wu)
    bg = (d + 1) * 2.0 ** -23 * np.einsum("ik,ik->i", np.abs(xi), np.abs(wg))
    bu = (d + 1) * 2.0 ** -23 * np.einsum("ik,ik->i", np.abs(xi), np.abs(wu))
    h_gpu = O.bf16_to_f32(bits16(H[i, j])).astype(np.float64)
    assert np.all(np.abs(h_gpu - O.silu(g64) * u64) <= h_bound(g64, u64, bg, bu, h_gpu)), "H"
    c = torch.from_numpy(rng.integers(0, d, 4096)).to(DEV)
    hi = O.bf16_to_f32(bits16(H[i])).astype(np.float64)
    wd = O.bf16_to_f32(bits16(torch.cat(down)[c])).astype(np.float64)
    ex = np.einsum("ik,ik->i", hi, wd)
    by = (f + 1) * 2.0 ** -23 * np.einsum("ik,ik->i", np.abs(hi), np.abs(wd))
    assert np.all(np.abs(f32(Y[i, c]).astype(np.float64) - ex) <= by + 1e-30), "Y"


@pytest.mark.parametrize("n,d,f,m,scratch", [(2, 512, 512, 200, False), (4, 1024, 1024, 130, True),
                                             (1, 256, 384, 257, False)])
def test_mlp_unit_pair_and_one_cta_kernels_bit_identical(z, n, d, f, m, scratch):
    """Gate-up and down projections on the CTA-pair kernels (the default) and on the one-CTA
    kernels: H and Y bit for bit the same."""
    gate, up, down, X = make_mlp(n, d, f, m, key=3 * d + f)
    outs = []
    for kernel in (0, 1):
        z.zero_set_gemm_kernel(kernel)
        H = torch.zeros(m, f, dtype=torch.bfloat16, device=DEV)
        Y = torch.full((m, d), float("nan"), device=DEV)
        sd = torch.empty(d, f, dtype=torch.bfloat16, device=DEV) if scratch else None
        z.fsdp_mlp_forward(gate, up, down, X, H, Y, scratch_down=sd, prefetch_stream=None)
        z.zero_device_status()
        outs.append((H.view(torch.int16).clone(), Y.view(torch.int32).clone()))
    assert torch.equal(outs[0][0], outs[1][0]), "H"
    assert torch.equal(outs[0][1], outs[1][1]), "Y"


@pytest.mark.parametrize("n,rows,k,m", [(3, 120, 72, 40), (5, 320, 200, 192), (4, 512, 256, 128), (8, 2048, 512, 96),
                                        (16, 1024, 192, 128), (1, 128, 64, 64), (2, 200, 72, 128), (3, 192, 40, 256)])
def test_backward_pair_and_one_cta_kernels_bit_identical(z, n, rows, k, m):
    """The backward under the default choice, on the one-CTA kernels everywhere and on the
    CTA-pair kernels everywhere (selectors 0, 1, 2) gives the same dX and dW bits: the
    transposed path (K-major operands) and the in-place path (MN-major W and dY; dX over all
    ranks' row pieces when M % 128 == 0, else per rank)."""
    outs = []
    for kernel in (0, 1, 2):
        z.zero_set_gemm_kernel(kernel)
        _, _, _, dX, dW = run_backward(z, n, rows, k, m, key=rows + 1)
        outs.append(([x.view(torch.int32).clone() for x in dX], dW.view(torch.int32).clone()))
    for sel in (1, 2):
        for q in range(n):
            assert torch.equal(outs[0][0][q], outs[sel][0][q]), f"dX of rank {q}, selector {sel}"
        assert torch.equal(outs[0][1], outs[sel][1]), f"dW, selector {sel}"


def test_fsdp_calls_replay_from_a_cuda_graph(z):
    """The FSDP calls are plain stream work (host-encoded tensor maps passed by value, no
    allocation, the MLP unit's prefetch stream forked and joined through events), so they
    can be captured once in a CUDA graph and replayed: the forward with its fused gather, the
    MLP unit with W_down gathered on a prefetch stream, and the backward give the same bits
    as eager calls."""
    n, R, K, M = 4, 1024, 256, 256
    shards = synth.weight_shards(R, K, n, device=DEV, seed_key=91)
    X = synth.activations(M, K, device=DEV, seed_key=92)
    gate, up, down, Xm = make_mlp(2, 512, 512, 200, key=93)
    Hm_e = torch.empty(200, 512, dtype=torch.bfloat16, device=DEV)
    Ym_e = torch.empty(200, 512, device=DEV)
    sd = torch.empty(512, 512, dtype=torch.bfloat16, device=DEV)
    A = [synth.activations(64, K, device=DEV, seed_key=94 + q) for q in range(n)]
    dY = [synth.upstream_grad(64, R, device=DEV, seed_key=94 + q) for q in range(n)]
    ws = torch.empty(z.fsdp_unit_backward_workspace(n, R, K, 64), dtype=torch.uint8, device=DEV)

    def run(Y, Hm, Ym, dX, dW, stream, side):
        z.fsdp_unit_forward(shards, X, Y, stream=stream)
        z.fsdp_mlp_forward(gate, up, down, Xm, Hm, Ym, scratch_down=sd, stream=stream, prefetch_stream=side)
        z.fsdp_unit_backward(shards, A, dY, dX, dW, ws, stream=stream)

    def fresh():
        return (torch.full((M, R), float("nan"), device=DEV),
                torch.zeros(200, 512, dtype=torch.bfloat16, device=DEV),
                torch.full((200, 512), float("nan"), device=DEV),
                [torch.full((64, K), float("nan"), device=DEV) for _ in range(n)],
                torch.full((R, K), float("nan"), device=DEV))

    eager = fresh()
    side = torch.cuda.Stream()
    run(*eager, torch.cuda.current_stream(), side)
    z.zero_device_status()
    got = fresh()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(g, stream=cap):
            run(*got, cap, side)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    z.zero_device_status()
    assert torch.equal(eager[0].view(torch.int32), got[0].view(torch.int32)), "forward"
    assert torch.equal(eager[1].view(torch.int16), got[1].view(torch.int16)), "MLP H"
    assert torch.equal(eager[2].view(torch.int32), got[2].view(torch.int32)), "MLP Y"
    for q in range(n):
        assert torch.equal(eager[3][q].view(torch.int32), got[3][q].view(torch.int32)), f"dX of rank {q}"
    assert torch.equal(eager[4].view(torch.int32), got[4].view(torch.int32)), "dW"


@pytest.mark.parametrize("n,R,K,M", [(4, 512, 256, 200), (8, 1024, 136, 130)])
def test_zero3_step_feeds_the_fsdp_unit(z, n, R, K, M):
    """The ZeRO-3 / FSDP cycle of one linear layer: its weight W [R, K] is the flat parameter
    (psi = R K), so a rank's ZeRO-3 shard [rS, (r+1)S) is exactly W's row shard r. Two fused
    optimizer steps (every rank, bf16 parameter shards out) must equal the oracle's ZeRO-3
    ranks bit for bit, and the next forward, gathering those shards inside the GEMM's loads,
    must stay within the fp32 bound of the oracle's float64 product with the oracle's W."""
    psi, bb = R * K, 1 << 16
    plan = z.zero_plan(psi, n, "zero3", bb)
    assert plan.psi_padded == psi and (R // n) * K == plan.shard_elems
    lay = O.make_layout(psi, n, bb)
    hp = O.AdamHyper()
    master0 = synth.master_params(psi, psi, seed_key=R)
    ranks = O.init_ranks("zero3", lay, master0.numpy())
    master = master0.to(DEV)
    m, v = torch.zeros(psi, device=DEV), torch.zeros(psi, device=DEV)
    param = torch.zeros(psi, dtype=torch.bfloat16, device=DEV)
    for t in (1, 2):
        grads = [synth.rank_grads(psi, psi, r, t, seed_key=R) for r in range(n)]
        z.zero_fused_step(plan, z.ZERO_ALL_RANKS, [g.to(DEV) for g in grads], master, m, v, param, hp, t)
        O.step_ranks(ranks, lay, [bits16(g) for g in grads], hp, t)
    z.zero_device_status()
    assert_bf16_identical(bits16(param), O.gather_params(ranks), "ZeRO-3 parameter shards")
    S = plan.shard_elems
    shards = [param[r * S:(r + 1) * S].view(R // n, K) for r in range(n)]
    X = synth.activations(M, K, device=DEV, seed_key=K)
    Y = torch.full((M, R), float("nan"), device=DEV)
    z.fsdp_unit_forward(shards, X, Y)
    z.zero_device_status()
    w_or = O.gather_params(ranks).reshape(R, K)
    check_gemm(f32(Y), bits16(X), [w_or[r * (R // n):(r + 1) * (R // n)] for r in range(n)],
               f"ZeRO-3 shards into the FSDP unit, n={n} R={R} K={K} M={M}")


@pytest.mark.parametrize("m,rows,k,n", [(255, 128, 8, 1), (257, 384, 56, 3), (1, 1152, 16, 9), (512, 256, 4104, 2),
                                        (256, 640, 64, 5), (129, 128, 200, 1)])
def test_pair_kernel_edge_shapes_vs_oracle(z, m, rows, k, n):
    """Edges of the CTA-pair tiling against the oracle: K shorter than one 64-wide block or
    ending in a ragged one, M just under / over a 256-row pair tile (the odd CTA's rows
    past M), R with a 128-row half past the last shard row, one to nine shards."""
    shards = synth.weight_shards(rows, k, n, device=DEV, seed_key=m + k)
    A = synth.activations(m, k, device=DEV, seed_key=rows)
    Y = torch.full((m, rows), float("nan"), device=DEV)
    z.fsdp_unit_forward(shards, A, Y)
    z.zero_device_status()
    check_gemm(f32(Y), bits16(A), [bits16(s) for s in shards], f"pair edge m={m} rows={rows} k={k} n={n}")
