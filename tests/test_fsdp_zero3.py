"""GPU parity of one ZeRO-3 / FSDP training step over a stack of units (fsdp_zero3_step).

The step follows a unit's life on a card ([Interview] Fig. 2): forward over the units
(gather, product, free), backward in reverse (gather again, dX, full-shape dW reduced over
the ranks so rank r keeps rows [r R/N, (r+1) R/N)), then each rank's Adam on its shard,
giving the new bf16 shards the next step's forward reads. Every buffer the step writes is
checked against the oracle, unit by unit, on the inputs the GPU gave that unit (each is an
exact bf16 or fp32 value):
  - X_{i+1} = bf16(X_i W_i^T) and dY_{i-1} = bf16(dY_i W_i): the kernel rounds an fp32 sum
    that lies within the fp32 bound B = (K + 1) 2^-23 sum|a w| of the exact product, so its
    bf16 output lies between RNE(exact - B) and RNE(exact + B) (rounding is monotone);
  - dW_i against (1/N) sum_q dY_q^T X_q under the fp32 bound, and each rank's rows against
    the oracle's reduce-scatter of the per-rank fp32 dW;
  - master, m, v and the new bf16 shards bit for bit against the oracle's Adam on the
    GPU's dW (the Adam arithmetic is exact on both sides);
  - the old W_i (not the updated one) feeds unit i's dX: the update follows the last use.
Flags (fused or materialised gather, with or without the prefetch stream) give the same bits.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle.zero_oracle as O
import synth
from _util import assert_bf16_identical, assert_f32_identical, bits16, f32

pytestmark = pytest.mark.gpu
DEV = "cuda"
HP = {"lr": 1e-4, "beta1": 0.9, "beta2": 0.999, "eps": 1e-8, "weight_decay": 0.0}


@pytest.fixture(scope="module")
def z():
    import __graft_entry__ as g
    g.build()
    import fsdp_sharded_optimizer_zero_gb300 as z
    return z


def make_units(z, n, shapes, m, key):
    """units[i]: W [R, K] (N row shards back to back) ~ N(0, 0.02) bf16, master = W in fp32,
    m = v = 0; unit 0's input batch and the last unit's loss gradient seeded bf16."""
    units = []
    nm = n * m
    for i, (R, K) in enumerate(shapes):
        w = torch.cat(synth.weight_shards(R, K, n, device=DEV, seed_key=100 * key + i), 0).contiguous()
        units.append({"plan": z.zero_plan(R * K, n, "zero3", 1 << 20), "w": w, "master": w.float().reshape(-1).clone(),
                      "m": torch.zeros(R * K, device=DEV), "v": torch.zeros(R * K, device=DEV),
                      "x": torch.zeros(nm, K, dtype=torch.bfloat16, device=DEV),
                      "dy": torch.zeros(nm, R, dtype=torch.bfloat16, device=DEV),
                      "dw": torch.full((R, K), float("nan"), device=DEV)})
    units[0]["x"].copy_(synth.activations(nm, shapes[0][1], device=DEV, seed_key=key))
    units[-1]["dy"].copy_(synth.upstream_grad(nm, shapes[-1][0], device=DEV, seed_key=key))
    return units


def clone_units(units):
    return [{k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in u.items()} for u in units]


def run_step(z, units, m, step, flags, y=True, dx=True, prefetch=True):
    nm = units[0]["x"].shape[0]
    shapes = [tuple(u["w"].shape) for u in units]
    ws = torch.empty(z.fsdp_zero3_step_workspace(units[0]["plan"].n_ranks, shapes, m, flags), dtype=torch.uint8,
                     device=DEV)
    y_out = torch.full((nm, shapes[-1][0]), float("nan"), dtype=torch.bfloat16, device=DEV) if y else None
    dx_out = torch.full((nm, shapes[0][1]), float("nan"), dtype=torch.bfloat16, device=DEV) if dx else None
    side = torch.cuda.Stream() if prefetch else None
    z.fsdp_zero3_step(units, m, HP, step, y_out=y_out, dx_out=dx_out, flags=flags, workspace=ws,
                      prefetch_stream=side)
    z.zero_device_status()
    return y_out, dx_out


def snapshot(units):
    return [{"w": bits16(u["w"]), "master": f32(u["master"]).copy(), "m": f32(u["m"]).copy(),
             "v": f32(u["v"]).copy(), "x": bits16(u["x"]), "dy": bits16(u["dy"])} for u in units]


def check_bf16_product(out_bits, exact, bound, what):
    """out = RNE(s) for an fp32 s within `bound` of `exact`: RNE(lo) <= out <= RNE(hi)."""
    lo = np.nextafter((exact - bound).astype(np.float32), np.float32(-np.inf))
    hi = np.nextafter((exact + bound).astype(np.float32), np.float32(np.inf))
    out = O.bf16_to_f32(out_bits)
    ok = (O.bf16_to_f32(O.f32_to_bf16(lo)) <= out) & (out <= O.bf16_to_f32(O.f32_to_bf16(hi)))
    assert ok.all(), f"{what}: {(~ok).sum()} of {ok.size} bf16 outputs outside the rounded bound"


def shards(bits, n):
    rs = bits.shape[0] // n
    return [bits[r * rs:(r + 1) * rs] for r in range(n)]


def check_step(z, n, m, before, units, y_out, dx_out, t):
    """Every buffer of one step against the oracle, on the GPU's own inputs to each unit."""
    L = len(units)
    hp = O.AdamHyper(**HP)
    for i in range(L):
        R, K = units[i]["w"].shape
        w_old = before[i]["w"]
        w64 = np.abs(O.bf16_to_f32(w_old).astype(np.float64))
        x_in = bits16(units[i]["x"]) if i > 0 else before[0]["x"]
        # forward output of unit i
        out = bits16(units[i + 1]["x"]) if i + 1 < L else (bits16(y_out) if y_out is not None else None)
        if out is not None:
            y64, _, _ = O.fsdp_linear_forward(x_in, shards(w_old, n))
            b = (K + 1) * 2.0 ** -23 * (np.abs(O.bf16_to_f32(x_in).astype(np.float64)) @ w64.T)
            check_bf16_product(out, y64, b, f"forward of unit {i}")
        # backward of unit i: dY_i is the GPU's (given for the last unit)
        dy = bits16(units[i]["dy"]) if i + 1 < L else before[i]["dy"]
        dy64 = O.bf16_to_f32(dy).astype(np.float64)
        dx_got = bits16(units[i - 1]["dy"]) if i > 0 else (bits16(dx_out) if dx_out is not None else None)
        if dx_got is not None:
            dx64 = dy64 @ O.bf16_to_f32(w_old).astype(np.float64)
            b = (R + 1) * 2.0 ** -23 * (np.abs(dy64) @ w64)
            check_bf16_product(dx_got, dx64, b, f"dX of unit {i}")
        # dW over every rank's tokens, and each rank's reduce-scattered rows
        x64 = O.bf16_to_f32(x_in).astype(np.float64)
        dws32, exact, bnd = [], np.zeros((R, K)), np.zeros((R, K))
        for q in range(n):
            rows = slice(q * m, (q + 1) * m)
            _, dwq = O.fsdp_linear_backward(x_in[rows], shards(w_old, n), dy[rows], n)
            dws32.append(dwq.astype(np.float32))
            exact += dwq
            bnd += np.abs(dy64[rows]).T @ np.abs(x64[rows])
        exact /= n
        bound = (n * m + 1) * 2.0 ** -23 * bnd / n + 2.0 ** -24 * np.abs(exact)
        dw = f32(units[i]["dw"])
        assert np.all(np.abs(dw - exact) <= bound), f"dW of unit {i}"
        rs = R // n
        for r in range(n):
            ref = O.reduce_rows(dws32, n, r).astype(np.float64)
            assert np.all(np.abs(dw[r * rs:(r + 1) * rs] - ref) <= 2 * bound[r * rs:(r + 1) * rs] + 1e-30), \
                f"rank {r}'s reduce-scattered rows of unit {i}"
        # each rank's Adam on its shard, from the GPU's dW: bit-exact
        S = R * K // n
        g = dw.reshape(-1)
        for r in range(n):
            sl = slice(r * S, (r + 1) * S)
            w_new, m_new, v_new = O.adam_update(before[i]["master"][sl], before[i]["m"][sl], before[i]["v"][sl],
                                                g[sl], hp, t)
            assert_f32_identical(f32(units[i]["master"])[sl], w_new, f"master of unit {i} rank {r}")
            assert_f32_identical(f32(units[i]["m"])[sl], m_new, f"m of unit {i} rank {r}")
            assert_f32_identical(f32(units[i]["v"])[sl], v_new, f"v of unit {i} rank {r}")
            assert_bf16_identical(bits16(units[i]["w"]).reshape(-1)[sl], O.f32_to_bf16(w_new),
                                  f"new bf16 shard of unit {i} rank {r}")


# shapes chain: unit i's k_in is unit i-1's rows_out
CASES = [
    # N = 4, shard rows 128 / 256: the fused gather; M = 100 tokens per rank (N M = 400: a ragged K block in dW)
    (4, [(512, 256), (1024, 512), (512, 1024)], 100, 0),
    # N = 3, unit 0's shard rows 64 do not tile the GEMM: materialised gather
    (3, [(192, 128), (384, 192)], 64, 1),
    # N = 8, one unit
    (8, [(2048, 512)], 128, 0),
]


@pytest.mark.parametrize("n,shapes,m,flags", CASES)
def test_zero3_step_every_buffer_vs_oracle(z, n, shapes, m, flags):
    units = make_units(z, n, shapes, m, key=len(shapes) + n)
    for t in (1, 2):  # the second step's forward reads the shards the first one wrote
        before = snapshot(units)
        y_out, dx_out = run_step(z, units, m, t, flags | z.FSDP_BACKWARD_PREFETCH | z.FSDP_OVERLAP_OPTIMIZER)
        check_step(z, n, m, before, units, y_out, dx_out, t)


@pytest.mark.parametrize("n,shapes,m", [(4, [(512, 256), (1024, 512), (512, 1024)], 96), (2, [(256, 64), (256, 256)], 200)])
def test_zero3_step_flags_give_the_same_bits(z, n, shapes, m):
    """Fused or materialised gather, serial, with the prefetch stream, with Adam fused into
    the dW GEMM (the default), as its own launch or on the side stream: same bits in every
    buffer, over two steps."""
    base = make_units(z, n, shapes, m, key=7)
    results = []
    for flags, prefetch in ((0, False), (2, True), (1, False), (3, True), (2, False), (4, True), (6, True), (7, True),
                            (4, False), (8, False), (10, True), (9, True)):
        units = clone_units(base)
        for t in (1, 2):
            y_out, dx_out = run_step(z, units, m, t, flags, prefetch=prefetch)
        results.append((units, y_out, dx_out))
    ref_units, ref_y, ref_dx = results[0]
    for units, y, dx in results[1:]:
        assert torch.equal(y.view(torch.int16), ref_y.view(torch.int16))
        assert torch.equal(dx.view(torch.int16), ref_dx.view(torch.int16))
        for a, b in zip(units, ref_units):
            for key in ("w", "x", "dy"):
                assert torch.equal(a[key].view(torch.int16), b[key].view(torch.int16)), key
            for key in ("master", "m", "v", "dw"):
                assert torch.equal(a[key].view(torch.int32), b[key].view(torch.int32)), key


def test_zero3_step_without_dw_output_same_update(z):
    """With the optimizer fused into the dW GEMM (the default), dW need not be written: a
    step with dw = None leaves master, m, v, the shards and every activation bit for bit as
    a step that writes dW, over two steps."""
    n, shapes, m = 4, [(512, 256), (1024, 512), (512, 1024)], 100
    a = make_units(z, n, shapes, m, key=13)
    b = clone_units(a)
    for u in b:
        u.pop("dw")
    for t in (1, 2):
        ya, dxa = run_step(z, a, m, t, 0)
        yb, dxb = run_step(z, b, m, t, 0)
        assert torch.equal(ya.view(torch.int16), yb.view(torch.int16))
        assert torch.equal(dxa.view(torch.int16), dxb.view(torch.int16))
    for ua, ub in zip(a, b):
        for key in ("w", "x", "dy"):
            assert torch.equal(ua[key].view(torch.int16), ub[key].view(torch.int16)), key
        for key in ("master", "m", "v"):
            assert torch.equal(ua[key].view(torch.int32), ub[key].view(torch.int32)), key


@pytest.mark.parametrize("flags", [0, 8])
def test_zero3_step_same_bits_on_both_gemm_kernels(z, flags):
    """The step on the one-CTA GEMM kernel (zero_set_gemm_kernel(1): its own layout
    instantiations, and its 4-warp fused-optimizer epilogue) leaves every buffer bit for bit
    as on the default CTA-pair kernel, over two steps, with Adam fused (0) or separate (8).
    Shard rows of 256 so that both kernels take the fused gather."""
    n, shapes, m = 4, [(1024, 256), (1024, 1024), (1024, 1024)], 72
    base = make_units(z, n, shapes, m, key=29)
    out = []
    try:
        for kernel in (0, 1):
            z.zero_set_gemm_kernel(kernel)
            units = clone_units(base)
            for t in (1, 2):
                y, dx = run_step(z, units, m, t, flags)
            out.append((units, y, dx))
    finally:
        z.zero_set_gemm_kernel(0)
    (ua, ya, dxa), (ub, yb, dxb) = out
    assert torch.equal(ya.view(torch.int16), yb.view(torch.int16))
    assert torch.equal(dxa.view(torch.int16), dxb.view(torch.int16))
    for a, b in zip(ua, ub):
        for key in ("w", "x", "dy"):
            assert torch.equal(a[key].view(torch.int16), b[key].view(torch.int16)), key
        for key in ("master", "m", "v", "dw"):
            assert torch.equal(a[key].view(torch.int32), b[key].view(torch.int32)), key


def test_zero3_step_units_equal_standalone_calls(z):
    """One unit's part of the step equals the standalone calls: the forward output equals
    fsdp_unit_forward's bf16 output, dX equals RNE of fsdp_unit_backward's fp32 dX, dW is
    identical, and the update equals zero_adam_step on that dW."""
    n, m = 4, 128
    (R0, K0), (R1, K1) = shapes = [(1024, 256), (512, 1024)]
    units = make_units(z, n, shapes, m, key=3)
    before = clone_units(units)
    run_step(z, units, m, 1, z.FSDP_BACKWARD_PREFETCH)
    b0 = before[0]
    sh0 = [s.contiguous() for s in b0["w"].view(n, R0 // n, K0).unbind(0)]
    yb = torch.empty(n * m, R0, dtype=torch.bfloat16, device=DEV)
    z.fsdp_unit_forward(sh0, b0["x"], None, Y_bf16=yb)
    assert torch.equal(yb.view(torch.int16), units[1]["x"].view(torch.int16))
    # unit 1's backward (W_1 [R1, K1] in 4 shards) gives unit 0's dY
    b1 = before[1]
    sh1 = [s.contiguous() for s in b1["w"].view(n, R1 // n, K1).unbind(0)]
    A = [units[1]["x"][q * m:(q + 1) * m].contiguous() for q in range(n)]
    dY = [b1["dy"][q * m:(q + 1) * m].contiguous() for q in range(n)]
    dX = [torch.empty(m, K1, device=DEV) for _ in range(n)]
    dW = torch.empty(R1, K1, device=DEV)
    ws = torch.empty(z.fsdp_unit_backward_workspace(n, R1, K1, m), dtype=torch.uint8, device=DEV)
    z.fsdp_unit_backward(sh1, A, dY, dX, dW, ws)
    z.zero_device_status()
    assert torch.equal(torch.cat(dX, 0).to(torch.bfloat16).view(torch.int16), units[0]["dy"].view(torch.int16))
    assert torch.equal(dW.view(torch.int32), units[1]["dw"].view(torch.int32))
    master, mm, vv = b1["master"].clone(), b1["m"].clone(), b1["v"].clone()
    w = torch.empty(R1 * K1, dtype=torch.bfloat16, device=DEV)
    z.zero_adam_step(b1["plan"], z.ZERO_ALL_RANKS, dW.view(-1), master, mm, vv, w, HP, 1)
    z.zero_device_status()
    assert torch.equal(master.view(torch.int32), units[1]["master"].view(torch.int32))
    assert torch.equal(w.view(torch.int16), units[1]["w"].view(-1).view(torch.int16))


@pytest.mark.parametrize("flags", [0, 2, 6, 8, 3])
def test_zero3_step_replays_from_a_cuda_graph(z, flags):
    """The step is plain stream work (host-encoded tensor maps by value, no allocation, the
    prefetch stream forked and joined through events), so it can be captured once in a CUDA
    graph: two replays leave every buffer bit for bit as two eager calls of the same step."""
    n, shapes, m = 4, [(512, 256), (1024, 512), (512, 1024)], 100
    a = make_units(z, n, shapes, m, key=17)
    b = clone_units(a)
    side = torch.cuda.Stream()
    ws = {k: torch.empty(z.fsdp_zero3_step_workspace(n, shapes, m, flags), dtype=torch.uint8, device=DEV)
          for k in ("a", "b", "c")}
    out = {k: (torch.empty(n * m, shapes[-1][0], dtype=torch.bfloat16, device=DEV),
               torch.empty(n * m, shapes[0][1], dtype=torch.bfloat16, device=DEV)) for k in ("a", "b", "c")}

    def run(units, k, stream):
        z.fsdp_zero3_step(units, m, HP, 1, y_out=out[k][0], dx_out=out[k][1], flags=flags, workspace=ws[k],
                          stream=stream, prefetch_stream=side)

    run(clone_units(a), "c", torch.cuda.current_stream())  # warm-up: events, kernel attributes
    torch.cuda.synchronize()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(g, stream=cap):
            run(b, "b", cap)
    for _ in range(2):
        run(a, "a", torch.cuda.current_stream())
        g.replay()
        torch.cuda.synchronize()
        z.zero_device_status()
        for x, y in zip(out["a"], out["b"]):
            assert torch.equal(x.view(torch.int16), y.view(torch.int16))
        for ua, ub in zip(a, b):
            for key in ("w", "x", "dy"):
                assert torch.equal(ua[key].view(torch.int16), ub[key].view(torch.int16)), key
            for key in ("master", "m", "v", "dw"):
                assert torch.equal(ua[key].view(torch.int32), ub[key].view(torch.int32)), key
