"""GPU parity of one ZeRO-3 training step over a stack of Mistral-style FSDP MLP units
(fsdp_zero3_mlp_step): H = silu(X W_gate^T) * (X W_up^T), Y = H W_down^T, each weight in N
row shards with its own ZeRO-3 state.

Every buffer the step writes is checked against the oracle, unit by unit, on the inputs the
GPU gave that unit (each an exact bf16 or fp32 value). A bf16 product output comes from an
fp32 sum within B = (K + 1) 2^-23 sum|a w| of the exact product, so it must lie between
RNE(exact - B) and RNE(exact + B):
  - forward: G | U against the oracle's float64 projections; H = bf16(silu(G) U) from the
    fp32 accumulators under the bound of the MLP forward tests; the next unit's X = bf16(H
    W_down^T) from the GPU's H;
  - backward: dH = bf16(dY W_down) and the previous unit's dY = bf16([dG | dU] [W_gate;
    W_up]) with the weights from before the step; dG | dU against the oracle's
    silu_gate_backward on the GPU's bf16 dH, G, U (fp32 with expf: within 10 and 8 units
    of 2^-24 of the exact terms, then one bf16 rounding); dW_down and dW_gate | dW_up under
    the fp32 bound, each rank's rows against the oracle's reduce-scatter;
  - each rank's Adam on its W_gate, W_up and W_down shards bit for bit from the GPU's dW;
  - two steps in a row: the second forward reads the shards the first one wrote.
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
U = 2.0 ** -24


@pytest.fixture(scope="module")
def z():
    import __graft_entry__ as g
    g.build()
    import fsdp_sharded_optimizer_zero_gb300 as z
    return z


def weight(z, rows, cols, n, key):
    w = torch.cat(synth.weight_shards(rows, cols, n, device=DEV, seed_key=key), 0).contiguous()
    return {"plan": z.zero_plan(rows * cols, n, "zero3", 1 << 20), "w": w, "master": w.float().reshape(-1).clone(),
            "m": torch.zeros(rows * cols, device=DEV), "v": torch.zeros(rows * cols, device=DEV)}


def make_units(z, n, d, f, n_units, m, key):
    nm = n * m
    bf = dict(dtype=torch.bfloat16, device=DEV)
    units = []
    for i in range(n_units):
        units.append({"d_model": d, "d_ff": f, "gate": weight(z, f, d, n, 100 * key + 10 * i + 1),
                      "up": weight(z, f, d, n, 100 * key + 10 * i + 2), "down": weight(z, d, f, n, 100 * key + 10 * i + 3),
                      "x": torch.zeros(nm, d, **bf), "gu": torch.full((nm, 2 * f), float("nan"), **bf),
                      "h": torch.full((nm, f), float("nan"), **bf), "dy": torch.zeros(nm, d, **bf),
                      "dh": torch.full((nm, f), float("nan"), **bf), "dgu": torch.full((nm, 2 * f), float("nan"), **bf),
                      "dw_gu": torch.full((2 * f, d), float("nan"), device=DEV),
                      "dw_down": torch.full((d, f), float("nan"), device=DEV)})
    units[0]["x"].copy_(synth.activations(nm, d, device=DEV, seed_key=key))
    units[-1]["dy"].copy_(synth.upstream_grad(nm, d, device=DEV, seed_key=key))
    return units


def run_step(z, units, m, step, flags=0):
    n = units[0]["gate"]["plan"].n_ranks
    nm = n * m
    shapes = [(u["d_model"], u["d_ff"]) for u in units]
    ws = torch.empty(z.fsdp_zero3_mlp_step_workspace(n, shapes, m), dtype=torch.uint8, device=DEV)
    y = torch.full((nm, shapes[-1][0]), float("nan"), dtype=torch.bfloat16, device=DEV)
    dx = torch.full((nm, shapes[0][0]), float("nan"), dtype=torch.bfloat16, device=DEV)
    z.fsdp_zero3_mlp_step(units, m, HP, step, y_out=y, dx_out=dx, workspace=ws, flags=flags)
    z.zero_device_status()
    return y, dx


def snapshot(units):
    out = []
    for u in units:
        d = {k: bits16(u[k]) for k in ("x", "dy")}
        for w in ("gate", "up", "down"):
            d[w] = {"w": bits16(u[w]["w"]), "master": f32(u[w]["master"]).copy(), "m": f32(u[w]["m"]).copy(),
                    "v": f32(u[w]["v"]).copy()}
        out.append(d)
    return out


def f64(bits):
    return O.bf16_to_f32(bits).astype(np.float64)


def check_bf16_product(out_bits, exact, bound, what):
    """out = RNE(s) for an fp32 s within `bound` of `exact`: RNE(lo) <= out <= RNE(hi)."""
    lo = np.nextafter((exact - bound).astype(np.float32), np.float32(-np.inf))
    hi = np.nextafter((exact + bound).astype(np.float32), np.float32(np.inf))
    out = O.bf16_to_f32(out_bits)
    ok = (O.bf16_to_f32(O.f32_to_bf16(lo)) <= out) & (out <= O.bf16_to_f32(O.f32_to_bf16(hi)))
    assert ok.all(), f"{what}: {(~ok).sum()} of {ok.size} bf16 outputs outside the rounded bound"


def check_gemm_bf16(out_bits, a64, w64, what):
    """out = bf16(A W^T) within the fp32 bound."""
    exact = a64 @ w64.T
    bound = (a64.shape[1] + 1) * 2.0 ** -23 * (np.abs(a64) @ np.abs(w64).T)
    check_bf16_product(out_bits, exact, bound, what)


def check_dw(dw_gpu, dy64, x64, n, m, what):
    """dW = (1/N) sum_q dY_q^T X_q under the fp32 bound, and each rank's rows against the
    oracle's reduce-scatter of the per-rank fp32 products."""
    R, K = dy64.shape[1], x64.shape[1]
    exact, bnd, per_rank = np.zeros((R, K)), np.zeros((R, K)), []
    for q in range(n):
        rows = slice(q * m, (q + 1) * m)
        p = dy64[rows].T @ x64[rows]
        per_rank.append(p.astype(np.float32))
        exact += p
        bnd += np.abs(dy64[rows]).T @ np.abs(x64[rows])
    exact /= n
    bound = (n * m + 1) * 2.0 ** -23 * bnd / n + 2.0 ** -24 * np.abs(exact)
    assert np.all(np.abs(dw_gpu - exact) <= bound), what
    rs = R // n
    for r in range(n):
        ref = O.reduce_rows(per_rank, n, r).astype(np.float64)
        assert np.all(np.abs(dw_gpu[r * rs:(r + 1) * rs] - ref) <= 2 * bound[r * rs:(r + 1) * rs] + 1e-30), \
            f"{what}: rank {r}'s reduce-scattered rows"


def check_adam(w_state, before, g, n, t, what):
    hp = O.AdamHyper(**HP)
    S = g.size // n
    for r in range(n):
        sl = slice(r * S, (r + 1) * S)
        w_new, m_new, v_new = O.adam_update(before["master"][sl], before["m"][sl], before["v"][sl], g[sl], hp, t)
        assert_f32_identical(f32(w_state["master"])[sl], w_new, f"{what} master, rank {r}")
        assert_f32_identical(f32(w_state["m"])[sl], m_new, f"{what} m, rank {r}")
        assert_f32_identical(f32(w_state["v"])[sl], v_new, f"{what} v, rank {r}")
        assert_bf16_identical(bits16(w_state["w"]).reshape(-1)[sl], O.f32_to_bf16(w_new), f"{what} shard, rank {r}")


def h_bound(g64, u64, bg, bu, h_gpu):
    """|H_gpu - H_exact| for H = silu(G) U computed from fp32 G, U within bg, bu of exact:
    |silu'| <= 1.1, a few fp32 roundings in silu and the product, one bf16 rounding."""
    sil = np.abs(O.silu(g64))
    return (1.1 * bg * np.abs(u64) + sil * bu + 1.1 * bg * bu + 16 * U * sil * np.abs(u64)
            + 2.0 ** -8 * 1.01 * np.abs(h_gpu) + 1e-38)


def check_step(n, m, before, units, y, dx, t):
    L = len(units)
    for i, u in enumerate(units):
        b = before[i]
        f = u["d_ff"]
        wg, wu, wd = f64(b["gate"]["w"]), f64(b["up"]["w"]), f64(b["down"]["w"])
        x64 = f64(bits16(u["x"]) if i > 0 else b["x"])
        # forward: G | U, H, the unit's output
        gu = bits16(u["gu"])
        ag = np.abs(x64)
        g_ex, u_ex = x64 @ wg.T, x64 @ wu.T
        bg = (x64.shape[1] + 1) * 2.0 ** -23 * (ag @ np.abs(wg).T)
        bu = (x64.shape[1] + 1) * 2.0 ** -23 * (ag @ np.abs(wu).T)
        check_bf16_product(gu[:, :f], g_ex, bg, f"G of unit {i}")
        check_bf16_product(gu[:, f:], u_ex, bu, f"U of unit {i}")
        h = bits16(u["h"])
        h_ex = O.silu(g_ex) * u_ex
        assert np.all(np.abs(f64(h) - h_ex) <= h_bound(g_ex, u_ex, bg, bu, f64(h))), f"H of unit {i}"
        out = bits16(units[i + 1]["x"]) if i + 1 < L else bits16(y)
        check_gemm_bf16(out, f64(h), wd, f"output of unit {i}")
        # backward: dH, dW_down, W_down's Adam
        dy64 = f64(bits16(u["dy"]) if i + 1 < L else b["dy"])
        check_gemm_bf16(bits16(u["dh"]), dy64, wd.T, f"dH of unit {i}")
        dw_down = f32(u["dw_down"]).astype(np.float64)
        check_dw(dw_down, dy64, f64(h), n, m, f"dW_down of unit {i}")
        check_adam(u["down"], b["down"], f32(u["dw_down"]).reshape(-1), n, t, f"W_down of unit {i}")
        # the SiLU-gate backward on the GPU's dH, G, U
        dh_b = bits16(u["dh"])
        dg_ex, du_ex = O.silu_gate_backward(dh_b, gu[:, :f], gu[:, f:])
        gg, uu, dd = f64(gu[:, :f]), f64(gu[:, f:]), f64(dh_b)
        with np.errstate(over="ignore"):
            s = 1.0 / (1.0 + np.exp(-gg))
        b_dg = 10 * U * np.abs(dd * uu) * s * (1.0 + np.abs(gg) * (1.0 - s)) + 1e-38
        b_du = 8 * U * np.abs(dd * gg * s) + 1e-38
        dgu = bits16(u["dgu"])
        check_bf16_product(dgu[:, :f], dg_ex, b_dg, f"dG of unit {i}")
        check_bf16_product(dgu[:, f:], du_ex, b_du, f"dU of unit {i}")
        # dX over both projections, dW_gate | dW_up, their Adam
        dgu64 = f64(dgu)
        dx_got = bits16(units[i - 1]["dy"]) if i > 0 else bits16(dx)
        check_gemm_bf16(dx_got, dgu64, np.concatenate([wg, wu], 0).T, f"dX of unit {i}")
        dw_gu = f32(u["dw_gu"])
        check_dw(dw_gu.astype(np.float64), dgu64, x64, n, m, f"dW_gate | dW_up of unit {i}")
        check_adam(u["gate"], b["gate"], dw_gu[:f].reshape(-1), n, t, f"W_gate of unit {i}")
        check_adam(u["up"], b["up"], dw_gu[f:].reshape(-1), n, t, f"W_up of unit {i}")


# d_ff / N a multiple of 128 (the gate-up kernel's shard tiles), d_model / N of 128 (W_down's)
# (12, 1536, 1536, 1, 16): past 8 ranks the 2N shards of [W_gate; W_up] exceed the GEMM's
# 16 pieces, so the dX GEMM reads them gathered into the workspace
@pytest.mark.parametrize("n,d,f,n_units,m", [(4, 512, 512, 2, 100), (2, 256, 1024, 3, 64), (8, 1024, 1024, 1, 48),
                                             (12, 1536, 1536, 1, 16)])
def test_zero3_mlp_step_every_buffer_vs_oracle(z, n, d, f, n_units, m):
    units = make_units(z, n, d, f, n_units, m, key=n + n_units)
    for t in (1, 2):
        before = snapshot(units)
        y, dx = run_step(z, units, m, t)
        check_step(n, m, before, units, y, dx, t)


def clone(units):
    out = []
    for u in units:
        c = {k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in u.items()}
        for w in ("gate", "up", "down"):
            c[w] = {k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in u[w].items()}
        out.append(c)
    return out


def test_zero3_mlp_optimizer_fused_or_separate_same_bits(z):
    """Adam fused into the dW GEMMs' epilogues (the default, here once with dW written and
    once without) and Adam as its own launches (FSDP_SEPARATE_OPTIMIZER) leave every
    buffer bit for bit the same, over two steps."""
    n, d, f, m = 4, 512, 512, 100
    base = make_units(z, n, d, f, 2, m, key=21)
    runs = {"fused": clone(base), "fused_no_dw": clone(base), "separate": clone(base)}
    for u in runs["fused_no_dw"]:
        u.pop("dw_gu")
        u.pop("dw_down")
    outs = {}
    for name, units in runs.items():
        for t in (1, 2):
            outs[name] = run_step(z, units, m, t, flags=z.FSDP_SEPARATE_OPTIMIZER if name == "separate" else 0)
    ref = runs["separate"]
    for name in ("fused", "fused_no_dw"):
        for a, b in zip(outs[name], outs["separate"]):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), name
        for ua, ub in zip(runs[name], ref):
            for key in ("x", "gu", "h", "dy", "dh", "dgu"):
                assert torch.equal(ua[key].view(torch.int16), ub[key].view(torch.int16)), (name, key)
            for w in ("gate", "up", "down"):
                assert torch.equal(ua[w]["w"].view(torch.int16), ub[w]["w"].view(torch.int16)), (name, w)
                for key in ("master", "m", "v"):
                    assert torch.equal(ua[w][key].view(torch.int32), ub[w][key].view(torch.int32)), (name, w, key)
    for ua, ub in zip(runs["fused"], ref):
        for key in ("dw_gu", "dw_down"):
            assert torch.equal(ua[key].view(torch.int32), ub[key].view(torch.int32)), key


@pytest.mark.parametrize("flags", [0, 8])
def test_zero3_mlp_step_same_bits_on_both_gemm_kernels(z, flags):
    """The MLP step on the one-CTA GEMM kernel (zero_set_gemm_kernel(1)) leaves every buffer
    bit for bit as on the default CTA-pair kernel, over two steps, Adam fused or separate."""
    n, d, f, m = 2, 512, 512, 72
    base = make_units(z, n, d, f, 2, m, key=31)
    out = []
    try:
        for kernel in (0, 1):
            z.zero_set_gemm_kernel(kernel)
            units = clone(base)
            for t in (1, 2):
                y, dx = run_step(z, units, m, t, flags)
            out.append((units, y, dx))
    finally:
        z.zero_set_gemm_kernel(0)
    (ua, ya, dxa), (ub, yb, dxb) = out
    assert torch.equal(ya.view(torch.int16), yb.view(torch.int16))
    assert torch.equal(dxa.view(torch.int16), dxb.view(torch.int16))
    for a, b in zip(ua, ub):
        for key in ("x", "gu", "h", "dy", "dh", "dgu"):
            assert torch.equal(a[key].view(torch.int16), b[key].view(torch.int16)), key
        for key in ("dw_gu", "dw_down"):
            assert torch.equal(a[key].view(torch.int32), b[key].view(torch.int32)), key
        for w in ("gate", "up", "down"):
            assert torch.equal(a[w]["w"].view(torch.int16), b[w]["w"].view(torch.int16)), w
            for key in ("master", "m", "v"):
                assert torch.equal(a[w][key].view(torch.int32), b[w][key].view(torch.int32)), (w, key)


def test_zero3_mlp_forward_equals_the_mlp_forward_call(z):
    """The step's forward equals fsdp_mlp_forward on the same shards: H bit for bit, and
    the unit's bf16 output equals RNE of that call's fp32 Y."""
    n, d, f, m = 4, 512, 512, 64
    units = make_units(z, n, d, f, 1, m, key=9)
    sh = {k: [s.contiguous() for s in units[0][k]["w"].view(n, -1, units[0][k]["w"].shape[1]).unbind(0)]
          for k in ("gate", "up", "down")}
    x = units[0]["x"].clone()
    H = torch.empty(n * m, f, dtype=torch.bfloat16, device=DEV)
    Y = torch.empty(n * m, d, device=DEV)
    z.fsdp_mlp_forward(sh["gate"], sh["up"], sh["down"], x, H, Y)
    y, _ = run_step(z, units, m, 1)
    assert torch.equal(units[0]["h"].view(torch.int16), H.view(torch.int16))
    assert torch.equal(y.view(torch.int16), Y.to(torch.bfloat16).view(torch.int16))


def test_zero3_mlp_step_rejects_bad_shapes(z):
    with pytest.raises(z.ZeroError) as e:
        z.fsdp_zero3_mlp_step_workspace(4, [(512, 384)], 64)  # d_ff / N = 96
    assert e.value.code == -1
    with pytest.raises(z.ZeroError):
        z.fsdp_zero3_mlp_step_workspace(4, [(512, 512), (256, 512)], 64)  # d_model changes


@pytest.mark.parametrize("flags", [0, 8])
def test_zero3_mlp_step_replays_from_a_cuda_graph(z, flags):
    """Captured once in a CUDA graph, two replays of the MLP step leave every buffer bit for
    bit as two eager calls of the same step."""
    n, d, f, m = 2, 256, 512, 64
    a = make_units(z, n, d, f, 2, m, key=27)
    b = clone(a)
    shapes = [(d, f)] * 2
    ws = {k: torch.empty(z.fsdp_zero3_mlp_step_workspace(n, shapes, m), dtype=torch.uint8, device=DEV)
          for k in ("a", "b", "c")}
    out = {k: (torch.empty(n * m, d, dtype=torch.bfloat16, device=DEV),
               torch.empty(n * m, d, dtype=torch.bfloat16, device=DEV)) for k in ("a", "b", "c")}

    def run(units, k, stream):
        z.fsdp_zero3_mlp_step(units, m, HP, 1, y_out=out[k][0], dx_out=out[k][1], workspace=ws[k], stream=stream,
                              flags=flags)

    run(clone(a), "c", torch.cuda.current_stream())  # warm-up: kernel attributes
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
            for key in ("x", "gu", "h", "dy", "dh", "dgu"):
                assert torch.equal(ua[key].view(torch.int16), ub[key].view(torch.int16)), key
            for key in ("dw_gu", "dw_down"):
                assert torch.equal(ua[key].view(torch.int32), ub[key].view(torch.int32)), key
            for w in ("gate", "up", "down"):
                assert torch.equal(ua[w]["w"].view(torch.int16), ub[w]["w"].view(torch.int16)), w
                for key in ("master", "m", "v"):
                    assert torch.equal(ua[w][key].view(torch.int32), ub[w][key].view(torch.int32)), (w, key)
