"""The ZeRO-3 MLP step in the configuration the bench times: two Mistral-7B MLP units
(d_model 4096, d_ff 14336; W_gate, W_up, W_down in 8 row shards each), 8 ranks x 1024
tokens, every gather fused into the GEMMs' loads, each rank's Adam fused into the dW GEMMs'
epilogues; checked on outputs the oracle computes one by one, with the bounds of the
small-shape tests (tests/test_fsdp_zero3_mlp.py):
  - the same step with Adam as its own launches (FSDP_SEPARATE_OPTIMIZER, dW written) leaves
    every buffer bit for bit as the fused one;
  - per unit, on sampled entries and the GPU's own inputs: G | U, H = silu(G) U, the unit's
    output, dH, dG | dU (the oracle's SiLU-gate backward), dX over both projections,
    dW_down and dW_gate | dW_up, and each rank's Adam on the three weights bit for bit.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle.zero_oracle as O
from _util import bits16, f32
from test_fsdp_zero3_mlp import (HP, check_bf16_product, clone, f64, h_bound, make_units,  # noqa: F401
                                 U, z)

pytestmark = pytest.mark.gpu
DEV = "cuda"
N, M, D, F = 8, 1024, 4096, 14336


def at(t, r, c):
    return t[torch.from_numpy(r).to(DEV), torch.from_numpy(c).to(DEV)]


def rows(t, r):
    return t[torch.from_numpy(r).to(DEV)]


def cols(t, c):
    return t[:, torch.from_numpy(c).to(DEV)].t().contiguous()


def check_dw_sampled(dw_gpu, a_cols, b_cols, what):
    """dW[row, col] = (1/N) sum over every token of A[t, row] B[t, col] (columns given as
    float64 [samples, tokens]) under the fp32 bound."""
    exact = np.einsum("st,st->s", a_cols, b_cols) / N
    bound = (N * M + 1) * 2.0 ** -23 * np.einsum("st,st->s", np.abs(a_cols), np.abs(b_cols)) / N \
        + 2.0 ** -24 * np.abs(exact)
    assert np.all(np.abs(dw_gpu - exact) <= bound), what


def check_adam_sampled(w_state, w_old_bits, dw_flat, idx, what):
    ti = torch.from_numpy(idx).to(DEV)
    g = f32(dw_flat[ti])
    zeros = np.zeros(idx.size, dtype=np.float32)
    w_new, m_new, v_new = O.adam_update(O.bf16_to_f32(w_old_bits.reshape(-1)[idx]), zeros, zeros, g,
                                        O.AdamHyper(**HP), 1)
    assert np.array_equal(f32(w_state["master"][ti]).view(np.uint32), w_new.view(np.uint32)), f"{what} master"
    assert np.array_equal(f32(w_state["m"][ti]).view(np.uint32), m_new.view(np.uint32)), f"{what} m"
    assert np.array_equal(f32(w_state["v"][ti]).view(np.uint32), v_new.view(np.uint32)), f"{what} v"
    assert np.array_equal(bits16(w_state["w"].reshape(-1)[ti]), O.f32_to_bf16(w_new)), f"{what} shard"


def shard_samples(rng, rows_, cols_, k=256):
    S = rows_ * cols_ // N
    return np.concatenate([r * S + rng.integers(0, S, k) for r in range(N)] + [np.array([0, S - 1, rows_ * cols_ - 1])])


def test_zero3_mlp_step_mistral_units_sampled(z):
    nm = N * M
    a = make_units(z, N, D, F, 2, M, key=41)
    for u in a:
        u.pop("dw_gu")
        u.pop("dw_down")
    old = [{w: bits16(u[w]["w"]) for w in ("gate", "up", "down")} for u in a]
    b = clone(a)
    for u in b:
        u["dw_gu"] = torch.full((2 * F, D), float("nan"), device=DEV)
        u["dw_down"] = torch.full((D, F), float("nan"), device=DEV)
    res = {}
    for name, units, flags in (("fused", a, 0), ("separate", b, z.FSDP_SEPARATE_OPTIMIZER)):
        y = torch.full((nm, D), float("nan"), dtype=torch.bfloat16, device=DEV)
        dx = torch.full((nm, D), float("nan"), dtype=torch.bfloat16, device=DEV)
        z.fsdp_zero3_mlp_step(units, M, HP, 1, y_out=y, dx_out=dx, flags=flags)
        z.zero_device_status()
        res[name] = (y, dx)
    for ta, tb in zip(res["fused"], res["separate"]):
        assert torch.equal(ta.view(torch.int16), tb.view(torch.int16))
    for ua, ub in zip(a, b):
        for key in ("x", "gu", "h", "dy", "dh", "dgu"):
            assert torch.equal(ua[key].view(torch.int16), ub[key].view(torch.int16)), key
        for w in ("gate", "up", "down"):
            assert torch.equal(ua[w]["w"].view(torch.int16), ub[w]["w"].view(torch.int16)), w
            for key in ("master", "m", "v"):
                assert torch.equal(ua[w][key].view(torch.int32), ub[w][key].view(torch.int32)), (w, key)
    del a
    y_out, dx_out = res["separate"]
    rng = np.random.default_rng(21)
    for i, u in enumerate(b):
        wg, wu, wd = (O.bf16_to_f32(old[i][w]).astype(np.float64) for w in ("gate", "up", "down"))
        # forward: G | U and H at sampled (token, d_ff column)
        r, c = rng.integers(0, nm, 512), rng.integers(0, F, 512)
        xr = f64(bits16(rows(u["x"], r)))
        g_ex, u_ex = np.einsum("sk,sk->s", xr, wg[c]), np.einsum("sk,sk->s", xr, wu[c])
        bg = (D + 1) * 2.0 ** -23 * np.einsum("sk,sk->s", np.abs(xr), np.abs(wg[c]))
        bu = (D + 1) * 2.0 ** -23 * np.einsum("sk,sk->s", np.abs(xr), np.abs(wu[c]))
        check_bf16_product(bits16(at(u["gu"], r, c)), g_ex, bg, f"G of unit {i}")
        check_bf16_product(bits16(at(u["gu"], r, c + F)), u_ex, bu, f"U of unit {i}")
        h_got = f64(bits16(at(u["h"], r, c)))
        h_ex = O.silu(g_ex) * u_ex
        assert np.all(np.abs(h_got - h_ex) <= h_bound(g_ex, u_ex, bg, bu, h_got)), f"H of unit {i}"
        # the unit's output from the GPU's H
        r, c = rng.integers(0, nm, 512), rng.integers(0, D, 512)
        hr = f64(bits16(rows(u["h"], r)))
        exact = np.einsum("sj,sj->s", hr, wd[c])
        bound = (F + 1) * 2.0 ** -23 * np.einsum("sj,sj->s", np.abs(hr), np.abs(wd[c]))
        out = b[i + 1]["x"] if i + 1 < len(b) else y_out
        check_bf16_product(bits16(at(out, r, c)), exact, bound, f"output of unit {i}")
        # dH = bf16(dY W_down)
        r, c = rng.integers(0, nm, 512), rng.integers(0, F, 512)
        dyr = f64(bits16(rows(u["dy"], r)))
        wdc = wd[:, c].T
        exact = np.einsum("sj,sj->s", dyr, wdc)
        bound = (D + 1) * 2.0 ** -23 * np.einsum("sj,sj->s", np.abs(dyr), np.abs(wdc))
        check_bf16_product(bits16(at(u["dh"], r, c)), exact, bound, f"dH of unit {i}")
        # dG | dU by the oracle's SiLU-gate backward on the GPU's dH, G, U
        gb, ub_, dhb = bits16(at(u["gu"], r, c)), bits16(at(u["gu"], r, c + F)), bits16(at(u["dh"], r, c))
        dg_ex, du_ex = O.silu_gate_backward(dhb, gb, ub_)
        gg, uu, dd = f64(gb), f64(ub_), f64(dhb)
        with np.errstate(over="ignore"):
            s = 1.0 / (1.0 + np.exp(-gg))
        b_dg = 10 * U * np.abs(dd * uu) * s * (1.0 + np.abs(gg) * (1.0 - s)) + 1e-38
        b_du = 8 * U * np.abs(dd * gg * s) + 1e-38
        check_bf16_product(bits16(at(u["dgu"], r, c)), dg_ex, b_dg, f"dG of unit {i}")
        check_bf16_product(bits16(at(u["dgu"], r, c + F)), du_ex, b_du, f"dU of unit {i}")
        # dX over both projections' concatenated K, from the GPU's dG | dU
        r, c = rng.integers(0, nm, 512), rng.integers(0, D, 512)
        dgur = f64(bits16(rows(u["dgu"], r)))
        wgu_c = np.concatenate([wg, wu], 0)[:, c].T
        exact = np.einsum("sj,sj->s", dgur, wgu_c)
        bound = (2 * F + 1) * 2.0 ** -23 * np.einsum("sj,sj->s", np.abs(dgur), np.abs(wgu_c))
        dxo = b[i - 1]["dy"] if i > 0 else dx_out
        check_bf16_product(bits16(at(dxo, r, c)), exact, bound, f"dX of unit {i}")
        # dW_down [D, F] = (1/N) dY^T H and dW_gate | dW_up [2F, D] = (1/N) [dG | dU]^T X
        rr, cc = rng.integers(0, D, 512), rng.integers(0, F, 512)
        check_dw_sampled(f32(at(u["dw_down"], rr, cc)).astype(np.float64), f64(bits16(cols(u["dy"], rr))),
                         f64(bits16(cols(u["h"], cc))), f"dW_down of unit {i}")
        rr, cc = rng.integers(0, 2 * F, 512), rng.integers(0, D, 512)
        check_dw_sampled(f32(at(u["dw_gu"], rr, cc)).astype(np.float64), f64(bits16(cols(u["dgu"], rr))),
                         f64(bits16(cols(u["x"], cc))), f"dW_gate | dW_up of unit {i}")
        # each rank's Adam on its shards of the three weights, from the GPU's dW
        check_adam_sampled(u["down"], old[i]["down"], u["dw_down"].reshape(-1), shard_samples(rng, D, F),
                           f"W_down of unit {i}")
        check_adam_sampled(u["gate"], old[i]["gate"], u["dw_gu"][:F].reshape(-1), shard_samples(rng, F, D),
                           f"W_gate of unit {i}")
        check_adam_sampled(u["up"], old[i]["up"], u["dw_gu"][F:].reshape(-1), shard_samples(rng, F, D),
                           f"W_up of unit {i}")
