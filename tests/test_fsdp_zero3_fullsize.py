"""The ZeRO-3 step in the configuration the bench times: four Mistral-shaped FSDP units
(14336 x 4096, 4096 x 14336, twice), 8 ranks x 1024 tokens, both gathers fused into the GEMMs'
loads, each rank's Adam fused into the dW GEMMs' epilogues, the prefetch stream given; checked
on outputs the oracle computes one by one:
  - the same step with Adam as its own launch (FSDP_SEPARATE_OPTIMIZER, dW written) leaves
    every buffer bit for bit as the fused one, so what is checked below holds for both;
  - per unit, sampled entries of the forward output X_{i+1} = bf16(X_i W_i^T) and of
    dY_{i-1} = bf16(dY_i W_i) (W_i the weights before the step) within the rounded fp32 bound
    of their float64 dot products on the GPU's own inputs;
  - sampled dW entries within the fp32 bound of (1/N) sum over all 8192 tokens;
  - Adam on the GPU's dW at sampled parameters of every rank's shard, bit for bit (master,
    m, v and the new bf16 shard), with the oracle's update.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle.zero_oracle as O
import synth
from _util import bits16, f32
from test_fsdp_zero3 import HP, check_bf16_product, clone_units, z  # noqa: F401  (z: fixture)

pytestmark = pytest.mark.gpu
DEV = "cuda"
SHAPES = [(14336, 4096), (4096, 14336), (14336, 4096), (4096, 14336)]
N, M = 8, 1024


def mistral_units(z):
    nm = N * M
    units = []
    for i, (R, K) in enumerate(SHAPES):
        w = torch.cat(synth.weight_shards(R, K, N, device=DEV, seed_key=70 + i), 0).contiguous()
        units.append({"plan": z.zero_plan(R * K, N, "zero3", 50 << 20), "w": w, "master": w.float().reshape(-1),
                      "m": torch.zeros(R * K, device=DEV), "v": torch.zeros(R * K, device=DEV),
                      "x": torch.zeros(nm, K, dtype=torch.bfloat16, device=DEV),
                      "dy": torch.zeros(nm, R, dtype=torch.bfloat16, device=DEV)})
    units[0]["x"].copy_(synth.activations(nm, SHAPES[0][1], device=DEV, seed_key=77))
    units[-1]["dy"].copy_(synth.upstream_grad(nm, SHAPES[-1][0], device=DEV, seed_key=77))
    return units


def rows_of(t, idx):
    return bits16(t[torch.from_numpy(idx).to(DEV)])


def test_zero3_step_mistral_units_sampled(z):
    nm = N * M
    a = mistral_units(z)
    w_old = [bits16(u["w"]) for u in a]  # the weights every GEMM of the step reads
    b = clone_units(a)
    for u in b:
        u["dw"] = torch.full(tuple(u["w"].shape), float("nan"), device=DEV)
    out = {}
    for name, units, flags, side in (("fused", a, 0, torch.cuda.Stream()),
                                     ("separate", b, z.FSDP_SEPARATE_OPTIMIZER, None)):
        y = torch.full((nm, SHAPES[-1][0]), float("nan"), dtype=torch.bfloat16, device=DEV)
        dx = torch.full((nm, SHAPES[0][1]), float("nan"), dtype=torch.bfloat16, device=DEV)
        z.fsdp_zero3_step(units, M, HP, 1, y_out=y, dx_out=dx, flags=flags, prefetch_stream=side)
        z.zero_device_status()
        out[name] = (y, dx)
    for ta, tb in zip(out["fused"], out["separate"]):
        assert torch.equal(ta.view(torch.int16), tb.view(torch.int16))
    for ua, ub in zip(a, b):
        for key in ("w", "x", "dy"):
            assert torch.equal(ua[key].view(torch.int16), ub[key].view(torch.int16)), key
        for key in ("master", "m", "v"):
            assert torch.equal(ua[key].view(torch.int32), ub[key].view(torch.int32)), key
    del a
    y_out, dx_out = out["separate"]
    rng = np.random.default_rng(12)
    hp = O.AdamHyper(**HP)
    L = len(SHAPES)
    for i, (R, K) in enumerate(SHAPES):
        u = b[i]
        w64 = O.bf16_to_f32(w_old[i]).astype(np.float64)
        # forward: X_{i+1}[r, c] over K, with the GPU's X_i
        r_s, c_s = rng.integers(0, nm, 512), rng.integers(0, R, 512)
        xr = O.bf16_to_f32(rows_of(u["x"], r_s)).astype(np.float64)
        exact = np.einsum("sk,sk->s", xr, w64[c_s])
        bound = (K + 1) * 2.0 ** -23 * np.einsum("sk,sk->s", np.abs(xr), np.abs(w64[c_s]))
        fw = b[i + 1]["x"] if i + 1 < L else y_out
        got = bits16(fw[torch.from_numpy(r_s).to(DEV), torch.from_numpy(c_s).to(DEV)])
        check_bf16_product(got, exact, bound, f"forward of unit {i}")
        # backward: dY_{i-1}[r, c] over R, with the GPU's dY_i and the old W_i
        r_s, c_s = rng.integers(0, nm, 512), rng.integers(0, K, 512)
        dyr = O.bf16_to_f32(rows_of(u["dy"], r_s)).astype(np.float64)
        wc = w64[:, c_s].T
        exact = np.einsum("sj,sj->s", dyr, wc)
        bound = (R + 1) * 2.0 ** -23 * np.einsum("sj,sj->s", np.abs(dyr), np.abs(wc))
        bw = b[i - 1]["dy"] if i > 0 else dx_out
        got = bits16(bw[torch.from_numpy(r_s).to(DEV), torch.from_numpy(c_s).to(DEV)])
        check_bf16_product(got, exact, bound, f"dX of unit {i}")
        # dW[row, col] = (1/N) sum over every rank's tokens, within the fp32 bound
        rr, cc = rng.integers(0, R, 512), rng.integers(0, K, 512)
        dyc = O.bf16_to_f32(bits16(u["dy"][:, torch.from_numpy(rr).to(DEV)].t().contiguous())).astype(np.float64)
        xc = O.bf16_to_f32(bits16(u["x"][:, torch.from_numpy(cc).to(DEV)].t().contiguous())).astype(np.float64)
        exact = np.einsum("st,st->s", dyc, xc) / N
        bound = (nm + 1) * 2.0 ** -23 * np.einsum("st,st->s", np.abs(dyc), np.abs(xc)) / N + 2.0 ** -24 * np.abs(exact)
        dw = f32(u["dw"][torch.from_numpy(rr).to(DEV), torch.from_numpy(cc).to(DEV)]).astype(np.float64)
        assert np.all(np.abs(dw - exact) <= bound), f"dW of unit {i}"
        # Adam on the GPU's dW at 512 parameters of every rank's shard, bit for bit
        S = R * K // N
        idx = np.concatenate([r * S + rng.integers(0, S, 512) for r in range(N)] + [np.array([0, S - 1, R * K - 1])])
        ti = torch.from_numpy(idx).to(DEV)
        g = f32(u["dw"].reshape(-1)[ti])
        master0 = O.bf16_to_f32(w_old[i].reshape(-1)[idx])
        zeros = np.zeros(idx.size, dtype=np.float32)
        w_new, m_new, v_new = O.adam_update(master0, zeros, zeros, g, hp, 1)
        assert np.array_equal(f32(u["master"][ti]).view(np.uint32), w_new.view(np.uint32)), f"master of unit {i}"
        assert np.array_equal(f32(u["m"][ti]).view(np.uint32), m_new.view(np.uint32)), f"m of unit {i}"
        assert np.array_equal(f32(u["v"][ti]).view(np.uint32), v_new.view(np.uint32)), f"v of unit {i}"
        assert np.array_equal(bits16(u["w"].reshape(-1)[ti]), O.f32_to_bf16(w_new)), f"bf16 shard of unit {i}"
