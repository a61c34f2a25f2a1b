"""Seeded synthetic inputs for the data-parallel optimizer step and the FSDP unit.

This module is shared by both sides of every parity check (the CPU oracle and the CUDA
library). It holds no arithmetic of the method itself: it only describes workload shapes
and draws seeded random tensors. The same bytes always feed both sides; neither side
regenerates data (host and device random streams differ).

Distributions (the reading of "N(0, s)" is: s is the standard deviation):
  * fp32 master parameters   ~ N(0, 0.02)
  * bf16 per-rank gradients  ~ N(0, 1e-3), a fresh draw per (rank, step)
  * bf16 FSDP weights        ~ N(0, 0.02)
  * bf16 FSDP activations    ~ N(0, 1)
Padding entries [psi, psi_padded) are zero in every buffer.

Seeds: a 64-bit SplitMix64 chain derives one torch.Generator seed per
(base seed, tensor id, rank, step), so every tensor is reproducible on its own.
"""
from __future__ import annotations

import torch

BASE_SEED = 20261202

# tensor ids used in seed derivation
TID_MASTER = 1
TID_GRAD = 2
TID_WEIGHT = 3
TID_ACT = 4
TID_STATE_M = 5
TID_STATE_V = 6
TID_DY = 7

_MASK64 = (1 << 64) - 1


def splitmix64(x: int) -> int:
    """One SplitMix64 output for state x (Steele, Lea, Flood 2014)."""
    z = (x + 0x9E3779B97F4A7C15) & _MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def derive_seed(*keys: int, base: int = BASE_SEED) -> int:
    s = splitmix64(base & _MASK64)
    for k in keys:
        s = splitmix64((s ^ (k & _MASK64)) & _MASK64)
    return s & ((1 << 63) - 1)


def _gen(device, *keys) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(derive_seed(*keys))
    return g


# ----------------------------------------------------------------------------------------
# workload shapes
# ----------------------------------------------------------------------------------------

def gpt2_small_tensors():
    """GPT-2-small parameter list as given by the workload: wte, wpe, 12 blocks of
    (qkv, proj, fc, fc2, ln_1.{w,b}, ln_2.{w,b}), ln_f.{w,b}; linear layers carry no bias."""
    d, v, ctx, ff = 768, 50257, 1024, 3072
    out = [("wte", (v, d)), ("wpe", (ctx, d))]
    for i in range(12):
        out += [
            (f"h{i}.qkv.w", (d, 3 * d)),
            (f"h{i}.proj.w", (d, d)),
            (f"h{i}.fc.w", (d, ff)),
            (f"h{i}.fc2.w", (ff, d)),
            (f"h{i}.ln_1.w", (d,)),
            (f"h{i}.ln_1.b", (d,)),
            (f"h{i}.ln_2.w", (d,)),
            (f"h{i}.ln_2.b", (d,)),
        ]
    out += [("ln_f.w", (d,)), ("ln_f.b", (d,))]
    return out


def mistral_7b_tensors():
    """Mistral-7B-shaped parameter list: 32 layers, d=4096, 32 q heads / 8 kv heads of
    head dim 128, MLP 14336, vocab 32000, untied lm_head."""
    d, ff, vocab, kv = 4096, 14336, 32000, 8 * 128
    out = [("embed", (vocab, d))]
    for i in range(32):
        out += [
            (f"l{i}.q", (d, d)),
            (f"l{i}.k", (kv, d)),
            (f"l{i}.v", (kv, d)),
            (f"l{i}.o", (d, d)),
            (f"l{i}.gate", (ff, d)),
            (f"l{i}.up", (ff, d)),
            (f"l{i}.down", (d, ff)),
            (f"l{i}.norm1", (d,)),
            (f"l{i}.norm2", (d,)),
        ]
    out += [("norm", (d,)), ("lm_head", (vocab, d))]
    return out


def numel(tensors) -> int:
    n = 0
    for _, shp in tensors:
        k = 1
        for s in shp:
            k *= s
        n += k
    return n


GPT2_SMALL_PSI = 124_356_864
MISTRAL_7B_PSI = 7_241_732_096


# ----------------------------------------------------------------------------------------
# seeded tensors
# ----------------------------------------------------------------------------------------

def _normal(n, std, device, dtype, *keys, out=None):
    g = _gen(device, *keys)
    t = out if out is not None else torch.empty(n, dtype=torch.float32, device=device)
    t.normal_(0.0, std, generator=g)
    return t if dtype == torch.float32 else t.to(dtype)


def master_params(psi: int, psi_padded: int, device="cpu", seed_key=0, std=0.02):
    """fp32 master weights of length psi_padded; entries past psi are zero."""
    t = torch.zeros(psi_padded, dtype=torch.float32, device=device)
    if psi:
        _normal(psi, std, device, torch.float32, TID_MASTER, seed_key, out=t[:psi])
    return t


def rank_grads(psi: int, psi_padded: int, rank: int, step: int, device="cpu", seed_key=0, std=1e-3):
    """One rank's bf16 local gradient for one step, length psi_padded, zero past psi."""
    t = torch.zeros(psi_padded, dtype=torch.bfloat16, device=device)
    if psi:
        f = _normal(psi, std, device, torch.float32, TID_GRAD, seed_key, rank, step)
        t[:psi] = f.to(torch.bfloat16)
    return t


def rank_grads_f32(psi: int, psi_padded: int, rank: int, step: int, device="cpu", seed_key=0, std=1e-3):
    """One rank's fp32 local gradient (kept in fp32, as the Megatron distributed optimizer
    accumulates it), length psi_padded, zero past psi."""
    t = torch.zeros(psi_padded, dtype=torch.float32, device=device)
    if psi:
        _normal(psi, std, device, torch.float32, TID_GRAD, seed_key, rank, step, out=t[:psi])
    return t


def chunk_grads(n: int, n_ranks: int, step: int, device="cpu", seed_key=0, std=1e-3):
    """The n_ranks incoming bf16 gradient chunks (each n elements) that one rank receives
    for its own shard; returned as one [n_ranks, n] tensor, row q = rank q's chunk."""
    t = torch.empty((n_ranks, n), dtype=torch.bfloat16, device=device)
    for q in range(n_ranks):
        t[q] = _normal(n, std, device, torch.float32, TID_GRAD, seed_key, q, step).to(torch.bfloat16)
    return t


def adam_moments(n: int, device="cpu", seed_key=0, step=1, std_m=1e-4, std_v=1e-7):
    """Non-zero Adam moments for tests that start mid-training: m ~ N(0, std_m),
    v = |N(0, std_v)| (v is a running mean of squares, so it is non-negative)."""
    m = _normal(n, std_m, device, torch.float32, TID_STATE_M, seed_key, step)
    v = _normal(n, std_v, device, torch.float32, TID_STATE_V, seed_key, step).abs_()
    return m, v


def weight_shards(rows_out: int, k_in: int, n_ranks: int, device="cpu", seed_key=0, std=0.02):
    """A bf16 [rows_out, k_in] weight split into n_ranks dim-0 row shards; returns a list
    of contiguous [rows_out/n_ranks, k_in] tensors, shard r = rows [r*R/N, (r+1)*R/N)."""
    assert rows_out % n_ranks == 0
    rs = rows_out // n_ranks
    out = []
    for r in range(n_ranks):
        out.append(_normal(rs * k_in, std, device, torch.bfloat16, TID_WEIGHT, seed_key, r).view(rs, k_in))
    return out


def activations(m_tokens: int, k_in: int, device="cpu", seed_key=0, std=1.0):
    """bf16 [m_tokens, k_in] activation, row-major."""
    return _normal(m_tokens * k_in, std, device, torch.bfloat16, TID_ACT, seed_key).view(m_tokens, k_in)


def upstream_grad(m_tokens: int, n_out: int, device="cpu", seed_key=0, std=1.0):
    """bf16 [m_tokens, n_out] upstream gradient dY for an FSDP linear backward."""
    return _normal(m_tokens * n_out, std, device, torch.bfloat16, TID_DY, seed_key).view(m_tokens, n_out)
