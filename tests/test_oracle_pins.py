"""Pins for the CPU oracle: each check ties the oracle to something other than itself —
numbers printed on the pages (tests/golden), closed forms, invariants the pages state,
library routines for special cases (torch's bf16 cast, torch.optim.Adam / AdamW), exact
rational arithmetic and brute force on tiny inputs. Mutation tests at the end plant
plausible mistakes in the oracle (on the CPU) and show that a pin catches each one.
"""
from __future__ import annotations

import math
from fractions import Fraction
from pathlib import Path

import numpy as np
import pytest
import torch

import oracle.zero_oracle as O

GOLDEN = Path(__file__).parent / "golden"
U32 = 2.0 ** -24  # unit roundoff of fp32 round-to-nearest


def golden_rows(name):
    rows = []
    for line in (GOLDEN / name).read_text().splitlines():
        line = line.strip()
        if line and not line.startswith("#"):
            rows.append(line.split())
    return rows


def torch_bf16_bits(x32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------------------------------
# bf16 conversions — pinned to torch's cast (a library routine) and hand-made ties
# ---------------------------------------------------------------------------------------

def test_bf16_widening_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = O.bf16_to_f32(bits)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    same = (ours.view(np.uint32) == ref.view(np.uint32)) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()


def test_bf16_rne_matches_torch_on_random_bits():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2 ** 32, size=400_000, dtype=np.uint64).astype(np.uint32)
    # exact ties: dropped half == 0x8000 with both parities of the kept LSB
    ties = (rng.integers(0, 2 ** 16, size=20_000, dtype=np.uint64).astype(np.uint32) << np.uint32(16)) | np.uint32(0x8000)
    x = np.concatenate([bits, ties]).view(np.float32)
    ours = O.f32_to_bf16(x)
    ref = torch_bf16_bits(x)
    fin = ~np.isnan(x)
    assert np.array_equal(ours[fin], ref[fin])
    assert np.isnan(O.bf16_to_f32(ours[~fin])).all()


def test_bf16_rne_hand_cases():
    cases = {
        0x3F808000: 0x3F80,  # 1 + 2^-8: tie, kept LSB even -> down
        0x3F818000: 0x3F82,  # 1 + 3*2^-8: tie, kept LSB odd -> up
        0x3F808001: 0x3F81,  # just above the tie -> up
        0x7F7FFFFF: 0x7F80,  # largest float rounds past bf16 max -> +inf
        0x00008000: 0x0000,  # smallest tie among denormals -> even (zero)
        0x00018000: 0x0002,  # denormal tie with odd kept LSB -> up
        0x80000000: 0x8000,  # -0 stays -0
        0xFF800000: 0xFF80,  # -inf
    }
    x = np.array(list(cases), dtype=np.uint32).view(np.float32)
    assert list(O.f32_to_bf16(x)) == list(cases.values())


# ---------------------------------------------------------------------------------------
# layout: brute force coverage on tiny inputs, hand-derived counts for the workloads
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("psi", [1, 7, 13, 1000])
@pytest.mark.parametrize("n", [1, 2, 3, 4, 8, 64])
@pytest.mark.parametrize("bucket_mult", [1, 3, 1000])
def test_layout_bruteforce(psi, n, bucket_mult):
    lay = O.make_layout(psi, n, 2 * n * bucket_mult)
    assert lay.psi_padded % n == 0 and psi <= lay.psi_padded < psi + n
    assert lay.shard * n == lay.psi_padded
    cover = np.zeros(lay.psi_padded, dtype=np.int64)
    for r in range(n):
        for k in range(lay.n_buckets):
            lo, hi = O.bucket_range(lay, r, k)
            assert 0 < hi - lo <= bucket_mult
            cover[lo:hi] += 1
            assert all(O.owner(lay, j) == r for j in range(lo, hi))
    assert (cover == 1).all()


def test_layout_workload_counts():
    mib = 1 << 20
    # tiny ZeRO-2 case: psi 2^20, N=4, 25 MiB buckets -> one bucket per shard
    lay = O.make_layout(1_048_576, 4, 25 * mib)
    assert (lay.psi_padded, lay.shard, lay.bucket_elems, lay.n_buckets) == (1_048_576, 262_144, 3_276_800, 1)
    # GPT-2-small list, N=8, 25 MiB: 15,544,608-element shards, 10 buckets of 1,638,400
    lay = O.make_layout(124_356_864, 8, 25 * mib)
    assert (lay.psi_padded, lay.shard, lay.bucket_elems, lay.n_buckets) == (124_356_864, 15_544_608, 1_638_400, 10)
    # Mistral-7B list, N=8, 50 MiB: 905,216,512-element shards, 277 buckets
    lay = O.make_layout(7_241_732_096, 8, 50 * mib)
    assert (lay.shard, lay.bucket_elems, lay.n_buckets) == (905_216_512, 3_276_800, 277)
    with pytest.raises(ValueError):
        O.make_layout(10, 4, 7)
    with pytest.raises(ValueError):
        O.make_layout(0, 4, 1024)


def test_workload_tensor_lists():
    import synth
    assert synth.numel(synth.gpt2_small_tensors()) == synth.GPT2_SMALL_PSI == 124_356_864
    assert synth.numel(synth.mistral_7b_tensors()) == synth.MISTRAL_7B_PSI == 7_241_732_096


# ---------------------------------------------------------------------------------------
# memory and communication accounting — numbers printed on the pages
# ---------------------------------------------------------------------------------------

def test_memory_table_7b_n8_golden():
    lay = O.make_layout(7_000_000_000, 8, 1 << 20)
    assert lay.psi_padded == 7_000_000_000
    for strategy, _formula, gb, comm in golden_rows("memory_7b_n8.txt"):
        want = Fraction(gb) * 10 ** 9
        if strategy == "megatron_unsharded":
            # 18 bytes per parameter held in full: bf16 param 2 + fp32 grad 4 + master/m/v 12
            one = O.make_layout(7_000_000_000, 1, 1 << 20)
            assert O.model_state_bytes("megatron", one)["total"] == want
            continue
        assert O.model_state_bytes(strategy, lay)["total"] == want, strategy
        assert O.comm_elements(strategy, lay)["total"] == int(comm) * lay.psi_padded


def test_stage_table_concepts_golden():
    rng = np.random.default_rng(7)
    rows = golden_rows("stage_table_concepts.txt")
    for _ in range(50):
        n = int(rng.integers(1, 129))
        psi = int(rng.integers(1, 10 ** 12)) * n
        lay = O.make_layout(psi, n, 1 << 20)
        P = Fraction(psi)
        for stage, _sharded, formula, comm in rows:
            expr = {"16P": 16 * P, "4P+12P/N": 4 * P + 12 * P / n, "2P+14P/N": 2 * P + 14 * P / n, "16P/N": 16 * P / n}[formula]
            assert O.model_state_bytes(stage, lay)["total"] == expr
            assert O.comm_elements(stage, lay)["total"] == int(comm) * psi
    lay = O.make_layout(8_000, 8, 1 << 20)
    assert Fraction(O.comm_elements("zero3", lay)["total"], O.comm_elements("ddp", lay)["total"]) == Fraction(3, 2)


def test_zero1_allreduce_variant_is_3psi():
    lay = O.make_layout(8_000, 8, 1 << 20)
    assert O.comm_elements("zero1", lay, zero1_via_allreduce=True)["total"] == 3 * 8_000
    assert O.comm_elements("zero1", lay)["total"] == 2 * 8_000


def test_full_shard_70b_golden():
    for psi, n, gb in golden_rows("full_shard_70b.txt"):
        lay = O.make_layout(int(float(psi)), int(n), 1 << 20)
        assert Fraction(O.model_state_bytes("zero3", lay)["total"]) == Fraction(gb) * 10 ** 9


def test_ring_allreduce_golden():
    for s_gb, n, gb in golden_rows("ring_allreduce_7b.txt"):
        s = float(s_gb) * 1e9
        if n == "inf":
            assert O.ring_allreduce_bytes(s, 10 ** 7) == pytest.approx(float(gb) * 1e9, rel=1e-6)
        else:
            assert O.ring_allreduce_bytes(s, int(n)) == pytest.approx(float(gb) * 1e9, rel=1e-15)
    # in elements: a ring reduce-scatter or all-gather of P sends (N-1)/N * P per rank, and
    # DDP's two of them at 2 bytes per bf16 element give the page's 2 (N-1)/N * S bytes
    lay = O.make_layout(7_000_000_000, 8, 1 << 20)
    c = O.comm_elements("ddp", lay)
    sent = O.ring_sent_elements(c["reduce_scatter"], 8) + O.ring_sent_elements(c["all_gather_fwd"], 8)
    assert 2 * sent == O.ring_allreduce_bytes(2 * 7e9, 8)


@pytest.mark.parametrize("stage", ["ddp", "zero1", "zero2", "zero3"])
def test_held_buffers_equal_counter(stage):
    lay = O.make_layout(1001, 4, 64)
    ranks = O.init_ranks(stage, lay, np.zeros(lay.psi_padded, np.float32))
    for st in ranks:
        assert st.nbytes() == O.model_state_bytes(stage, lay)["total"]


# ---------------------------------------------------------------------------------------
# reduction
# ---------------------------------------------------------------------------------------

def bf16_of(vals):
    return O.f32_to_bf16(np.asarray(vals, dtype=np.float32))


def test_reduce_exact_on_small_integers():
    rng = np.random.default_rng(3)
    for n in (1, 2, 4, 8, 64):
        ints = rng.integers(-100, 101, size=(n, 999))
        grads = [bf16_of(row) for row in ints]
        got = O.reduce_sum_scale(grads, 0, 999)
        want = ints.sum(axis=0) / n  # exact: integer sums < 2^24, N a power of two
        assert np.array_equal(got.astype(np.float64), want)


def test_reduce_rank_order_is_left_to_right():
    # ((2^24 + 1) + 1) + 0 rounds back to 2^24 at each step (ties to even); any other
    # association, e.g. 2^24 + (1 + 1), gives 2^24 + 2
    grads = [bf16_of([2.0 ** 24]), bf16_of([1.0]), bf16_of([1.0]), bf16_of([0.0])]
    assert O.reduce_sum_scale(grads, 0, 1)[0] == np.float32(2.0 ** 22)


@pytest.mark.parametrize("n", [2, 3, 5, 8, 64])
def test_reduce_mean_within_rounding_bound(n):
    rng = np.random.default_rng(n)
    x = rng.normal(0, 1e-3, size=(n, 4001)).astype(np.float32)
    grads = [bf16_of(r) for r in x]
    got = O.reduce_sum_scale(grads, 0, 4001).astype(np.float64)
    vals = np.stack([O.bf16_to_f32(g).astype(np.float64) for g in grads])
    exact = np.array([math.fsum(vals[:, j]) for j in range(vals.shape[1])]) / n
    # recursive summation: |err| <= (n-1) u sum|x| ; scaling by f32(1/N): 2u relative
    bound = (n - 1) * U32 * np.abs(vals).sum(axis=0) / n * (1 + 3 * U32) + 3 * U32 * np.abs(exact)
    assert (np.abs(got - exact) <= bound + 1e-45).all()


@pytest.mark.parametrize("psi,n,bucket_bytes", [(1, 1, 2), (13, 4, 8), (1000, 3, 6 * 7), (4099, 8, 1 << 20)])
def test_allreduce_equals_reduce_scatter_then_all_gather(psi, n, bucket_bytes):
    lay = O.make_layout(psi, n, bucket_bytes)
    rng = np.random.default_rng(psi)
    grads = [bf16_of(np.pad(rng.normal(0, 1e-3, psi), (0, lay.psi_padded - psi))) for _ in range(n)]
    ar = O.all_reduce(lay, grads)
    rs_ag = O.all_gather([O.reduce_scatter(lay, grads, r) for r in range(n)])
    assert ar.view(np.uint32).tobytes() == rs_ag.view(np.uint32).tobytes()


# ---------------------------------------------------------------------------------------
# Adam
# ---------------------------------------------------------------------------------------

def f32_nearest(x: Fraction) -> np.float32:
    """The fp32 value nearest the exact rational x (ties to even)."""
    f = np.float32(float(x))
    best = None
    for c in (np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))):
        d = abs(Fraction(float(c)) - x)
        key = (d, int(np.array(c).view(np.uint32)) & 1)
        if best is None or key < best[0]:
            best = (key, c)
    return best[1]


def test_bias_corrections_exact():
    hp = O.AdamHyper()
    b1 = Fraction(float(np.float32(hp.beta1)))
    b2 = Fraction(float(np.float32(hp.beta2)))
    for t in range(1, 301):
        bc1, bc2 = O.bias_corrections(hp, t)
        assert bc1 == f32_nearest(1 - b1 ** t), t
        assert bc2 == f32_nearest(1 - b2 ** t), t


def check_step1_closed_form(adam_update):
    """Step 1 from m = v = 0: the bias corrections give mh = g and vh = g^2, so the update
    is u = lr g / (|g| + eps) ~ lr sign(g) — checked on u itself (subtracting u from a
    master near 0.02 would cancel digits)."""
    hp = O.AdamHyper()
    rng = np.random.default_rng(11)
    g = rng.normal(0, 1e-3, 20000).astype(np.float32)
    z = np.zeros_like(g)
    _, m, v, u = adam_update(z + np.float32(0.02), z, z, g, hp, 1, return_update=True)
    lr, eps = float(np.float32(hp.lr)), float(np.float32(hp.eps))
    gd = g.astype(np.float64)
    want = lr * gd / (np.abs(gd) + eps)
    assert np.all(np.abs(u - want) <= 1e-6 * np.abs(want))
    assert np.all(np.abs(m - (1 - float(np.float32(hp.beta1))) * gd) <= 2 * U32 * np.abs(gd))


def test_adam_step1_closed_form():
    check_step1_closed_form(O.adam_update)


def run_torch_adam(p0, grads, hp, decoupled):
    p = torch.tensor(p0.astype(np.float64), requires_grad=True)
    kw = dict(lr=float(np.float32(hp.lr)), betas=(float(np.float32(hp.beta1)), float(np.float32(hp.beta2))),
              eps=float(np.float32(hp.eps)), weight_decay=float(np.float32(hp.weight_decay)), foreach=False)
    opt = (torch.optim.AdamW if decoupled else torch.optim.Adam)([p], **kw)
    for g in grads:
        p.grad = torch.tensor(g.astype(np.float64))
        opt.step()
    st = opt.state[p]
    return p.detach().numpy(), st["exp_avg"].numpy(), st["exp_avg_sq"].numpy()


def check_adam_against_torch(adam_update, wd=0.0, steps=6):
    """Cross-check with torch.optim.Adam / AdamW run in float64 (a library routine, exact
    to ~1e-16): same fp32 inputs, same hyper-parameters. Values of |g| near eps make the
    eps placement visible; the tolerances are fp32 rounding bounds over `steps` steps."""
    hp = O.AdamHyper(weight_decay=wd)
    rng = np.random.default_rng(5)
    n = 6000
    p0 = rng.normal(0, 0.02, n).astype(np.float32)
    grads = []
    for t in range(steps):
        g = rng.normal(0, 1e-3, n)
        g[: n // 6] *= 1e-5  # |g| ~ 1e-8, comparable to eps
        grads.append(g.astype(np.float32))
    w, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    for t, g in enumerate(grads, start=1):
        w, m, v = adam_update(w, m, v, g, hp, t)
    tw, tm, tv = run_torch_adam(p0, grads, hp, decoupled=wd != 0.0)
    gmax = max(np.abs(g).max() for g in grads)
    assert np.all(np.abs(m - tm) <= 4 * steps * U32 * gmax)
    assert np.all(np.abs(v - tv) <= 4 * steps * U32 * gmax * gmax)
    # master: one fp32 rounding of master per step plus ~12 roundings on an update <= ~lr
    lr = float(np.float32(hp.lr))
    tol = steps * (np.abs(tw) * U32 * 2 + 16 * U32 * lr)
    assert np.all(np.abs(w - tw) <= tol)


def test_adam_matches_torch_adam():
    check_adam_against_torch(O.adam_update)


def test_adamw_decoupled_decay_matches_torch_adamw():
    check_adam_against_torch(O.adam_update, wd=0.1)


def test_adam_zero_grad_on_zero_state_is_identity():
    hp = O.AdamHyper()
    w0 = np.array([0.0, 0.02, -1.5, 3e-39], dtype=np.float32)
    z = np.zeros(4, np.float32)
    for t in (1, 2, 1000):
        w, m, v = O.adam_update(w0, z, z, z, hp, t)
        assert w.tobytes() == w0.tobytes() and not m.any() and not v.any()


# ---------------------------------------------------------------------------------------
# strategies: every ZeRO stage equals DDP; DDP replicas identical; N = 1 is plain Adam
# ---------------------------------------------------------------------------------------

def run_strategy(stage, lay, master0, all_grads, hp):
    ranks = O.init_ranks(stage, lay, master0)
    for t, grads in enumerate(all_grads, start=1):
        O.step_ranks(ranks, lay, grads, hp, t)
    return ranks


def make_case(psi, n, steps, seed):
    rng = np.random.default_rng(seed)
    pad = (-psi) % n
    master0 = np.pad(rng.normal(0, 0.02, psi).astype(np.float32), (0, pad))
    all_grads = [[bf16_of(np.pad(rng.normal(0, 1e-3, psi), (0, pad))) for _ in range(n)] for _ in range(steps)]
    return master0, all_grads


@pytest.mark.parametrize("psi,n", [(1, 1), (7, 2), (13, 3), (13, 4), (1000, 8), (1001, 64), (4097, 5)])
def test_all_stages_equal_ddp(psi, n):
    hp = O.AdamHyper()
    master0, all_grads = make_case(psi, n, 3, psi * 100 + n)
    lay_small = O.make_layout(psi, n, 2 * n)       # one element per rank per bucket
    lay_big = O.make_layout(psi, n, 1 << 30)       # one bucket per shard
    ddp = run_strategy("ddp", lay_big, master0, all_grads, hp)
    ref_param = ddp[0].buffers["param"]
    ref_master = ddp[0].buffers["master"]
    for st in ddp[1:]:  # DDP replicas stay identical
        assert st.buffers["master"].tobytes() == ref_master.tobytes()
        assert st.buffers["param"].tobytes() == ref_param.tobytes()
    for stage in ("zero1", "zero2", "zero3"):
        for lay in (lay_small, lay_big):
            ranks = run_strategy(stage, lay, master0, all_grads, hp)
            assert O.gather_params(ranks).tobytes() == ref_param.tobytes(), stage
            assert O.gather_master(ranks, lay).tobytes() == ref_master.tobytes(), stage
            if stage in ("zero1", "zero2"):
                for st in ranks:
                    assert st.buffers["param"].tobytes() == ref_param.tobytes()
    # padding stays zero
    assert not ref_master[psi:].any() and not ref_param[psi:].any()


def test_single_rank_is_plain_adam():
    hp = O.AdamHyper()
    master0, all_grads = make_case(3001, 1, 4, 9)
    ranks = run_strategy("zero2", O.make_layout(3001, 1, 1 << 20), master0, all_grads, hp)
    w, m, v = master0.copy(), np.zeros_like(master0), np.zeros_like(master0)
    for t, grads in enumerate(all_grads, start=1):
        w, m, v = O.adam_update(w, m, v, O.bf16_to_f32(grads[0]), hp, t)
    assert ranks[0].buffers["master"].tobytes() == w.tobytes()
    tw, _, _ = run_torch_adam(master0, [O.bf16_to_f32(g[0]) for g in all_grads], hp, decoupled=False)
    assert np.all(np.abs(w - tw) <= 4 * (np.abs(tw) * 2 * U32 + 16 * U32 * 1e-4))


def test_fused_elements_equals_strategy_step():
    hp = O.AdamHyper()
    psi, n = 1000, 4
    master0, all_grads = make_case(psi, n, 2, 77)
    lay = O.make_layout(psi, n, 40)
    ranks = run_strategy("zero2", lay, master0, all_grads, hp)
    w, m, v = master0.copy(), np.zeros(psi, np.float32), np.zeros(psi, np.float32)
    for t, grads in enumerate(all_grads, start=1):
        w, m, v, p = O.fused_step_elements(grads, w, m, v, hp, t)
    assert O.gather_master(ranks, lay).tobytes() == w.tobytes()
    assert O.gather_params(ranks).tobytes() == p.tobytes()


def test_megatron_fp32_grads_reduce_in_rank_order():
    grads = [np.array([2.0 ** 24], np.float32), np.array([1.0], np.float32), np.array([1.0], np.float32),
             np.array([0.0], np.float32)]
    assert O.reduce_sum_scale(grads, 0, 1)[0] == np.float32(2.0 ** 22)
    with pytest.raises(TypeError):
        O.reduce_sum_scale([np.zeros(2, np.float64)], 0, 2)


@pytest.mark.parametrize("psi,n", [(13, 3), (1000, 8), (1001, 64)])
def test_megatron_equals_zero1_on_bf16_exact_grads(psi, n):
    """Megatron's distributed optimizer is ZeRO-1-style ([Interview] worked table note):
    with fp32 gradients that are exactly the widened bf16 ones it must give ZeRO-1's
    parameters bit for bit; with general fp32 gradients it must match plain fp32 Adam."""
    hp = O.AdamHyper()
    master0, all_grads = make_case(psi, n, 3, psi + 7 * n)
    lay = O.make_layout(psi, n, 2 * n * 5)
    z1 = run_strategy("zero1", lay, master0, all_grads, hp)
    mg = run_strategy("megatron", lay, master0, [[O.bf16_to_f32(g) for g in gs] for gs in all_grads], hp)
    assert O.gather_params(mg).tobytes() == O.gather_params(z1).tobytes()
    assert O.gather_master(mg, lay).tobytes() == O.gather_master(z1, lay).tobytes()
    assert mg[0].buffers["grad"].dtype == np.float32 and mg[0].buffers["grad"].size == lay.psi_padded


def test_megatron_single_rank_is_plain_adam_on_fp32_grads():
    hp = O.AdamHyper()
    rng = np.random.default_rng(12)
    master0 = rng.normal(0, 0.02, 999).astype(np.float32)
    grads = [[rng.normal(0, 1e-3, 999).astype(np.float32)] for _ in range(3)]
    ranks = run_strategy("megatron", O.make_layout(999, 1, 1 << 20), master0, grads, hp)
    tw, _, _ = run_torch_adam(master0, [g[0] for g in grads], hp, decoupled=False)
    assert np.all(np.abs(ranks[0].buffers["master"] - tw) <= 3 * (np.abs(tw) * 2 * U32 + 16 * U32 * 1e-4))


# ---------------------------------------------------------------------------------------
# FSDP linear: brute force in exact rational arithmetic, orientation and shard order
# ---------------------------------------------------------------------------------------

def test_fsdp_linear_bruteforce_exact():
    rng = np.random.default_rng(21)
    m, k, rows, n = 3, 5, 6, 3
    a = bf16_of(rng.normal(0, 1, (m, k)))
    shards = [bf16_of(rng.normal(0, 0.02, (rows // n, k))) for _ in range(n)]
    y64, y32, ybf = O.fsdp_linear_forward(a, shards)
    af = O.bf16_to_f32(a)
    wf = np.concatenate([O.bf16_to_f32(s) for s in shards])
    for i in range(m):
        for j in range(rows):
            exact = sum(Fraction(float(af[i, q])) * Fraction(float(wf[j, q])) for q in range(k))
            assert abs(Fraction(float(y64[i, j])) - exact) <= abs(exact) * Fraction(1, 2 ** 50)
            assert y32[i, j] == f32_nearest(exact)
            assert ybf[i, j] == O.f32_to_bf16(np.float32(y32[i, j]))


def test_fsdp_linear_orientation_and_shard_order():
    # W row n (global index) holds the value n in column 0; A selects column 0, so
    # Y[:, n] = n only if the shards are concatenated in rank order and Y = A W^T
    n_ranks, rs, k = 4, 3, 8
    shards = []
    for r in range(n_ranks):
        w = np.zeros((rs, k), np.float32)
        w[:, 0] = np.arange(r * rs, (r + 1) * rs)
        shards.append(bf16_of(w))
    a = np.zeros((2, k), np.float32)
    a[:, 0] = 1.0
    _, y32, _ = O.fsdp_linear_forward(bf16_of(a), shards)
    assert y32.shape == (2, n_ranks * rs)
    assert (y32 == np.arange(n_ranks * rs, dtype=np.float32)).all()


def test_fsdp_linear_backward_bruteforce():
    rng = np.random.default_rng(4)
    m, k, rows, n = 4, 3, 4, 2
    a = bf16_of(rng.normal(0, 1, (m, k)))
    shards = [bf16_of(rng.normal(0, 0.02, (rows // n, k))) for _ in range(n)]
    dy = bf16_of(rng.normal(0, 1, (m, rows)))
    dx, dw = O.fsdp_linear_backward(a, shards, dy, n)
    af, dyf = O.bf16_to_f32(a), O.bf16_to_f32(dy)
    wf = np.concatenate([O.bf16_to_f32(s) for s in shards])
    for i in range(m):
        for q in range(k):
            assert dx[i, q] == pytest.approx(sum(float(dyf[i, j]) * float(wf[j, q]) for j in range(rows)), rel=1e-14)
    for j in range(rows):
        for q in range(k):
            assert dw[j, q] == pytest.approx(sum(float(dyf[i, j]) * float(af[i, q]) for i in range(m)), rel=1e-14)


def test_transpose_cat_bruteforce():
    rng = np.random.default_rng(17)
    srcs = [rng.integers(0, 65535, (3, 5)).astype(np.uint16) for _ in range(4)]
    dst = O.transpose_cat(srcs)
    assert dst.shape == (5, 12)
    for q in range(4):
        for r in range(3):
            for c in range(5):
                assert dst[c, q * 3 + r] == srcs[q][r, c]
    # W^T from row shards equals the transpose of the gathered W
    assert np.array_equal(O.transpose_cat(srcs), O.gather_rows(srcs).T)


def test_reduce_rows_matches_elementwise_reduction():
    rng = np.random.default_rng(8)
    n, rows, k = 4, 8, 5
    dws = [rng.normal(0, 1, (rows, k)).astype(np.float32) for _ in range(n)]
    for r in range(n):
        got = O.reduce_rows(dws, n, r)
        acc = dws[0][r * 2:(r + 1) * 2].copy()
        for q in range(1, n):
            acc = (acc + dws[q][r * 2:(r + 1) * 2]).astype(np.float32)
        assert got.tobytes() == (acc * np.float32(0.25)).astype(np.float32).tobytes()


def test_silu_matches_torch_and_identities():
    x = np.concatenate([np.linspace(-60, 60, 2001), [0.0, -1e-300, 1e-300, -800.0, 800.0]])
    ref = torch.nn.functional.silu(torch.tensor(x, dtype=torch.float64)).numpy()
    assert np.allclose(O.silu(x), ref, rtol=1e-15, atol=1e-300)
    assert O.silu(0.0) == 0.0
    y = np.linspace(-30, 30, 601)
    assert np.allclose(O.silu(y) - O.silu(-y), y, rtol=1e-14, atol=1e-14)  # silu(x) - silu(-x) = x


def test_mlp_unit_forward_bruteforce():
    rng = np.random.default_rng(31)
    m, d, f, n = 3, 4, 6, 2
    x = bf16_of(rng.normal(0, 1, (m, d)))
    gate = [bf16_of(rng.normal(0, 0.5, (f // n, d))) for _ in range(n)]
    up = [bf16_of(rng.normal(0, 0.5, (f // n, d))) for _ in range(n)]
    down = [bf16_of(rng.normal(0, 0.5, (d // n, f))) for _ in range(n)]
    g, u, h, y = O.mlp_unit_forward(x, gate, up, down)
    xf = O.bf16_to_f32(x).astype(float)
    wg = np.concatenate([O.bf16_to_f32(s) for s in gate]).astype(float)
    wu = np.concatenate([O.bf16_to_f32(s) for s in up]).astype(float)
    wd = np.concatenate([O.bf16_to_f32(s) for s in down]).astype(float)
    for i in range(m):
        for j in range(f):
            gij = sum(xf[i, k] * wg[j, k] for k in range(d))
            uij = sum(xf[i, k] * wu[j, k] for k in range(d))
            assert g[i, j] == pytest.approx(gij, rel=1e-14, abs=1e-300)
            assert h[i, j] == pytest.approx(gij / (1 + math.exp(-gij)) * uij, rel=1e-13, abs=1e-300)
        for j in range(d):
            assert y[i, j] == pytest.approx(sum(h[i, k] * wd[j, k] for k in range(f)), rel=1e-12, abs=1e-300)


def test_silu_gate_backward_matches_torch_autograd():
    """The SiLU-gate backward against torch's automatic differentiation of silu(g) * u in
    float64 (a library routine that differentiates the forward; it shares nothing with the
    oracle's closed form), on bf16 inputs over the range activations take."""
    rng = np.random.default_rng(41)
    n = 20000
    g = bf16_of(np.concatenate([rng.normal(0, 3, n - 6), [0.0, -30.0, 30.0, -1.278, 1e-3, -88.0]]))
    u = bf16_of(rng.normal(0, 2, n))
    dh = bf16_of(rng.normal(0, 1, n))
    dg, du = O.silu_gate_backward(dh, g, u)
    gt = torch.tensor(O.bf16_to_f32(g).astype(np.float64), requires_grad=True)
    ut = torch.tensor(O.bf16_to_f32(u).astype(np.float64), requires_grad=True)
    (torch.nn.functional.silu(gt) * ut).backward(torch.tensor(O.bf16_to_f32(dh).astype(np.float64)))
    assert np.allclose(dg, gt.grad.numpy(), rtol=1e-12, atol=1e-300)
    assert np.allclose(du, ut.grad.numpy(), rtol=1e-12, atol=1e-300)


def test_silu_gate_backward_is_the_derivative_of_the_forward():
    """Central differences of the oracle's own forward silu(g) * u (O.silu) reproduce the
    backward: d/dg and d/du of dh * silu(g) * u."""
    g = np.linspace(-12, 12, 481)
    g_b, u_b, dh_b = bf16_of(g), bf16_of(np.full_like(g, 1.5)), bf16_of(np.full_like(g, -0.75))
    gf, uf, dhf = (O.bf16_to_f32(x).astype(np.float64) for x in (g_b, u_b, dh_b))
    dg, du = O.silu_gate_backward(dh_b, g_b, u_b)
    h = 1e-6
    num_dg = dhf * uf * (O.silu(gf + h) - O.silu(gf - h)) / (2 * h)
    num_du = dhf * O.silu(gf)
    assert np.allclose(dg, num_dg, rtol=1e-7, atol=1e-9)
    assert np.allclose(du, num_du, rtol=1e-14, atol=1e-300)


def test_silu_gate_backward_closed_forms():
    """g = 0: silu = 0 and silu' = 1/2, so dU = 0 and dG = dh u / 2; large |g|: silu' -> 1
    (g -> +inf) and -> 0 (g -> -inf)."""
    dh, u = bf16_of(np.array([0.5, -2.0, 3.0])), bf16_of(np.array([4.0, 1.5, -0.25]))
    dg, du = O.silu_gate_backward(dh, bf16_of(np.zeros(3)), u)
    assert np.array_equal(du, np.zeros(3))
    assert np.array_equal(dg, O.bf16_to_f32(dh) * O.bf16_to_f32(u) * 0.5)
    dg, _ = O.silu_gate_backward(bf16_of(np.ones(2)), bf16_of(np.array([80.0, -80.0])), bf16_of(np.ones(2)))
    assert dg[0] == pytest.approx(1.0, rel=1e-15) and abs(dg[1]) < 1e-30


# ---------------------------------------------------------------------------------------
# mutation tests: a planted mistake in the oracle must fail one of the pins above
# ---------------------------------------------------------------------------------------

def _adam_eps_inside_sqrt(master, m, v, g, hp, t, return_update=False):
    b1, b2 = np.float32(hp.beta1), np.float32(hp.beta2)
    bc1, bc2 = O.bias_corrections(hp, t)
    m1 = b1 * m + (np.float32(1) - b1) * g
    v1 = b2 * v + (np.float32(1) - b2) * (g * g)
    u = np.float32(hp.lr) * ((m1 / bc1) / np.sqrt(v1 / bc2 + np.float32(hp.eps)))
    return (master - u, m1, v1, u) if return_update else (master - u, m1, v1)


def _adam_no_bias_correction(master, m, v, g, hp, t, return_update=False):
    b1, b2 = np.float32(hp.beta1), np.float32(hp.beta2)
    m1 = b1 * m + (np.float32(1) - b1) * g
    v1 = b2 * v + (np.float32(1) - b2) * (g * g)
    u = np.float32(hp.lr) * (m1 / (np.sqrt(v1) + np.float32(hp.eps)))
    return (master - u, m1, v1, u) if return_update else (master - u, m1, v1)


def _adam_swapped_betas(master, m, v, g, hp, t, return_update=False):
    return O.adam_update(master, m, v, g, O.AdamHyper(hp.lr, hp.beta2, hp.beta1, hp.eps, hp.weight_decay), t, return_update)


@pytest.mark.parametrize("bad", [_adam_eps_inside_sqrt, _adam_no_bias_correction, _adam_swapped_betas])
def test_mutations_of_adam_are_caught(bad):
    caught = 0
    for check in (check_step1_closed_form, check_adam_against_torch):
        try:
            check(bad)
        except AssertionError:
            caught += 1
    assert caught >= 1


def test_mutation_reversed_rank_order_is_caught(monkeypatch):
    def reversed_sum(grads, lo, hi):
        acc = O.bf16_to_f32(grads[-1][lo:hi]).copy()
        for q in range(len(grads) - 2, -1, -1):
            acc = acc + O.bf16_to_f32(grads[q][lo:hi])
        return acc * O.inv_n(len(grads))
    monkeypatch.setattr(O, "reduce_sum_scale", reversed_sum)
    with pytest.raises(AssertionError):
        test_reduce_rank_order_is_left_to_right()


def test_mutation_reversed_shard_order_is_caught(monkeypatch):
    monkeypatch.setattr(O, "gather_rows", lambda shards: np.concatenate([np.asarray(s) for s in shards][::-1], axis=0))
    with pytest.raises(AssertionError):
        test_fsdp_linear_orientation_and_shard_order()


def test_mutation_dropped_padding_is_caught(monkeypatch):
    real = O.make_layout

    def no_pad(psi, n, bb):
        lay = real(psi, n, bb)
        s = psi // n
        return O.Layout(psi, n, bb, s * n, s, lay.bucket_elems, max(1, -(-s // lay.bucket_elems)))
    monkeypatch.setattr(O, "make_layout", no_pad)
    with pytest.raises(AssertionError):
        test_layout_bruteforce(13, 4, 3)


def _silu_gate_backward_wrong_derivative(dh_bf16, g_bf16, u_bf16):
    dh, g, u = (O.bf16_to_f32(x).astype(np.float64) for x in (dh_bf16, g_bf16, u_bf16))
    s = 1.0 / (1.0 + np.exp(-g))
    return dh * u * (s * (1.0 + g * s)), dh * (g * s)  # (1 - s) dropped


@pytest.mark.parametrize("bad", [_silu_gate_backward_wrong_derivative])
def test_mutations_of_silu_gate_backward_are_caught(bad, monkeypatch):
    monkeypatch.setattr(O, "silu_gate_backward", bad)
    with pytest.raises(AssertionError):
        test_silu_gate_backward_matches_torch_autograd()
    with pytest.raises(AssertionError):
        test_silu_gate_backward_is_the_derivative_of_the_forward()


def test_mutation_swapped_silu_gate_outputs_is_caught(monkeypatch):
    good = O.silu_gate_backward
    monkeypatch.setattr(O, "silu_gate_backward", lambda dh, g, u: good(dh, g, u)[::-1])
    with pytest.raises(AssertionError):
        test_silu_gate_backward_closed_forms()
