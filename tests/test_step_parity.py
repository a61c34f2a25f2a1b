"""GPU parity of the optimizer-step kernels against the CPU oracle, through the C ABI.

Small cases compare every element, bit for bit (the GPU path fixes the same summation
order and IEEE fp32 operation sequence as the oracle, with no FMA contraction), across
every strategy, every rank mode, bucket splits, the TMA / register / scalar kernels, odd
sizes with ragged tails, N = 1 .. 64 and special values. Full-size workloads (GPT-2-small
list at N = 8, one rank of a Mistral-7B list at N = 8, the 1.5B-parameter sweep) are
checked on sampled indices, which the oracle computes one by one — exact because the step
is elementwise.
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
HP = O.AdamHyper()
MIB = 1 << 20


@pytest.fixture(scope="module")
def z():
    import __graft_entry__ as g
    g.build()
    import fsdp_sharded_optimizer_zero_gb300 as z
    yield z
    z.zero_set_fused_kernel(0)


@pytest.fixture(autouse=True)
def _default_kernel(z):
    z.zero_set_fused_kernel(0)
    yield
    z.zero_device_status()
    z.zero_set_fused_kernel(0)


# ---------------------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------------------

def make_inputs(psi, n, steps, seed=0, moments=False):
    lay_p = -(-psi // n) * n
    master0 = synth.master_params(psi, lay_p, seed_key=seed)
    grads = [[synth.rank_grads(psi, lay_p, r, t, seed_key=seed) for r in range(n)] for t in range(1, steps + 1)]
    if moments:
        m0, v0 = synth.adam_moments(lay_p, seed_key=seed)
        m0[psi:] = 0
        v0[psi:] = 0
    else:
        m0 = torch.zeros(lay_p)
        v0 = torch.zeros(lay_p)
    return master0, m0, v0, grads


def oracle_run(stage, psi, n, bb, master0, m0, v0, grads, hp=HP):
    lay = O.make_layout(psi, n, bb)
    ranks = O.init_ranks(stage, lay, master0.numpy())
    m_np, v_np = m0.numpy(), v0.numpy()
    for r, st in enumerate(ranks):
        lo, hi = O.shard_range(lay, r)
        st.buffers["m"][:] = m_np if stage == "ddp" else m_np[lo:hi]
        st.buffers["v"][:] = v_np if stage == "ddp" else v_np[lo:hi]
    for t, gs in enumerate(grads, start=1):
        O.step_ranks(ranks, lay, [bits16(g) for g in gs], hp, t)

    def cat(name):
        if stage == "ddp":
            return ranks[0].buffers[name]
        return np.concatenate([st.buffers[name] for st in ranks])
    return cat("master"), cat("m"), cat("v"), O.gather_params(ranks)


def offset_buf(n, dtype, misalign):
    """A contiguous length-n CUDA tensor whose data pointer is shifted by one element when
    misalign is set (so no vector path applies)."""
    if not misalign:
        return torch.zeros(n, dtype=dtype, device=DEV)
    return torch.zeros(n + 1, dtype=dtype, device=DEV)[1:]


def gpu_run(z, stage, mode, psi, n, bb, master0, m0, v0, grads, hp=HP, misalign=False):
    plan = z.zero_plan(psi, n, stage, bb)
    P, S, NB = plan.psi_padded, plan.shard_elems, plan.n_buckets
    master = offset_buf(P, torch.float32, misalign)
    m = offset_buf(P, torch.float32, misalign)
    v = offset_buf(P, torch.float32, misalign)
    param = offset_buf(P, torch.bfloat16, misalign)
    master.copy_(master0)
    m.copy_(m0)
    v.copy_(v0)
    param.copy_(master0.to(torch.bfloat16))
    sl = lambda t, r: t[r * S:(r + 1) * S]
    ptarget = (lambda r: param) if stage != "zero3" else (lambda r: sl(param, r))
    gbuf = [offset_buf(P, torch.bfloat16, misalign) for _ in range(n)]
    for t, gs in enumerate(grads, start=1):
        for q in range(n):
            gbuf[q].copy_(gs[q])
        if mode == "all":
            z.zero_fused_step(plan, z.ZERO_ALL_RANKS, gbuf, master, m, v, param, hp, t)
        elif mode == "all_buckets":  # every rank, one launch per bucket
            for k in range(NB):
                z.zero_fused_step_buckets(plan, z.ZERO_ALL_RANKS, k, k + 1, gbuf, master, m, v, param, hp, t)
        elif mode == "ranks":
            for r in range(n):
                z.zero_fused_step(plan, r, gbuf, sl(master, r), sl(m, r), sl(v, r), ptarget(r), hp, t)
        elif mode == "buckets":
            for r in range(n):
                for k in range(0, NB, 2):
                    z.zero_fused_step_buckets(plan, r, k, min(k + 2, NB), gbuf, sl(master, r), sl(m, r), sl(v, r),
                                              ptarget(r), hp, t)
        elif mode == "rank_view":
            for r in range(n):
                chunks = [sl(g, r) for g in gbuf]
                z.zero_fused_step(plan, z.ZERO_RANK_VIEW, chunks, sl(master, r), sl(m, r), sl(v, r), sl(param, r),
                                  hp, t)
        elif mode == "unfused":  # reduce-scatter, then Adam with the cast
            for r in range(n):
                g = offset_buf(S, torch.float32, misalign)
                z.zero_reduce_scatter(plan, r, gbuf, g)
                z.zero_adam_step(plan, r, g, sl(master, r), sl(m, r), sl(v, r), ptarget(r), hp, t)
        elif mode == "unfused_ag":  # reduce-scatter, Adam without cast, then the all-gather
            for r in range(n):
                g = offset_buf(S, torch.float32, misalign)
                z.zero_reduce_scatter(plan, r, gbuf, g)
                z.zero_adam_step(plan, r, g, sl(master, r), sl(m, r), sl(v, r), None, hp, t)
            z.zero_allgather_params(plan, [sl(master, r) for r in range(n)], param)
        elif mode == "ddp":  # all-reduce into a full fp32 gradient, Adam over the whole replica
            g = offset_buf(P, torch.float32, misalign)
            z.ddp_allreduce(plan, gbuf, g)
            z.zero_adam_step(plan, z.ZERO_ALL_RANKS, g, master, m, v, param, hp, t)
        else:
            raise ValueError(mode)
    z.zero_device_status()
    return f32(master), f32(m), f32(v), bits16(param)


def compare(got, want, what):
    for name, a, b in zip(("master", "m", "v"), got[:3], want[:3]):
        assert_f32_identical(a, b, f"{what} {name}")
    assert_bf16_identical(got[3], want[3], f"{what} param")


# ---------------------------------------------------------------------------------------
# small cases: every element, bit for bit
# ---------------------------------------------------------------------------------------

def test_tiny_zero2_vs_ddp_workload(z):
    """psi = 2^20, N = 4, 25 MiB buckets, 3 steps: ZeRO-2 fused vs the oracle's DDP and
    ZeRO-2 runs, plus the GPU DDP path (all-reduce + full-replica Adam)."""
    psi, n, bb = 1_048_576, 4, 25 * MIB
    master0, m0, v0, grads = make_inputs(psi, n, 3)
    want = oracle_run("ddp", psi, n, bb, master0, m0, v0, grads)
    want2 = oracle_run("zero2", psi, n, bb, master0, m0, v0, grads)
    compare(want2, want, "oracle zero2 vs ddp")
    compare(gpu_run(z, "zero2", "all", psi, n, bb, master0, m0, v0, grads), want, "gpu zero2 fused")
    compare(gpu_run(z, "ddp", "ddp", psi, n, bb, master0, m0, v0, grads), want, "gpu ddp")


CASES = [(1, 1, 2), (7, 2, 4), (13, 3, 6), (1000, 8, 48), (100_003, 5, 1 << 12), (65_539, 16, 1 << 14),
         (20_001, 64, 1 << 10), (262_147, 4, 1 << 16),
         (5, 64, 128)]  # psi < N: 59 of the 64 one-element shards are padding


@pytest.mark.parametrize("psi,n,bb", CASES)
@pytest.mark.parametrize("stage,mode", [("zero1", "ranks"), ("zero2", "all"), ("zero2", "all_buckets"),
                                        ("zero2", "buckets"), ("zero2", "rank_view"), ("zero3", "ranks"),
                                        ("zero2", "unfused"), ("zero1", "unfused_ag"), ("ddp", "ddp")])
def test_strategies_and_modes_bit_exact(z, psi, n, bb, stage, mode):
    master0, m0, v0, grads = make_inputs(psi, n, 2, seed=psi + n, moments=True)
    want = oracle_run(stage, psi, n, bb, master0, m0, v0, grads)
    compare(gpu_run(z, stage, mode, psi, n, bb, master0, m0, v0, grads), want, f"{stage}/{mode}")


@pytest.mark.parametrize("psi,n,bb", CASES)
@pytest.mark.parametrize("variant", [1, 2])
def test_kernel_variants_bit_exact(z, psi, n, bb, variant):
    """TMA pipeline (1) and register streaming (2) over aligned buffers; both must equal
    the oracle exactly."""
    z.zero_set_fused_kernel(variant)
    master0, m0, v0, grads = make_inputs(psi, n, 2, seed=7 * psi + n, moments=True)
    want = oracle_run("zero2", psi, n, bb, master0, m0, v0, grads)
    compare(gpu_run(z, "zero2", "all", psi, n, bb, master0, m0, v0, grads), want, f"variant {variant}")
    compare(gpu_run(z, "zero2", "all_buckets", psi, n, bb, master0, m0, v0, grads), want, f"variant {variant} buckets")


@pytest.mark.parametrize("psi,n,bb", [(1000, 8, 48), (100_003, 5, 1 << 12), (20_001, 64, 1 << 10)])
@pytest.mark.parametrize("stage,mode", [("zero2", "all"), ("zero2", "buckets"), ("zero2", "unfused"), ("ddp", "ddp"),
                                        ("zero1", "unfused_ag")])
def test_misaligned_buffers_take_scalar_path_bit_exact(z, psi, n, bb, stage, mode):
    master0, m0, v0, grads = make_inputs(psi, n, 2, seed=3, moments=True)
    want = oracle_run(stage, psi, n, bb, master0, m0, v0, grads)
    compare(gpu_run(z, stage, mode, psi, n, bb, master0, m0, v0, grads, misalign=True), want, f"misaligned {mode}")


def test_weight_decay_and_late_step(z):
    hp = O.AdamHyper(lr=3e-4, beta1=0.8, beta2=0.95, eps=1e-6, weight_decay=0.1)
    psi, n, bb = 30_011, 3, 1 << 12
    master0, m0, v0, grads = make_inputs(psi, n, 1, seed=5, moments=True)
    plan_want = oracle_run("zero2", psi, n, bb, master0, m0, v0, grads, hp=hp)
    compare(gpu_run(z, "zero2", "all", psi, n, bb, master0, m0, v0, grads, hp=hp), plan_want, "wd")
    # t = 1000: bias corrections near 1
    lay = O.make_layout(psi, n, bb)
    plan = z.zero_plan(psi, n, "zero2", bb)
    P = plan.psi_padded
    master, m, v = master0.to(DEV), m0.to(DEV), v0.to(DEV)
    param = torch.zeros(P, dtype=torch.bfloat16, device=DEV)
    gd = [g.to(DEV) for g in grads[0]]
    z.zero_fused_step(plan, z.ZERO_ALL_RANKS, gd, master, m, v, param, hp, 1000)
    w, m1, v1, p = O.fused_step_elements([bits16(g) for g in grads[0]], master0.numpy(), m0.numpy(), v0.numpy(), hp,
                                         1000)
    compare((f32(master), f32(m), f32(v), bits16(param)), (w, m1, v1, p), "t=1000")
    assert lay.psi_padded == P


def test_special_values(z):
    """inf / NaN / denormal gradients and denormal, zero and huge masters: same bits as the
    oracle (NaN compared as NaN)."""
    n, psi = 4, 4096
    rng = np.random.default_rng(0)
    specials = np.array([np.inf, -np.inf, np.nan, 0.0, -0.0, 1e-40, -1e-40, 3e38, -3e38, 1e-45], dtype=np.float32)
    gs = []
    for q in range(n):
        x = rng.normal(0, 1e-3, psi).astype(np.float32)
        x[rng.integers(0, psi, 200)] = rng.choice(specials, 200)
        gs.append(torch.from_numpy(O.f32_to_bf16(x).view(np.int16)).view(torch.bfloat16))
    w0 = rng.normal(0, 0.02, psi).astype(np.float32)
    w0[:10] = specials
    w0[10:20] = np.float32(1e-39)
    master0 = torch.from_numpy(w0)
    m0 = torch.zeros(psi)
    v0 = torch.zeros(psi)
    with np.errstate(over="ignore", invalid="ignore"):  # inf and NaN inputs are the point here
        want = oracle_run("zero2", psi, n, 1 << 12, master0, m0, v0, [gs])
    for variant in (1, 2):
        z.zero_set_fused_kernel(variant)
        compare(gpu_run(z, "zero2", "all", psi, n, 1 << 12, master0, m0, v0, [gs]), want, f"specials v{variant}")
    compare(gpu_run(z, "zero2", "all", psi, n, 1 << 12, master0, m0, v0, [gs], misalign=True), want, "specials scalar")


def test_zero_inputs_keep_padding_zero(z):
    psi, n = 1001, 8  # padded to 1008
    master0, m0, v0, _ = make_inputs(psi, n, 1)
    grads = [[torch.zeros(1008, dtype=torch.bfloat16) for _ in range(n)] for _ in range(3)]
    got = gpu_run(z, "zero3", "ranks", psi, n, 64, master0, m0, v0, grads)
    assert_f32_identical(got[0], master0.numpy(), "master unchanged by zero gradients")
    assert not got[0][psi:].any() and not got[3][psi:].any() and not got[1].any() and not got[2].any()


def test_reduce_scatter_and_allreduce_equal_rs_then_ag(z):
    """all-reduce = reduce-scatter + all-gather, on the GPU, bit for bit, and both equal
    the oracle's definition of the all-reduce."""
    for psi, n in ((100_003, 5), (65_536, 8), (999, 64)):
        plan = z.zero_plan(psi, n, "ddp", 1 << 14)
        P, S = plan.psi_padded, plan.shard_elems
        _, _, _, grads = make_inputs(psi, n, 1, seed=11)
        gd = [g.to(DEV) for g in grads[0]]
        ar = torch.empty(P, device=DEV)
        z.ddp_allreduce(plan, gd, ar)
        parts = []
        for r in range(n):
            g = torch.empty(S, device=DEV)
            z.zero_reduce_scatter(plan, r, gd, g)
            parts.append(g)
        allr = torch.empty(P, device=DEV)
        z.zero_reduce_scatter(plan, z.ZERO_ALL_RANKS, gd, allr)
        lay = O.make_layout(psi, n, 1 << 14)
        want = O.all_reduce(lay, [bits16(g) for g in grads[0]])
        assert_f32_identical(f32(ar), want, "ddp_allreduce")
        assert_f32_identical(f32(torch.cat(parts)), want, "reduce_scatter per rank, concatenated")
        assert_f32_identical(f32(allr), want, "reduce_scatter all ranks")


def test_allgather_params_cast(z):
    psi, n = 50_003, 7
    plan = z.zero_plan(psi, n, "zero1", 1 << 14)
    P, S = plan.psi_padded, plan.shard_elems
    rng = np.random.default_rng(2)
    w = rng.normal(0, 0.02, P).astype(np.float32)
    w[::97] = rng.normal(0, 1e30, w[::97].size)
    masters = [torch.from_numpy(w[r * S:(r + 1) * S].copy()).to(DEV) for r in range(n)]
    full = torch.zeros(P, dtype=torch.bfloat16, device=DEV)
    z.zero_allgather_params(plan, masters, full)
    assert_bf16_identical(bits16(full), O.all_gather([O.f32_to_bf16(w[r * S:(r + 1) * S]) for r in range(n)]),
                          "all-gather cast")


# ---------------------------------------------------------------------------------------
# Megatron distributed optimizer: fp32 gradient contributions
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("psi,n,bb,misalign", [(1_048_576, 4, 25 * MIB, False), (100_003, 5, 1 << 12, False),
                                               (20_001, 64, 1 << 10, False), (65_539, 16, 1 << 14, True),
                                               (13, 3, 6, False)]
                         # every rank count with its own fp32-gradient instance, and 17 (generic)
                         + [(40_009, n, 1 << 14, False) for n in (1, 2, 6, 7, 8, 9, 10, 11, 12, 13, 14, 15, 17)])
def test_megatron_fp32_grads_bit_exact(z, psi, n, bb, misalign):
    P = -(-psi // n) * n
    master0 = synth.master_params(psi, P, seed_key=n)
    m0, v0 = synth.adam_moments(P, seed_key=n)
    m0[psi:] = 0
    v0[psi:] = 0
    steps = [[synth.rank_grads_f32(psi, P, r, t, seed_key=n) for r in range(n)] for t in (1, 2)]
    lay = O.make_layout(psi, n, bb)
    ranks = O.init_ranks("megatron", lay, master0.numpy())
    for r, st in enumerate(ranks):
        lo, hi = O.shard_range(lay, r)
        st.buffers["m"][:] = m0.numpy()[lo:hi]
        st.buffers["v"][:] = v0.numpy()[lo:hi]
    for t, gs in enumerate(steps, start=1):
        O.step_ranks(ranks, lay, [g.numpy() for g in gs], HP, t)
    want = (O.gather_master(ranks, lay), np.concatenate([st.buffers["m"] for st in ranks]),
            np.concatenate([st.buffers["v"] for st in ranks]), O.gather_params(ranks))
    plan = z.zero_plan(psi, n, "megatron", bb)
    assert plan.state_total_bytes == 6 * P + 12 * (P // n)
    for mode in ("all", "ranks"):
        S = plan.shard_elems
        master, m, v = (offset_buf(P, torch.float32, misalign) for _ in range(3))
        param = offset_buf(P, torch.bfloat16, misalign)
        master.copy_(master0)
        m.copy_(m0)
        v.copy_(v0)
        gbuf = [offset_buf(P, torch.float32, misalign) for _ in range(n)]
        for t, gs in enumerate(steps, start=1):
            for q in range(n):
                gbuf[q].copy_(gs[q])
            if mode == "all":
                z.zero_fused_step_fp32_grads(plan, z.ZERO_ALL_RANKS, gbuf, master, m, v, param, HP, t)
            else:
                for r in range(n):
                    sl = slice(r * S, (r + 1) * S)
                    z.zero_fused_step_fp32_grads(plan, r, gbuf, master[sl], m[sl], v[sl], param, HP, t)
        z.zero_device_status()
        compare((f32(master), f32(m), f32(v), bits16(param)), want, f"megatron {mode}")


def test_megatron_gpt2_small_n8_sampled(z):
    """GPT-2-small list, N = 8, fp32 gradients (8 x 497 MB), 2 steps, every rank in one
    launch, against the oracle on sampled indices."""
    psi, n = synth.GPT2_SMALL_PSI, 8
    plan = z.zero_plan(psi, n, "megatron", 25 * MIB)
    P, S, C = plan.psi_padded, plan.shard_elems, plan.bucket_elems
    master = synth.master_params(psi, P, device=DEV)
    m = torch.zeros(P, device=DEV)
    v = torch.zeros(P, device=DEV)
    param = torch.empty(P, dtype=torch.bfloat16, device=DEV)
    idx = sample_indices(P, S, C, n, seed=5)
    idx_t = torch.from_numpy(idx).to(DEV)
    w_s, m_s, v_s = f32(take(master, idx_t)), f32(take(m, idx_t)), f32(take(v, idx_t))
    for t in (1, 2):
        grads = [synth.rank_grads_f32(psi, P, r, t, device=DEV) for r in range(n)]
        gs = [f32(take(g, idx_t)) for g in grads]
        w_s, m_s, v_s, p_s = O.fused_step_elements(gs, w_s, m_s, v_s, HP, t)
        z.zero_fused_step_fp32_grads(plan, z.ZERO_ALL_RANKS, grads, master, m, v, param, HP, t)
        del grads
    z.zero_device_status()
    compare((f32(take(master, idx_t)), f32(take(m, idx_t)), f32(take(v, idx_t)), bits16(take(param, idx_t))),
            (w_s, m_s, v_s, p_s), "megatron gpt2 sampled")


def test_zero1_via_allreduce_equals_zero1(z):
    """ZeRO-1 implemented with a full gradient all-reduce and a parameter all-gather (3 psi
    of communication — [Interview] follow-up on ZeRO-1 vs ZeRO-2 communication) computes the
    same parameters as the reduce-scatter form (2 psi), bit for bit."""
    psi, n, bb = 100_003, 5, 1 << 12
    master0, m0, v0, grads = make_inputs(psi, n, 2, seed=21, moments=True)
    want = oracle_run("zero1", psi, n, bb, master0, m0, v0, grads)
    plan = z.zero_plan(psi, n, "zero1", bb)
    P, S = plan.psi_padded, plan.shard_elems
    master, m, v = master0.to(DEV), m0.to(DEV), v0.to(DEV)
    param = torch.zeros(P, dtype=torch.bfloat16, device=DEV)
    g_full = torch.empty(P, device=DEV)
    for t, gs in enumerate(grads, start=1):
        gd = [g.to(DEV) for g in gs]
        z.ddp_allreduce(plan, gd, g_full)
        for r in range(n):
            sl = slice(r * S, (r + 1) * S)
            z.zero_adam_step(plan, r, g_full[sl], master[sl], m[sl], v[sl], None, HP, t)
        z.zero_allgather_params(plan, [master[r * S:(r + 1) * S] for r in range(n)], param)
    z.zero_device_status()
    compare((f32(master), f32(m), f32(v), bits16(param)), want, "zero1 via all-reduce")


@pytest.mark.parametrize("mode", ["all", "unfused", "ddp"])
@pytest.mark.parametrize("n", range(1, 18))
def test_every_rank_count_bit_exact(z, n, mode):
    """Every rank count with its own kernel instance (N = 1..16) and the first one on the
    generic path (17), for the fused step, the standalone reduce-scatter + Adam, and the DDP
    all-reduce + Adam: two steps over all ranks, bit for bit against the oracle, on an odd
    psi so the padding and the scalar tail are exercised too."""
    psi, bb = 120_001, 1 << 14
    master0, m0, v0, grads = make_inputs(psi, n, 2, seed=40 + n, moments=True)
    want = oracle_run("zero2", psi, n, bb, master0, m0, v0, grads)
    got = gpu_run(z, "zero2", mode, psi, n, bb, master0, m0, v0, grads)
    compare(got, want, f"N={n} mode={mode}")


def test_buckets_in_gradient_ready_order(z):
    """Backward produces gradients last layer first, so DDP reduces buckets in reverse
    order of the flat buffer ([Concepts] "Plain data parallel (DDP)"); launching the
    buckets from last to first must give the same bits as one launch."""
    psi, n, bb = 262_147, 4, 1 << 12
    master0, m0, v0, grads = make_inputs(psi, n, 2, seed=23, moments=True)
    want = oracle_run("zero2", psi, n, bb, master0, m0, v0, grads)
    plan = z.zero_plan(psi, n, "zero2", bb)
    P, NB = plan.psi_padded, plan.n_buckets
    assert NB > 50
    master, m, v = master0.to(DEV), m0.to(DEV), v0.to(DEV)
    param = torch.zeros(P, dtype=torch.bfloat16, device=DEV)
    for t, gs in enumerate(grads, start=1):
        gd = [g.to(DEV) for g in gs]
        for k in reversed(range(NB)):
            z.zero_fused_step_buckets(plan, z.ZERO_ALL_RANKS, k, k + 1, gd, master, m, v, param, HP, t)
    z.zero_device_status()
    compare((f32(master), f32(m), f32(v), bits16(param)), want, "reverse-order buckets")


def test_buckets_on_four_streams_equal_the_oracle(z):
    """Buckets are disjoint, so a caller may launch them on several streams at once (DDP
    overlapping the per-bucket steps): bucket k on stream k % 4, forked from and joined to
    the default stream, over two steps, must match the oracle bit for bit."""
    psi, n, bb = 300_007, 8, 1 << 13
    master0, m0, v0, grads = make_inputs(psi, n, 2, seed=29, moments=True)
    want = oracle_run("zero2", psi, n, bb, master0, m0, v0, grads)
    plan = z.zero_plan(psi, n, "zero2", bb)
    P, NB = plan.psi_padded, plan.n_buckets
    assert NB > 50
    master, m, v = master0.to(DEV), m0.to(DEV), v0.to(DEV)
    param = torch.zeros(P, dtype=torch.bfloat16, device=DEV)
    main = torch.cuda.current_stream()
    side = [torch.cuda.Stream() for _ in range(3)]
    for t, gs in enumerate(grads, start=1):
        gd = [g.to(DEV) for g in gs]
        fork = torch.cuda.Event()
        fork.record(main)
        for s in side:
            s.wait_event(fork)
        streams = [main] + side
        for k in range(NB):
            z.zero_fused_step_buckets(plan, z.ZERO_ALL_RANKS, k, k + 1, gd, master, m, v, param, HP, t,
                                      streams[k % 4])
        for s in side:
            join = torch.cuda.Event()
            join.record(s)
            main.wait_event(join)
    z.zero_device_status()
    compare((f32(master), f32(m), f32(v), bits16(param)), want, "buckets on four streams")


# ---------------------------------------------------------------------------------------
# gradients and parameters in page-locked host memory, read / written over the host link
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("psi,n,bb", [(1_048_576, 4, 25 * MIB), (100_003, 5, 1 << 12), (20_001, 64, 1 << 10)])
def test_host_memory_step_bit_exact(z, psi, n, bb):
    master0, m0, v0, grads = make_inputs(psi, n, 2, seed=41, moments=True)
    want = oracle_run("zero2", psi, n, bb, master0, m0, v0, grads)
    plan = z.zero_plan(psi, n, "zero2", bb)
    P, S = plan.psi_padded, plan.shard_elems
    for mode in ("all", "ranks"):
        master, m, v = master0.to(DEV), m0.to(DEV), v0.to(DEV)
        hparam = torch.zeros(P, dtype=torch.bfloat16).pin_memory()
        for t, gs in enumerate(grads, start=1):
            hg = [g.pin_memory() for g in gs]
            if mode == "all":
                z.zero_fused_step_host(plan, z.ZERO_ALL_RANKS, hg, master, m, v, hparam, HP, t)
            else:
                for r in range(n):
                    sl = slice(r * S, (r + 1) * S)
                    z.zero_fused_step_host(plan, r, hg, master[sl], m[sl], v[sl], hparam, HP, t)
            torch.cuda.synchronize()
        z.zero_device_status()
        compare((f32(master), f32(m), f32(v), bits16(hparam)), want, f"host memory {mode}")


def test_host_memory_step_rejects_pageable_buffers(z):
    import ctypes as C
    plan = z.zero_plan(4096, 2, "zero2", 1 << 12)
    master = torch.zeros(4096, device=DEV)
    pageable = [torch.zeros(4096, dtype=torch.bfloat16) for _ in range(2)]
    hparam = torch.zeros(4096, dtype=torch.bfloat16).pin_memory()
    with pytest.raises(ValueError):
        z.zero_fused_step_host(plan, z.ZERO_ALL_RANKS, pageable, master, master, master, hparam, HP, 1)
    lib = z.library()
    arr = (C.c_void_p * 2)(pageable[0].data_ptr(), pageable[1].data_ptr())
    adam = z._lib.zero_adam(1e-4, 0.9, 0.999, 1e-8, 0.0)
    rc = lib.zero_fused_step_host(plan.handle, z.ZERO_ALL_RANKS, arr, master.data_ptr(), master.data_ptr(),
                                  master.data_ptr(), hparam.data_ptr(), C.byref(adam), 1, None)
    assert rc == -1 and b"page-locked" in lib.zero_last_error()


def test_device_status_is_clean_after_all_kernels(z):
    z.zero_device_status()


# ---------------------------------------------------------------------------------------
# full-size workloads: sampled indices, oracle one element at a time
# ---------------------------------------------------------------------------------------

def sample_indices(P, S, C, n, k=1 << 16, seed=0):
    rng = np.random.default_rng(seed)
    idx = set(rng.integers(0, P, k).tolist())
    for r in range(n + 1):
        for j in (r * S - 1, r * S, r * S + 1):
            if 0 <= j < P:
                idx.add(j)
        for b in range(0, S, C):
            for j in (r * S + b - 1, r * S + b):
                if 0 <= j < P:
                    idx.add(j)
    idx.add(P - 1)
    return np.array(sorted(idx), dtype=np.int64)


def take(t, idx_t):
    return t.index_select(0, idx_t)


class SampledOracle:
    """Tracks master / m / v at sampled flat indices through the oracle's per-element step."""

    def __init__(self, idx, master, m, v):
        self.idx = idx
        self.idx_t = torch.from_numpy(idx).to(DEV)
        self.w, self.m, self.v = f32(take(master, self.idx_t)), f32(take(m, self.idx_t)), f32(take(v, self.idx_t))

    def step(self, grads_dev, t, hp=HP):
        gs = [bits16(take(g, self.idx_t)) for g in grads_dev]
        self.w, self.m, self.v, self.p = O.fused_step_elements(gs, self.w, self.m, self.v, hp, t)

    def check(self, master, m, v, param, what):
        compare((f32(take(master, self.idx_t)), f32(take(m, self.idx_t)), f32(take(v, self.idx_t)),
                 bits16(take(param, self.idx_t))), (self.w, self.m, self.v, self.p), what)


def test_gpt2_small_n8_all_stages_sampled(z):
    """GPT-2-small list (psi = 124,356,864), N = 8, 5 steps. ZeRO-2 in the launch the
    benchmark times (every rank, one fused launch) is checked against the oracle on
    sampled indices; ZeRO-1 (per-rank launches), ZeRO-3 (per-rank shards) and DDP
    (all-reduce + replica Adam) must equal it bit for bit over the whole buffer."""
    psi, n, bb = synth.GPT2_SMALL_PSI, 8, 25 * MIB
    plan = z.zero_plan(psi, n, "zero2", bb)
    P, S, C = plan.psi_padded, plan.shard_elems, plan.bucket_elems
    master0 = synth.master_params(psi, P, device=DEV)
    states = {k: (master0.clone(), torch.zeros(P, device=DEV), torch.zeros(P, device=DEV),
                  master0.to(torch.bfloat16)) for k in ("zero2", "zero1", "zero3", "ddp")}
    plans = {k: z.zero_plan(psi, n, k, bb) for k in states}
    so = SampledOracle(sample_indices(P, S, C, n), *states["zero2"][:3])
    g_full = torch.empty(P, device=DEV)
    sl = lambda t, r: t[r * S:(r + 1) * S]
    for t in range(1, 6):
        grads = [synth.rank_grads(psi, P, r, t, device=DEV) for r in range(n)]
        so.step(grads, t)
        w, m, v, p = states["zero2"]
        z.zero_fused_step(plans["zero2"], z.ZERO_ALL_RANKS, grads, w, m, v, p, HP, t)
        w, m, v, p = states["zero1"]
        for r in range(n):
            z.zero_fused_step(plans["zero1"], r, grads, sl(w, r), sl(m, r), sl(v, r), p, HP, t)
        w, m, v, p = states["zero3"]
        for r in range(n):
            z.zero_fused_step(plans["zero3"], r, grads, sl(w, r), sl(m, r), sl(v, r), sl(p, r), HP, t)
        w, m, v, p = states["ddp"]
        z.ddp_allreduce(plans["ddp"], grads, g_full)
        z.zero_adam_step(plans["ddp"], z.ZERO_ALL_RANKS, g_full, w, m, v, p, HP, t)
        del grads
    z.zero_device_status()
    so.check(*states["zero2"], "gpt2 zero2 sampled")
    ref = states["zero2"]
    for k in ("zero1", "zero3", "ddp"):
        for a, b, name in zip(states[k], ref, ("master", "m", "v", "param")):
            assert torch.equal(a.view(torch.int32) if a.dtype == torch.float32 else a.view(torch.int16),
                               b.view(torch.int32) if b.dtype == torch.float32 else b.view(torch.int16)), (k, name)


def test_mistral7b_rank_view_n8_sampled(z):
    """One rank's view of the Mistral-7B list at N = 8, ZeRO-3, 50 MiB buckets: the 8
    incoming chunks of S = 905,216,512 elements. The single fused launch and the per-bucket
    launches (277 of them) must agree bit for bit and with the oracle at sampled indices."""
    psi, n, bb = synth.MISTRAL_7B_PSI, 8, 50 * MIB
    plan = z.zero_plan(psi, n, "zero3", bb)
    S, C, NB = plan.shard_elems, plan.bucket_elems, plan.n_buckets
    assert (S, NB) == (905_216_512, 277)
    chunks = synth.chunk_grads(S, n, 1, device=DEV)
    rows = [chunks[q] for q in range(n)]
    master = synth.master_params(S, S, device=DEV, seed_key=3)
    m = torch.zeros(S, device=DEV)
    v = torch.zeros(S, device=DEV)
    so = SampledOracle(sample_indices(S, S, C, 1, k=1 << 20, seed=1), master, m, v)  # 2^20 random + every edge
    so.step(rows, 1)
    w2, m2, v2 = master.clone(), m.clone(), v.clone()
    p1 = torch.empty(S, dtype=torch.bfloat16, device=DEV)
    p2 = torch.empty(S, dtype=torch.bfloat16, device=DEV)
    z.zero_fused_step(plan, z.ZERO_RANK_VIEW, rows, master, m, v, p1, HP, 1)
    for k in range(NB):
        z.zero_fused_step_buckets(plan, z.ZERO_RANK_VIEW, k, k + 1, rows, w2, m2, v2, p2, HP, 1)
    z.zero_device_status()
    so.check(master, m, v, p1, "mistral rank view")
    assert torch.equal(master.view(torch.int32), w2.view(torch.int32))
    assert torch.equal(m.view(torch.int32), m2.view(torch.int32))
    assert torch.equal(v.view(torch.int32), v2.view(torch.int32))
    assert torch.equal(p1.view(torch.int16), p2.view(torch.int16))


@pytest.mark.parametrize("n,mode", [(2, "full"), (4, "full"), (8, "full"), (16, "full"), (64, "rank"), (64, "full")])
def test_sweep_1p5b_sampled(z, n, mode):
    """psi = 1.5e9 flat, bf16 grads N(0, 1e-3): full simulation of all N ranks (N = 64 only
    when its 213 GB fit in free device memory with a margin, as the sweep does) or one
    rank's view; sampled against the oracle. Also checks the plan's per-stage model-state
    bytes against the closed forms."""
    psi, bb = 1_500_000_000, 5 * MIB
    plan = z.zero_plan(psi, n, "zero2", bb)
    P, S, C = plan.psi_padded, plan.shard_elems, plan.bucket_elems
    assert P == psi
    for stage, total in (("ddp", 16 * P), ("zero1", 4 * P + 12 * P // n), ("zero2", 2 * P + 14 * P // n),
                         ("zero3", 16 * P // n)):
        assert z.zero_plan(psi, n, stage, bb).state_total_bytes == total
    if mode == "full":
        torch.cuda.empty_cache()
        # the library states the step's need before anything is allocated: (2N + 14) P
        # bytes of gradients, state and parameters, against the free memory less 8 GiB
        free = torch.cuda.mem_get_info()[0]
        try:
            need, budget = z.zero_plan_check_memory(plan, z.ZERO_ALL_RANKS, max(1, free - (8 << 30)))
        except z.ZeroError as e:
            assert e.code == -2 and str((2 * n + 14) * P) in str(e)
            pytest.skip(f"{(2 * n + 14) * P / 1e9:.0f} GB of buffers do not fit in free device memory")
        assert need == (2 * n + 14) * P
        need0, free0 = z.zero_plan_check_memory(plan, z.ZERO_ALL_RANKS)
        assert need0 == need and free0 == free
        grads = [synth.rank_grads(psi, P, r, 1, device=DEV) for r in range(n)]
        master = synth.master_params(psi, P, device=DEV)
        m = torch.zeros(P, device=DEV)
        v = torch.zeros(P, device=DEV)
        param = torch.empty(P, dtype=torch.bfloat16, device=DEV)
        so = SampledOracle(sample_indices(P, S, C, n, seed=n), master, m, v)
        so.step(grads, 1)
        z.zero_fused_step(plan, z.ZERO_ALL_RANKS, grads, master, m, v, param, HP, 1)
    else:
        chunks = synth.chunk_grads(S, n, 1, device=DEV)
        grads = [chunks[q] for q in range(n)]
        master = synth.master_params(S, S, device=DEV)
        m = torch.zeros(S, device=DEV)
        v = torch.zeros(S, device=DEV)
        param = torch.empty(S, dtype=torch.bfloat16, device=DEV)
        so = SampledOracle(sample_indices(S, S, C, 1, seed=n), master, m, v)
        so.step(grads, 1)
        z.zero_fused_step(plan, z.ZERO_RANK_VIEW, grads, master, m, v, param, HP, 1)
    z.zero_device_status()
    so.check(master, m, v, param, f"sweep N={n}")


def test_bounded_wait_runs_out_and_reports(z):
    """A wait that nothing satisfies gives up after its limit and reports through the
    device error word; the context stays usable (a fused step afterwards is still exact)."""
    z.zero_device_status()
    z.zero_selftest_bounded_wait(200)
    with pytest.raises(z.ZeroError) as e:
        z.zero_device_status()
    assert e.value.code == -5 and "0x301" in str(e.value)
    z.zero_device_status()  # the word was cleared
    psi, n = 4099, 4
    master0, m0, v0, grads = make_inputs(psi, n, 1, seed=2)
    want = oracle_run("zero2", psi, n, 1 << 12, master0, m0, v0, grads)
    compare(gpu_run(z, "zero2", "all", psi, n, 1 << 12, master0, m0, v0, grads), want, "after a timed-out wait")


def test_shard_above_2_pow_31_elements(z):
    """One rank's view with S = 2^31 + 4099 elements (byte offsets far beyond 4 GiB, a
    ragged tail): sampled against the oracle, including the last elements."""
    n, S = 2, (1 << 31) + 4099
    plan = z.zero_plan(S * n, n, "zero3", 64 * MIB)
    assert plan.shard_elems == S
    chunks = synth.chunk_grads(S, n, 1, device=DEV, seed_key=9)
    rows = [chunks[q] for q in range(n)]
    master = synth.master_params(S, S, device=DEV, seed_key=9)
    m = torch.zeros(S, device=DEV)
    v = torch.zeros(S, device=DEV)
    p = torch.empty(S, dtype=torch.bfloat16, device=DEV)
    idx = np.unique(np.concatenate([sample_indices(S, S, plan.bucket_elems, 1, k=1 << 14, seed=3),
                                    np.arange(S - 64, S), np.arange((1 << 31) - 32, (1 << 31) + 32)]))
    so = SampledOracle(idx, master, m, v)
    so.step(rows, 1)
    z.zero_fused_step(plan, z.ZERO_RANK_VIEW, rows, master, m, v, p, HP, 1)
    z.zero_device_status()
    so.check(master, m, v, p, "S > 2^31")
