"""Host-side tests of the C ABI (no GPU): the library loads and exports every entry point
include/zero.h declares; the plan's layout, per-stage bytes and communication counts equal
the oracle's exactly; invalid arguments are rejected before anything is launched."""
from __future__ import annotations

import ctypes as C
import re
from pathlib import Path

import pytest

import oracle.zero_oracle as O

ROOT = Path(__file__).resolve().parents[1]


@pytest.fixture(scope="module")
def z():
    import __graft_entry__ as g
    g.build()
    import fsdp_sharded_optimizer_zero_gb300 as z
    return z


def declared_symbols():
    names = set()
    for h in (ROOT / "include").glob("*.h"):
        names |= set(re.findall(r"^ZERO_API\s+[\w\s\*]+?\b(\w+)\s*\(", h.read_text(), flags=re.M))
    return names


def test_header_declares_the_boundary():
    want = {"zero_plan", "zero_plan_query", "zero_plan_destroy", "zero_reduce_scatter", "zero_adam_step",
            "zero_fused_step", "zero_allgather_params", "ddp_allreduce", "fsdp_unit_forward"}
    assert want <= declared_symbols()


def test_library_exports_every_declared_symbol(z):
    lib = C.CDLL(str(z.LIB_PATH))
    names = declared_symbols()
    assert names == set(z.EXPORTS)
    for name in names:
        assert hasattr(lib, name), name


STAGES = ["ddp", "zero1", "zero2", "zero3", "megatron"]


@pytest.mark.parametrize("psi,n,bb", [(1, 1, 2), (7, 2, 4), (13, 3, 6), (1000, 8, 40), (1_000_003, 64, 1 << 20),
                                      (1_048_576, 4, 25 << 20), (124_356_864, 8, 25 << 20),
                                      (7_241_732_096, 8, 50 << 20), (1_500_000_000, 64, 1 << 20)])
@pytest.mark.parametrize("stage", STAGES)
def test_plan_matches_oracle(z, psi, n, bb, stage):
    p = z.zero_plan(psi, n, stage, bb)
    lay = O.make_layout(psi, n, bb)
    L = p.layout
    assert (L["psi"], L["psi_padded"], L["shard_elems"], L["bucket_elems"], L["n_buckets"]) == \
        (lay.psi, lay.psi_padded, lay.shard, lay.bucket_elems, lay.n_buckets)
    mb = O.model_state_bytes(stage, lay)
    assert (L["state_param_bytes"], L["state_grad_bytes"], L["state_master_bytes"], L["state_m_bytes"],
            L["state_v_bytes"], L["state_total_bytes"]) == (mb["param"], mb["grad"], mb["master"], mb["m"], mb["v"],
                                                            mb["total"])
    c = O.comm_elements(stage, lay)
    assert (L["comm_reduce_scatter"], L["comm_all_gather_fwd"], L["comm_all_gather_bwd"], L["comm_total"]) == \
        (c["reduce_scatter"], c["all_gather_fwd"], c["all_gather_bwd"], c["total"])
    assert L["ring_sent_elems"] == O.ring_sent_elements(c["total"], n)
    grad_bytes = 4 if stage == "megatron" else 2
    assert L["fused_step_bytes"] == lay.psi_padded * (grad_bytes * n + 26)


def test_plan_matches_oracle_on_random_sizes(z):
    """400 seeded (psi, N, bucket bytes, stage) draws, psi from 1 to 2^40 on a log scale,
    N from 1 to 64, buckets from 2N bytes (one element per rank) to 4 GiB: layout, bytes and
    counts equal the oracle's, and the first, last and a middle bucket of the first and
    last rank equal its bucket ranges."""
    import numpy as np
    rng = np.random.default_rng(20261202)
    for _ in range(400):
        psi = int(np.exp(rng.uniform(0.0, 40.0 * np.log(2.0))))
        psi = max(psi, 1)
        n = int(rng.integers(1, 65))
        bb = int(rng.integers(2 * n, (4 << 30) + 1))
        stage = STAGES[int(rng.integers(0, len(STAGES)))]
        p = z.zero_plan(psi, n, stage, bb)
        lay = O.make_layout(psi, n, bb)
        L = p.layout
        case = (psi, n, bb, stage)
        assert (L["psi_padded"], L["shard_elems"], L["bucket_elems"], L["n_buckets"]) == \
            (lay.psi_padded, lay.shard, lay.bucket_elems, lay.n_buckets), case
        mb = O.model_state_bytes(stage, lay)
        assert L["state_total_bytes"] == mb["total"], case
        c = O.comm_elements(stage, lay)
        assert L["comm_total"] == c["total"], case
        for r in {0, n - 1}:
            for k in {0, lay.n_buckets // 2, lay.n_buckets - 1}:
                assert z.zero_bucket_range(p, r, k) == O.bucket_range(lay, r, k), case


@pytest.mark.parametrize("psi,n,bb", [(13, 3, 6), (1000, 8, 48), (4099, 5, 1 << 10)])
def test_bucket_ranges_match_oracle(z, psi, n, bb):
    p = z.zero_plan(psi, n, "zero2", bb)
    lay = O.make_layout(psi, n, bb)
    for r in range(n):
        for k in range(lay.n_buckets):
            assert z.zero_bucket_range(p, r, k) == O.bucket_range(lay, r, k)
    with pytest.raises(z.ZeroError):
        z.zero_bucket_range(p, n, 0)
    with pytest.raises(z.ZeroError):
        z.zero_bucket_range(p, 0, lay.n_buckets)


@pytest.mark.parametrize("args", [(0, 4, 2, 1 << 20), (10, 0, 2, 1 << 20), (10, 65, 2, 1 << 20), (10, 4, 5, 1 << 20),
                                  (10, 4, -1, 1 << 20), (10, 4, 2, 7)])
def test_plan_rejects_bad_arguments(z, args):
    with pytest.raises(z.ZeroError) as e:
        z.zero_plan(*args)
    assert e.value.code == -1


def test_step_calls_reject_missing_rank_before_launch(z):
    """A NULL among the N rank pointers (a missing replica) is an argument error: nothing
    is launched, so this runs without a GPU."""
    lib = z.library()
    p = z.zero_plan(1024, 4, "zero2", 1 << 20)
    grads = (C.c_void_p * 4)(16, 32, None, 64)
    adam = z._lib.zero_adam(1e-4, 0.9, 0.999, 1e-8, 0.0)
    rc = lib.zero_fused_step(p.handle, 0, grads, 256, 512, 768, 1024, C.byref(adam), 1, None)
    assert rc == -1 and b"grads[2] is NULL" in lib.zero_last_error()
    rc = lib.zero_reduce_scatter(p.handle, 0, grads, 256, None)
    assert rc == -1
    rc = lib.ddp_allreduce(p.handle, grads, 256, None)
    assert rc == -1
    good = (C.c_void_p * 4)(16, 32, 48, 64)
    for bad_rank in (4, -3):
        assert lib.zero_fused_step(p.handle, bad_rank, good, 256, 512, 768, 1024, C.byref(adam), 1, None) == -1
    assert lib.zero_fused_step(p.handle, 0, good, 256, 512, 768, 1024, C.byref(adam), 0, None) == -1  # step 0
    bad_adam = z._lib.zero_adam(1e-4, 1.0, 0.999, 1e-8, 0.0)
    assert lib.zero_fused_step(p.handle, 0, good, 256, 512, 768, 1024, C.byref(bad_adam), 1, None) == -1
    assert lib.zero_fused_step_buckets(p.handle, 0, 1, 1, good, 256, 512, 768, 1024, C.byref(adam), 1, None) == -1
    assert lib.fsdp_unit_forward(3, good, 8, 16, 128, 4, 256, None, None, None) == -1   # rows % N
    assert lib.fsdp_unit_forward(4, good, 8, 12, 128, 4, 256, None, None, None) == -1   # k % 8
    assert lib.fsdp_gather_rows(4, grads, 8, 16, 256, None) == -1
    assert lib.zero_set_fused_kernel(3) == -1
    assert lib.zero_set_gemm_kernel(3) == -1 and lib.zero_set_gemm_kernel(-1) == -1
    assert lib.zero_set_gemm_kernel(2) == 0 and lib.zero_set_gemm_kernel(1) == 0 and lib.zero_set_gemm_kernel(0) == 0
    # host-memory step: a buffer that is not page-locked host memory is rejected before launch
    import numpy as np
    buf = np.zeros(1024, np.uint16)
    hosts = (C.c_void_p * 4)(*([buf.ctypes.data] * 4))
    assert lib.zero_fused_step_host(p.handle, -2, hosts, 256, 512, 768, buf.ctypes.data, C.byref(adam), 1, None) == -1


def test_newer_entry_points_reject_bad_arguments_before_launch(z):
    """fp32-gradient step, FSDP backward, MLP unit, static-scratch forward and the self-test:
    argument errors come back as ZERO_ERR_INVALID_ARG with nothing launched."""
    lib = z.library()
    adam = z._lib.zero_adam(1e-4, 0.9, 0.999, 1e-8, 0.0)
    p = z.zero_plan(1024, 4, "megatron", 1 << 20)
    assert p.state_total_bytes == 6 * 1024 + 12 * 256
    grads = (C.c_void_p * 4)(16, 32, None, 64)
    assert lib.zero_fused_step_fp32_grads(p.handle, 0, grads, 256, 512, 768, 1024, C.byref(adam), 1, None) == -1
    assert b"grads[2] is NULL" in lib.zero_last_error()
    good = (C.c_void_p * 4)(16, 32, 48, 64)
    assert lib.zero_fused_step_fp32_grads(p.handle, 4, good, 256, 512, 768, 1024, C.byref(adam), 1, None) == -1
    # backward: rows % N, K % 8, workspace size, NULL rank pointer
    ws = C.c_uint64()
    # every operand read in place (R/N, K and M multiples of 64, N <= 16): no workspace;
    # otherwise W^T, dY^T, X^T
    assert lib.fsdp_unit_backward_workspace(4, 512, 256, 128, C.byref(ws)) == 0
    assert ws.value == 0
    assert lib.fsdp_unit_backward_workspace(4, 512, 256, 40, C.byref(ws)) == 0
    assert ws.value == 2 * 512 * 256 + 2 * 512 * 160 + 2 * 256 * 160
    assert lib.fsdp_unit_backward_workspace(17, 17 * 64, 256, 128, C.byref(ws)) == 0
    assert ws.value > 2 * 256 * 17 * 128  # more than 16 ranks: one GEMM operand cannot hold every piece
    assert lib.fsdp_unit_backward_workspace(4, 512, 192, 128, C.byref(ws)) == 0
    assert ws.value == 0
    assert lib.fsdp_unit_backward_workspace(4, 512, 200, 128, C.byref(ws)) == 0
    assert ws.value > 2 * 200 * 512  # K not a multiple of 64
    assert lib.fsdp_unit_backward_workspace(0, 512, 256, 128, C.byref(ws)) == -1
    args = lambda rows, k, m, wsb: (4, good, rows, k, good, good, m, good, 4096, 8192, wsb, None)
    assert lib.fsdp_unit_backward(*args(510, 256, 128, 1 << 30)) == -1
    assert lib.fsdp_unit_backward(*args(512, 252, 128, 1 << 30)) == -1
    assert lib.fsdp_unit_backward(*args(512, 256, 40, 100)) == -1
    assert b"workspace" in lib.zero_last_error()
    assert lib.fsdp_unit_backward(4, good, 512, 256, good, good, 40, good, 4096, None, 1 << 30, None) == -1
    assert b"workspace" in lib.zero_last_error()
    assert lib.fsdp_unit_backward(4, grads, 512, 256, good, good, 128, good, 4096, 8192, 1 << 30, None) == -1
    # MLP unit: d_model / d_ff multiples of N and of 8, aligned buffers
    assert lib.fsdp_mlp_forward(4, good, good, good, 4096, 14330, 4096, 8, 4096, 4096, None, None, None) == -1
    assert lib.fsdp_mlp_forward(4, good, good, grads, 4096, 14336, 4096, 8, 4096, 4096, None, None, None) == -1
    assert lib.fsdp_mlp_forward(4, good, good, good, 4096, 14336, 4097, 8, 4096, 4096, None, None, None) == -1
    # static scratch: weights above 8,388,608 elements whose shards (2 x 2056 rows) do not
    # tile the GEMM, so they would need the array
    assert lib.fsdp_unit_forward_static_scratch(2, good, 4112, 4104, 4096, 128, 8192, None, None) == -1
    assert b"static scratch" in lib.zero_last_error()
    # self-test limit
    assert lib.zero_selftest_bounded_wait(0, None) == -1
    assert lib.zero_selftest_bounded_wait(5000, None) == -1


def buffer_bytes(plan, rank):
    """Bytes of the buffers one step call addresses, summed from the pointer conventions of
    include/zero.h buffer by buffer (gradients, master, m, v, parameters)."""
    P, S, n = plan.psi_padded, plan.shard_elems, plan.n_ranks
    gbytes = 4 if plan.stage == 4 else 2
    if rank == z_ALL:
        bufs = [(P, gbytes)] * n + [(P, 4)] * 3 + [(P, 2)]
    elif rank == z_VIEW:
        bufs = [(S, gbytes)] * n + [(S, 4)] * 3 + [(S, 2)]
    else:
        bufs = [(P, gbytes)] * n + [(S, 4)] * 3 + [(S if plan.stage == 3 else P, 2)]
    return sum(e * b for e, b in bufs)


z_ALL, z_VIEW = -2, -1


@pytest.mark.parametrize("psi,n,stage", [(1000, 8, "zero2"), (7, 3, "zero3"), (1_500_000_000, 64, "zero2"),
                                         (7_241_732_096, 8, "zero3"), (124_356_864, 8, "megatron"),
                                         (124_356_864, 8, "ddp")])
def test_memory_check_counts_the_step_buffers(z, psi, n, stage):
    plan = z.zero_plan(psi, n, stage, 1 << 20)
    for rank in (z_ALL, z_VIEW, 0, n - 1):
        want = buffer_bytes(plan, rank)
        need, budget = z.zero_plan_check_memory(plan, rank, want)
        assert (need, budget) == (want, want)
        with pytest.raises(z.ZeroError) as e:
            z.zero_plan_check_memory(plan, rank, want - 1)
        assert e.value.code == -2 and str(want) in str(e.value)


def test_memory_check_mistral_ddp_does_not_fit_an_80gb_gpu(z):
    # [Wiring] "Fully Sharded Data Parallel (FSDP)": Mistral-7B ran out of memory under DDP
    # on 80 GB GPUs. A DDP rank holds the whole model state, 16 bytes per parameter (one
    # rank of a one-rank plan addresses exactly that), while a ZeRO-3 rank's view at N = 4
    # (its shard plus the 4 incoming gradient chunks) fits.
    budget = 80 * 10**9
    ddp = z.zero_plan(7_241_732_096, 1, "ddp", 50 << 20)
    with pytest.raises(z.ZeroError) as e:
        z.zero_plan_check_memory(ddp, 0, budget)
    assert e.value.code == -2
    assert buffer_bytes(ddp, 0) == 16 * 7_241_732_096 == ddp.state_total_bytes
    z3 = z.zero_plan(7_241_732_096, 4, "zero3", 50 << 20)
    need, _ = z.zero_plan_check_memory(z3, z_VIEW, budget)
    assert need == (2 * 4 + 14) * z3.shard_elems < budget


def test_memory_check_rejects_bad_rank(z):
    plan = z.zero_plan(1000, 4, "zero2", 1 << 20)
    with pytest.raises(z.ZeroError) as e:
        z.zero_plan_check_memory(plan, 4, 1 << 30)
    assert e.value.code == -1


def test_zero3_step_rejects_bad_arguments_before_launch(z):
    """fsdp_zero3_step validates every unit, the chain, the plans, the flags, the Adam
    arguments and the workspace before anything is launched (fake device addresses)."""
    lib = z.library()
    S = z._lib.fsdp_unit_state
    adam = z._lib.zero_adam(1e-4, 0.9, 0.999, 1e-8, 0.0)
    n, m = 4, 64

    def units(shapes, plans=None, fill=0x10000):
        arr = (S * len(shapes))()
        for i, (r, k) in enumerate(shapes):
            arr[i].rows_out, arr[i].k_in = r, k
            arr[i].plan = plans[i].handle if plans else None
            for j, name in enumerate(("w", "master", "m", "v", "x", "dy", "dw")):
                setattr(arr[i], name, fill + 0x1000 * (8 * i + j))
        return arr

    good = [(512, 256), (1024, 512)]
    plans = [z.zero_plan(r * k, n, "zero3", 1 << 20) for r, k in good]
    ws = C.c_uint64()
    # nothing with the fused gather (every backward operand read in place); with the
    # materialised gather one slot for the largest unit's W, two with the backward prefetch
    assert lib.fsdp_zero3_step_workspace(n, 2, units(good), m, 0, C.byref(ws)) == 0
    assert ws.value == 0
    assert lib.fsdp_zero3_step_workspace(n, 2, units(good), m, 2, C.byref(ws)) == 0
    assert ws.value == 0
    assert lib.fsdp_zero3_step_workspace(n, 2, units(good), m, 1, C.byref(ws)) == 0
    assert ws.value == 2 * 1024 * 512
    assert lib.fsdp_zero3_step_workspace(n, 2, units(good), m, 3, C.byref(ws)) == 0
    assert ws.value == 2 * (2 * 1024 * 512)

    def call(arr, nu=2, flags=0, wsb=1 << 30, step=1, hp=adam, mm=m, nr=n):
        return lib.fsdp_zero3_step(nr, nu, arr, mm, None, None, C.byref(hp), step, flags, 0x100000, wsb, None, None)

    # chain: unit 1's k_in must be unit 0's rows_out
    assert call(units([(512, 256), (1024, 256)], plans)) == -1
    assert b"is not unit 0's rows_out" in lib.zero_last_error()
    # rows_out / N and k_in multiples of 64 (the backward reads W's shards, dY and X as
    # MN-major operands)
    assert call(units([(512, 252), (1024, 512)], plans)) == -1
    assert b"multiple of 64" in lib.zero_last_error()
    assert call(units([(4 * 72, 256)], plans[:1]), nu=1) == -1
    assert b"multiple of 64" in lib.zero_last_error()
    # shards of 64 rows do not tile the fused gather: FSDP_GATHER_MATERIALIZE needed
    p64 = [z.zero_plan(256 * 256, n, "zero3", 1 << 20)]  # kept alive: destroying a plan clears the message
    assert call(units([(256, 256)], p64), nu=1) == -1
    assert b"FSDP_GATHER_MATERIALIZE" in lib.zero_last_error()
    # plan must describe the unit: psi = R K, N ranks, ZeRO-3
    assert call(units(good, [plans[1], plans[0]])) == -1
    assert b"plan" in lib.zero_last_error()
    p2 = [z.zero_plan(512 * 256, n, "zero2", 1 << 20), plans[1]]
    assert call(units(good, p2)) == -1
    assert call(units(good)) == -1                               # no plans
    assert call(units(good, plans, fill=0x10008)) == -1          # misaligned buffers
    assert call(units(good, plans), flags=16) == -1              # unknown flag
    assert call(units(good, plans), step=0) == -1                # Adam step counts from 1
    bad = z._lib.zero_adam(1e-4, 1.0, 0.999, 1e-8, 0.0)
    assert call(units(good, plans), hp=bad) == -1                # beta1 outside [0, 1)
    assert call(units(good, plans), flags=1, wsb=100) == -1      # workspace too small (materialised gather)
    assert b"workspace" in lib.zero_last_error()
    assert call(units(good, plans), nr=17) == -1                 # at most 16 ranks
    assert call(units(good, plans), mm=3) == -1                  # N M a multiple of 8
    assert call(units(good, plans), nu=0) == -1


def test_zero3_mlp_step_workspace_sizes(z):
    """The MLP step reads every backward operand in place up to 8 ranks (no workspace);
    past 8 the 2N shards of [W_gate; W_up] exceed the GEMM's 16 pieces and the largest
    unit's [W_gate; W_up] is gathered into the workspace (4 d_ff d_model bytes)."""
    assert z.fsdp_zero3_mlp_step_workspace(8, [(4096, 14336)] * 2, 1024) == 0
    assert z.fsdp_zero3_mlp_step_workspace(2, [(256, 1024)] * 3, 64) == 0
    assert z.fsdp_zero3_mlp_step_workspace(12, [(1536, 1536)], 16) == 4 * 1536 * 1536
    assert z.fsdp_zero3_mlp_step_workspace(16, [(2048, 2048), (2048, 4096)], 16) == 4 * 4096 * 2048
