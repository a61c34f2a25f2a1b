"""The binding checks every buffer's length against the plan (or the FSDP shapes) before it
calls the C ABI, whose calls take raw pointers: a short buffer is a Python error and
nothing is launched (the device status stays clean and the buffers untouched)."""
import pytest
import torch

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module")
def z():
    import __graft_entry__ as g
    g.build()
    import fsdp_sharded_optimizer_zero_gb300 as z
    return z


def _step_buffers(P, S, n, state_len, param_len, grad_len):
    grads = [torch.zeros(grad_len, dtype=torch.bfloat16, device=DEV) for _ in range(n)]
    state = [torch.full((state_len,), 7.0, device=DEV) for _ in range(3)]
    param = torch.zeros(param_len, dtype=torch.bfloat16, device=DEV)
    return grads, state, param


@pytest.mark.parametrize("rank,stage,short", [(-2, "zero2", "master"), (-2, "zero2", "grads"), (-1, "zero3", "grads"),
                                              (3, "zero2", "param"), (3, "zero1", "v"), (-1, "zero2", "param")])
def test_short_step_buffers_are_rejected_before_launch(z, rank, stage, short):
    n, psi = 4, 10_000
    plan = z.zero_plan(psi, n, stage, 1 << 16)
    P, S = plan.psi_padded, plan.shard_elems
    full = rank == z.ZERO_ALL_RANKS
    g_len = S if rank == z.ZERO_RANK_VIEW else P
    s_len = P if full else S
    p_len = S if rank == z.ZERO_RANK_VIEW or (stage == "zero3" and rank >= 0) else P
    grads, (w, m, v), p = _step_buffers(P, S, n, s_len - (short in ("master", "v")),
                                        p_len - (short == "param"), g_len)
    if short == "grads":
        grads[1] = grads[1][:-1]
    z.zero_device_status()
    with pytest.raises(ValueError, match="needs at least"):
        z.zero_fused_step(plan, rank, grads, w, m, v, p, {"lr": 1e-3}, 1)
    z.zero_device_status()
    assert torch.all(w == 7.0) and torch.all(v == 7.0)


def test_rank_r_param_shard_rule(z):
    """rank = r writes its bf16 slice into the full buffer under ZeRO-1/2 but into its own
    S-element shard under ZeRO-3: an S-element param_out is enough only for ZeRO-3."""
    n, psi = 4, 10_000
    for stage, ok in (("zero3", True), ("zero2", False)):
        plan = z.zero_plan(psi, n, stage, 1 << 16)
        P, S = plan.psi_padded, plan.shard_elems
        grads, (w, m, v), p = _step_buffers(P, S, n, S, S, P)
        if ok:
            z.zero_fused_step(plan, 1, grads, w, m, v, p, {"lr": 1e-3}, 1)
            z.zero_device_status()
        else:
            with pytest.raises(ValueError):
                z.zero_fused_step(plan, 1, grads, w, m, v, p, {"lr": 1e-3}, 1)


def test_wrong_rank_count_is_rejected(z):
    plan = z.zero_plan(1000, 4, "zero2", 1 << 16)
    P = plan.psi_padded
    grads, (w, m, v), p = _step_buffers(P, P, 3, P, P, P)
    with pytest.raises(ValueError, match="rank buffers"):
        z.zero_fused_step(plan, z.ZERO_ALL_RANKS, grads, w, m, v, p, {"lr": 1e-3}, 1)


def test_fsdp_shapes_are_checked(z):
    shards = [torch.zeros(256, 64, dtype=torch.bfloat16, device=DEV) for _ in range(2)]
    A = torch.zeros(128, 64, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(ValueError, match="needs at least"):
        z.fsdp_unit_forward(shards, A, torch.empty(128, 511, device=DEV))
    with pytest.raises(ValueError, match="one shape"):
        z.fsdp_unit_forward([shards[0], shards[1][:128]], A, torch.empty(128, 512, device=DEV))
    with pytest.raises(ValueError, match="A must be"):
        z.fsdp_unit_forward(shards, torch.zeros(128, 32, dtype=torch.bfloat16, device=DEV),
                            torch.empty(128, 512, device=DEV))
    with pytest.raises(ValueError, match="w_full"):
        z.fsdp_gather_rows(shards, torch.empty(511, 64, dtype=torch.bfloat16, device=DEV))
    with pytest.raises(ValueError, match="needs at least"):
        z.fsdp_transpose_cat(shards, torch.empty(64, 511, dtype=torch.bfloat16, device=DEV))
    dY = [torch.zeros(64, 512, dtype=torch.bfloat16, device=DEV) for _ in range(2)]
    Xs = [torch.zeros(64, 64, dtype=torch.bfloat16, device=DEV) for _ in range(2)]
    dX = [torch.empty(64, 64, device=DEV), torch.empty(64, 63, device=DEV)]
    ws = torch.empty(z.fsdp_unit_backward_workspace(2, 512, 64, 64), dtype=torch.uint8, device=DEV)
    with pytest.raises(ValueError, match="dX"):
        z.fsdp_unit_backward(shards, Xs, dY, dX, torch.empty(512, 64, device=DEV), ws)
    z.zero_device_status()
