"""A first use of the library: one fused ZeRO-2 step of every rank over the GPT-2-small
parameter count (8 ranks), then an FSDP unit forward with W gathered inside the GEMM's
loads. Zero inputs, so the update and the output are exactly zero. Run with
`python -m fsdp_sharded_optimizer_zero_gb300.example` on a GPU."""
import torch

import fsdp_sharded_optimizer_zero_gb300 as z


def main():
    n, psi = 8, 124_356_864
    plan = z.zero_plan(psi, n, "zero2", 25 << 20)   # padded length P, shard S, buckets
    P = plan.psi_padded
    grads = [torch.zeros(P, dtype=torch.bfloat16, device="cuda") for _ in range(n)]  # each rank's flat gradient
    master, m, v = (torch.zeros(P, device="cuda") for _ in range(3))
    param = torch.empty(P, dtype=torch.bfloat16, device="cuda")
    hp = {"lr": 1e-4, "beta1": 0.9, "beta2": 0.999, "eps": 1e-8, "weight_decay": 0.0}
    z.zero_fused_step(plan, z.ZERO_ALL_RANKS, grads, master, m, v, param, hp, step=1)
    z.zero_device_status()   # synchronises; raises ZeroError if a device-side check fired

    # FSDP unit: Y = X W^T, W held as 8 row shards and gathered inside the GEMM's loads
    shards = [torch.zeros(1792, 4096, dtype=torch.bfloat16, device="cuda") for _ in range(8)]
    X = torch.zeros(8192, 4096, dtype=torch.bfloat16, device="cuda")
    Y = torch.empty(8192, 14336, device="cuda")
    z.fsdp_unit_forward(shards, X, Y)
    z.zero_device_status()
    return master, param, Y


if __name__ == "__main__":
    main()
