"""Benchmark of the fused ZeRO optimizer step on GB300.

Default workload: one rank's view of the Mistral-7B parameter list (7,241,732,096
parameters) at N = 8 simulated data-parallel ranks, ZeRO-3, 50 MiB buckets. The rank owns
a 905,216,512-element shard; it holds the shard's fp32 master / m / v and receives the 8
ranks' bf16 gradient chunks for it. One step = one launch of the fused reduce-scatter +
Adam + bf16 cast over the whole shard (all 277 buckets): it reads the 8 chunks and master /
m / v and writes master / m / v and the bf16 shard, S * (2N + 26) = 38.02 GB of HBM traffic
per step, ~300x the 129 MB L2, so no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--sweep]

Prints ONE JSON line (rank 0). Under torchrun each rank runs an independent replica on
its own GPU (the simulated ranks live on one GPU; there is no inter-GPU exchange), and
`value` is the parameters all GPUs updated per second over the slowest rank's time.
--impl reference times the CPU oracle on the host cores on a bounded sample of the same
workload. --sweep prints one line per point of the 1.5B-parameter bandwidth sweep.
"""
from __future__ import annotations

import os

# Each oracle call (cpu_baseline, the reference arm, the timings beside each leg) runs on
# one host thread; cpu_baseline and the reference arm run one such call per core on
# disjoint ranges. Pin numpy's BLAS before numpy is first imported, so the cores they
# report are exact.
os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")

import argparse
import hashlib
import json
import statistics
import subprocess
import sys
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = "fused ZeRO step params/s and HBM GB/s (% of GB300 peak), 1 GPU"
UNIT = "params/s"
MIB = 1 << 20
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


HP = {"lr": 1e-4, "beta1": 0.9, "beta2": 0.999, "eps": 1e-8, "weight_decay": 0.0}


def workload_config(psi, n, stage, bb, shard):
    """The bench line's workload: one rank's view of the Mistral-7B list (its shard of
    `shard` elements and the n incoming gradient chunks for it)."""
    return {
        "workload": f"Mistral-7B parameter list ({psi:,} params), one rank's view at N={n} simulated data-parallel "
                    f"ranks, {stage.upper()}: fused reduce-scatter + Adam + bf16 cast over the rank's {shard:,}-element "
                    f"shard from the {n} incoming bf16 gradient chunks, {bb // MIB} MiB buckets, all buckets in one "
                    "launch per step",
        "psi": psi, "n_ranks": n, "stage": stage, "bucket_bytes": bb, "shard_elems": shard,
        "adam": HP, "grads": "bf16 N(0,1e-3) per incoming chunk", "master": "fp32 N(0,0.02)",
        "l2": f"inputs larger than L2 ({shard * (2 * n + 26) / 1e9:.2f} GB per step vs 129 MB L2): no flush",
    }


def gpt2_config(psi, n, stage, bb):
    return {
        "workload": f"GPT-2-small parameter list ({psi:,} params) flattened, N={n} simulated data-parallel ranks, "
                    f"{stage.upper()} fused reduce-scatter + Adam + bf16 param all-gather, {bb // MIB} MiB buckets, "
                    "every rank's shard in one launch per step",
        "psi": psi, "n_ranks": n, "stage": stage, "bucket_bytes": bb,
    }


# ---------------------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        mhz, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                mhz.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not mhz:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(mhz)}


# ---------------------------------------------------------------------------------------
# traffic from the committed ncu summary (valid only while the kernel source is unchanged)
# ---------------------------------------------------------------------------------------

def kernel_source_digest():
    h = hashlib.sha256()
    for name in ("fused_step.cu", "step_common.cuh", "device_common.cuh"):
        h.update((ROOT / "fsdp_sharded_optimizer_zero_gb300" / "csrc" / name).read_bytes())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, units: float, mode: str = "all_ranks"):
    """dram read + write bytes per launch of `kernel` in rank mode `mode` from
    profiles/ncu_traffic.txt, scaled to this launch by the units (parameters) it processes,
    or None when absent or taken on other source."""
    p = ROOT / "profiles" / "ncu_traffic.txt"
    if not p.exists():
        return None
    for line in p.read_text().splitlines():
        if line.startswith("#") or not line.strip():
            continue
        f = dict(kv.split("=", 1) for kv in line.split() if "=" in kv)
        if (f.get("kernel") == kernel and f.get("mode", "all_ranks") == mode
                and f.get("source") == kernel_source_digest()):
            return float(f["dram_bytes_per_unit"]) * units
    return None


# ---------------------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------------------

def init_dist(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return world, rank, local


def max_over_ranks(x: float, world: int) -> float:
    """The largest x over all ranks (the slowest rank's time). Host bookkeeping only: NCCL
    on the GPU machine, gloo in the CPU tests."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, steps: int, world: int, seconds_max: float) -> float:
    """Whole-job throughput of N independent replicas: every rank's units over the slowest
    rank's time."""
    return world * units_per_rank * steps / seconds_max


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def mistral_rank_view(z, synth, dev):
    """The bench workload on the device: the plan, the 8 incoming bf16 chunks for the
    rank's shard, fp32 master / m / v and the bf16 shard out (27.2 GB)."""
    import torch
    psi, n, stage, bb = synth.MISTRAL_7B_PSI, 8, "zero3", 50 * MIB
    plan = z.zero_plan(psi, n, stage, bb)
    S = plan.shard_elems
    ch = synth.chunk_grads(S, n, 1, device=dev)
    st = {"plan": plan, "psi": psi, "n": n, "stage": stage, "bb": bb, "S": S, "chunks": ch,
          "grads": [ch[q] for q in range(n)], "master": synth.master_params(S, S, device=dev),
          "m": torch.zeros(S, device=dev), "v": torch.zeros(S, device=dev),
          "param": torch.empty(S, dtype=torch.bfloat16, device=dev)}
    return st


def run_ours(args):
    import torch

    import fsdp_sharded_optimizer_zero_gb300 as z
    import synth

    world, rank, local = init_dist(args)
    dev = torch.device("cuda", torch.cuda.current_device())
    hbm_peak, tf_burst, tf_sust, peak_src = peaks()
    w = mistral_rank_view(z, synth, dev)
    plan, n, S = w["plan"], w["n"], w["S"]
    bytes_per_step = S * (2 * n + 26)
    stream = torch.cuda.current_stream()
    step_no = 0

    def step():
        nonlocal step_no
        step_no += 1
        z.zero_fused_step(plan, z.ZERO_RANK_VIEW, w["grads"], w["master"], w["m"], w["v"], w["param"], HP, step_no,
                          stream)

    for _ in range(args.warmup):
        step()
    z.zero_device_status(stream)
    torch.cuda.synchronize()
    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        t0.record(stream)
        for i in range(K):
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        t1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    z.zero_device_status(stream)
    ms_total = max_over_ranks(t0.elapsed_time(t1), world)
    ms_step = ms_total / K
    launch_ms = statistics.fmean(s.elapsed_time(e) for s, e in zip(starts, ends))
    value = job_throughput(S, K, world, ms_total / 1e3)
    achieved = bytes_per_step / (launch_ms / 1e3) / 1e9
    clocks = clk.summary()

    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded; Mistral-7B parameter count and shard layout, random values; no dataset, no "
                "weights)",
        "config": workload_config(w["psi"], n, w["stage"], w["bb"], S),
        "hbm_gbs": bytes_per_step * K * world / (ms_total / 1e3) / 1e9,
        "hbm_pct_of_peak": 100.0 * (bytes_per_step * K / (ms_total / 1e3) / 1e9) / hbm_peak,
        "roofline": {"bound": "hbm", "kernel": "fused_vec_kernel<8>", "achieved": achieved, "peak": hbm_peak,
                     "unit": "GB/s", "frac": achieved / hbm_peak, "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_src == "measured" else "fallback 6.8 TB/s",
                     "traffic": ncu_traffic("fused_vec_kernel", S, mode="rank_view"),
                     "traffic_note": "dram read + write bytes per parameter from an ncu capture of the same kernel "
                                     "in the same rank-view mode on 33,554,432-element chunks, times the shard's "
                                     "parameters (the kernel is a pure stream)",
                     "algorithmic_bytes_per_launch": bytes_per_step, "bytes_per_param": 2 * n + 26,
                     "launch_ms": launch_ms},
        "clocks": clocks,
        "gpu_launches": K,
    }
    # the same step as one launch per 50 MiB bucket (277 launches, replayed from a CUDA graph)
    bucket_leg = None
    if not args.no_legs and rank == 0:
        bucket_leg = per_bucket_leg(z, w, hbm_peak, stream)
    # end to end through the public API: the incoming chunks from page-locked host memory,
    # the bf16 shard back to it
    out["e2e"] = e2e_leg(z, w, world, args)
    del w
    torch.cuda.empty_cache()
    # the other rows, reported by rank 0 only (they hold no collective, so the other ranks
    # need not run them)
    if not args.no_legs and rank == 0:
        out["legs"] = extra_legs(z, synth, dev, hbm_peak, tf_burst, peak_src, args)
        out["legs"]["mistral_rank_view_per_bucket"] = bucket_leg
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(budget_s=args.cpu_seconds)
        if "legs" in out:
            oracle_beside_legs(out["legs"])
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def per_bucket_leg(z, w, hbm_peak, stream):
    """The headline step as DDP / ZeRO issue it, one launch per 50 MiB bucket as backward
    produces it: 277 launches captured in a CUDA graph, on one stream and round-robin on
    four (the buckets are disjoint, so launches on different streams may overlap). Same
    bits as the one launch (tested)."""
    import torch
    plan, n, S = w["plan"], w["n"], w["S"]
    byts = S * (2 * n + 26)
    a = (w["grads"], w["master"], w["m"], w["v"], w["param"], HP, 1)
    res = {"n_buckets": plan.n_buckets, "bucket_elems": plan.bucket_elems, "bytes": byts}
    side = torch.cuda.Stream()  # graphs are captured on a stream other than the default one
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for ns in (1, 4):
            g = bucket_graph(z, plan, z.ZERO_RANK_VIEW, a, ns)
            ms = time_launches(lambda: g.replay(), 10, side)
            res[f"streams_{ns}"] = {"ms": ms, "gbs": byts / ms / 1e6, "frac": byts / ms / 1e6 / hbm_peak,
                                    "launches_per_step": plan.n_buckets}
            del g
    stream.wait_stream(side)
    z.zero_device_status(side)
    return res


def host_mem_available() -> int:
    """MemAvailable of this host in bytes (0 if unknown)."""
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


def e2e_elems(S: int, n: int, world: int, avail: int, bucket: int) -> int:
    """Shard elements the e2e leg moves through host memory per step: the whole shard when
    every rank's page-locked buffers ((2n + 2) bytes per element, rounded up to powers of two
    by the pinned allocator) fit in half of the host's available memory, otherwise the
    largest whole number of buckets that does (at least one)."""
    def pinned(L):
        return (n + 1) * (1 << (2 * L - 1).bit_length())
    if avail <= 0 or world * pinned(S) <= avail // 2:
        return S
    L = S
    while L > bucket and world * pinned(L) > avail // 2:
        L = max(bucket, (L // 2) // bucket * bucket)
    return L


def e2e_leg(z, w, world, args):
    """The same metric end to end through the public API with HOST buffers: every step the 8
    incoming bf16 gradient chunks come from page-locked host memory and the bf16 shard goes
    back to it. zero_fused_step_host reads the chunks and writes the shard straight over
    the host link inside the kernel (each byte crosses once); the staged variant copies
    them with cudaMemcpyAsync around zero_fused_step instead. When the host cannot pin the
    whole shard's buffers for every rank, a stated prefix of whole buckets is moved."""
    import torch
    n, S = w["n"], w["S"]
    L = e2e_elems(S, n, world, host_mem_available(), w["plan"].bucket_elems)
    plan = w["plan"] if L == S else z.zero_plan(n * L, n, w["stage"], w["bb"])
    host_chunks = [torch.empty(L, dtype=torch.bfloat16, pin_memory=True) for _ in range(n)]
    for q in range(n):
        host_chunks[q].copy_(w["grads"][q][:L])
    host_param = torch.empty(L, dtype=torch.bfloat16, pin_memory=True)
    master, m, v = w["master"][:L], w["m"][:L], w["v"][:L]
    stream = torch.cuda.current_stream()
    steps = max(3, args.e2e_steps)

    def run(step, first):
        for t in range(first, first + 3):
            step(t)
        torch.cuda.synchronize()
        barrier(world)
        t0 = time.perf_counter()
        for t in range(first + 3, first + 3 + steps):
            step(t)
        torch.cuda.synchronize()
        el = max_over_ranks(time.perf_counter() - t0, world)
        z.zero_device_status(stream)
        return el

    def direct(t):
        z.zero_fused_step_host(plan, z.ZERO_RANK_VIEW, host_chunks, master, m, v, host_param, HP, t, stream)

    el = run(direct, 1)
    dgrads = [w["grads"][q][:L] for q in range(n)]
    param = w["param"][:L]

    def staged(t):
        for q in range(n):
            dgrads[q].copy_(host_chunks[q], non_blocking=True)
        z.zero_fused_step(plan, z.ZERO_RANK_VIEW, dgrads, master, m, v, param, HP, t, stream)
        host_param.copy_(param, non_blocking=True)

    el_staged = run(staged, 100)
    del host_chunks, host_param
    return {"value": job_throughput(L, steps, world, el), "unit": UNIT, "h2d_bytes_per_step": 2 * L * n,
            "d2h_bytes_per_step": 2 * L, "steps": steps, "ms_per_step": 1e3 * el / steps,
            "elems_per_step": L, "whole_shard": L == S,
            "how": "zero_fused_step_host: the kernel reads the 8 incoming bf16 gradient chunks from page-locked host "
                   "memory and writes the bf16 shard back to it over the host link; wall clock over the steps"
                   + ("" if L == S else f"; the first {L:,} of the {S:,} shard elements (whole 50 MiB buckets), as "
                                        "the host could not pin the whole shard's buffers for every rank"),
            "staged_copies": {"value": job_throughput(L, steps, world, el_staged), "ms_per_step": 1e3 * el_staged / steps,
                              "how": "cudaMemcpyAsync host->device of the chunks, zero_fused_step, device->host "
                                     "copy of the shard"}}


def time_launches(fn, iters, stream):
    import torch
    fn()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
    for s, e in evs:
        s.record(stream)
        fn()
        e.record(stream)
    torch.cuda.synchronize()
    return statistics.fmean(s.elapsed_time(e) for s, e in evs)


def extra_legs(z, synth, dev, hbm_peak, tf_burst, peak_src, args):
    """The other rows of the path, each timed on its own after the main region:
    the DDP all-reduce + replica Adam, the unfused reduce-scatter -> Adam -> all-gather
    pipeline (ablation), and the FSDP unit forward on the Mistral-7B MLP shapes."""
    import torch
    legs = {}
    stream = torch.cuda.current_stream()
    psi, n = synth.GPT2_SMALL_PSI, 8
    hp = {"lr": 1e-4, "beta1": 0.9, "beta2": 0.999, "eps": 1e-8, "weight_decay": 0.0}
    plan = z.zero_plan(psi, n, "ddp", 25 * MIB)
    P, S = plan.psi_padded, plan.shard_elems
    grads = [synth.rank_grads(psi, P, r, 1, device=dev) for r in range(n)]
    master = synth.master_params(psi, P, device=dev)
    m = torch.zeros(P, device=dev)
    v = torch.zeros(P, device=dev)
    param = torch.empty(P, dtype=torch.bfloat16, device=dev)
    g = torch.empty(P, device=dev)
    it = 50
    ms_ar = time_launches(lambda: z.ddp_allreduce(plan, grads, g, stream), it, stream)
    ms_ad = time_launches(lambda: z.zero_adam_step(plan, z.ZERO_ALL_RANKS, g, master, m, v, None, hp, 1, stream),
                          it, stream)
    ms_ag = time_launches(lambda: z.zero_allgather_params(plan, [master[r * S:(r + 1) * S] for r in range(n)], param,
                                                          stream), it, stream)
    b_ar, b_ad, b_ag = P * (2 * n + 4), P * 28, P * 6
    legs["ddp_allreduce"] = {"ms": ms_ar, "gbs": b_ar / ms_ar / 1e6, "frac": b_ar / ms_ar / 1e6 / hbm_peak,
                             "bytes": b_ar, "params_per_s": P / ms_ar * 1e3}
    legs["adam_step"] = {"ms": ms_ad, "gbs": b_ad / ms_ad / 1e6, "frac": b_ad / ms_ad / 1e6 / hbm_peak, "bytes": b_ad,
                         "params_per_s": P / ms_ad * 1e3}
    legs["allgather_params"] = {"ms": ms_ag, "gbs": b_ag / ms_ag / 1e6, "frac": b_ag / ms_ag / 1e6 / hbm_peak,
                                "bytes": b_ag, "params_per_s": P / ms_ag * 1e3}
    legs["unfused_pipeline_ms"] = ms_ar + ms_ad + ms_ag
    # the same list at N = 8, ZeRO-2, every rank's shard in one fused launch (5.22 GB)
    plan2 = z.zero_plan(psi, n, "zero2", 25 * MIB)
    ms_f = time_launches(lambda: z.zero_fused_step(plan2, z.ZERO_ALL_RANKS, grads, master, m, v, param, hp, 1, stream),
                         200, stream)
    b_f = P * (2 * n + 26)
    legs["gpt2_small_fused_step"] = {"config": gpt2_config(psi, n, "zero2", 25 * MIB), "ms": ms_f,
                                     "gbs": b_f / ms_f / 1e6, "frac": b_f / ms_f / 1e6 / hbm_peak, "bytes": b_f,
                                     "params_per_s": psi / ms_f * 1e3, "kernel": "fused_vec_kernel<8>"}
    z.zero_set_fused_kernel(1)
    ms_tma = time_launches(lambda: z.zero_fused_step(plan, z.ZERO_ALL_RANKS, grads, master, m, v, param, hp, 1,
                                                     stream), it, stream)
    z.zero_set_fused_kernel(0)
    legs["fused_tma_pipeline_variant"] = {"ms": ms_tma, "gbs": b_f / ms_tma / 1e6, "frac": b_f / ms_tma / 1e6 / hbm_peak}
    del grads, g
    # Megatron distributed optimizer: the same fused step on fp32 gradients, 4N + 26 B/param
    plan_mg = z.zero_plan(psi, n, "megatron", 25 * MIB)
    grads32 = [synth.rank_grads_f32(psi, P, r, 1, device=dev) for r in range(n)]
    ms_mg = time_launches(lambda: z.zero_fused_step_fp32_grads(plan_mg, z.ZERO_ALL_RANKS, grads32, master, m, v, param,
                                                               hp, 1, stream), it, stream)
    b_mg = plan_mg.fused_step_bytes
    legs["megatron_fp32_grads"] = {"ms": ms_mg, "gbs": b_mg / ms_mg / 1e6, "frac": b_mg / ms_mg / 1e6 / hbm_peak,
                                   "bytes": b_mg, "params_per_s": P / ms_mg * 1e3}
    del grads32, master, m, v, param
    torch.cuda.empty_cache()
    # the tensor-core legs are compared with the burst bf16 peak (a short cuBLAS loop on a
    # cool GPU): let the GPU idle for a moment after the seconds of HBM streaming above, and
    # record the SM clocks each of them ran at
    gpu = torch.cuda.current_device()
    time.sleep(args.leg_idle_s)
    with ClockSampler(gpu) as clk:
        legs["fsdp_unit_forward"] = fsdp_leg(z, synth, dev, tf_burst, peak_src, stream)
    legs["fsdp_unit_forward"]["clocks"] = clk.summary()
    legs["fsdp_unit_forward"]["idle_before_s"] = args.leg_idle_s
    torch.cuda.empty_cache()
    time.sleep(args.leg_idle_s)
    with ClockSampler(gpu) as clk:
        legs["fsdp_zero3_step"] = zero3_leg(z, synth, dev, tf_burst, hbm_peak, stream)
    legs["fsdp_zero3_step"]["clocks"] = clk.summary()
    legs["fsdp_zero3_step"]["idle_before_s"] = args.leg_idle_s
    torch.cuda.empty_cache()
    time.sleep(args.leg_idle_s)
    with ClockSampler(gpu) as clk:
        legs["fsdp_zero3_mlp_step"] = zero3_mlp_leg(z, synth, dev, tf_burst, stream)
    legs["fsdp_zero3_mlp_step"]["clocks"] = clk.summary()
    legs["fsdp_zero3_mlp_step"]["idle_before_s"] = args.leg_idle_s
    # beside each fraction of the burst bf16 peak, the fraction of the sustained one (the
    # same cuBLAS GEMM looped for seconds under the power cap): these legs run for tens of
    # milliseconds after seconds of other work, and the tensor-core kernels reach the power
    # cap themselves
    tf_sust = peaks()[2]
    for leg in (legs["fsdp_unit_forward"], legs["fsdp_zero3_step"], legs["fsdp_zero3_mlp_step"]):
        for v in [leg] + list(leg.values()):
            if isinstance(v, dict) and "tflops" in v:
                v["frac_of_sustained_bf16_peak"] = v["tflops"] / tf_sust
    return legs


ZERO3_SHAPES = [(14336, 4096), (4096, 14336), (14336, 4096), (4096, 14336)]
MLP_UNITS = 2  # Mistral-7B MLP units (d_model 4096, d_ff 14336) in the MLP stack leg


def zero3_mlp_units(z, synth, dev, n, m, n_units=MLP_UNITS, d=4096, f=14336):
    """A stack of Mistral-7B MLP units (W_gate, W_up [14336, 4096], W_down [4096, 14336],
    each in n row shards with its ZeRO-3 state), n ranks of m tokens."""
    import torch
    nm = n * m
    bf = dict(dtype=torch.bfloat16, device=dev)

    def weight(rows, cols, key):
        w = torch.cat(synth.weight_shards(rows, cols, n, device=dev, seed_key=key), 0).contiguous()
        return {"plan": z.zero_plan(rows * cols, n, "zero3", 50 * MIB), "w": w, "master": w.float().reshape(-1),
                "m": torch.zeros(rows * cols, device=dev), "v": torch.zeros(rows * cols, device=dev)}
    units = [{"d_model": d, "d_ff": f, "gate": weight(f, d, 40 + 3 * i), "up": weight(f, d, 41 + 3 * i),
              "down": weight(d, f, 42 + 3 * i), "x": torch.empty(nm, d, **bf), "gu": torch.empty(nm, 2 * f, **bf),
              "h": torch.empty(nm, f, **bf), "dy": torch.empty(nm, d, **bf), "dh": torch.empty(nm, f, **bf),
              "dgu": torch.empty(nm, 2 * f, **bf), "dw_gu": torch.empty(2 * f, d, device=dev),
              "dw_down": torch.empty(d, f, device=dev)} for i in range(n_units)]
    units[0]["x"].copy_(synth.activations(nm, d, device=dev))
    units[-1]["dy"].copy_(synth.upstream_grad(nm, d, device=dev))
    return units


def zero3_mlp_leg(z, synth, dev, tf_peak, stream):
    """One ZeRO-3 training step over a stack of Mistral-7B MLP units, N = 8 ranks of 1024
    tokens: forward (gate-up kernel saving G | U, down projection), backward in reverse
    (dH, dW_down, SiLU-gate backward, dX over both projections, dW_gate | dW_up), each
    rank's Adam on its three shards."""
    import torch
    n, m = 8, 1024
    res = {"units": MLP_UNITS, "d_model": 4096, "d_ff": 14336, "n_ranks": n, "tokens_per_rank": m}
    try:
        units = zero3_mlp_units(z, synth, dev, n, m)
        nm = n * m
        y = torch.empty(nm, 4096, dtype=torch.bfloat16, device=dev)
        dx = torch.empty(nm, 4096, dtype=torch.bfloat16, device=dev)
        wsb = z.fsdp_zero3_mlp_step_workspace(n, [(4096, 14336)] * MLP_UNITS, m)
        ws = torch.empty(wsb, dtype=torch.uint8, device=dev) if wsb else None
        flop = MLP_UNITS * 3 * 3 * 2.0 * nm * 4096 * 14336  # 3 matrices, forward + 2 backward GEMMs each
        # the fused optimizer (the default) writes no dW; the separate form reads it back
        no_dw = [{k: v for k, v in u.items() if k not in ("dw_gu", "dw_down")} for u in units]
        for name, flags, us in (("fused_optimizer", 0, no_dw), ("separate_optimizer", z.FSDP_SEPARATE_OPTIMIZER,
                                                                 units)):
            t = [0]

            def step():
                t[0] += 1
                z.fsdp_zero3_mlp_step(us, m, HP, t[0], y_out=y, dx_out=dx, workspace=ws, stream=stream, flags=flags)

            ms = time_launches(step, 10, stream)
            res[name] = {"ms": ms, "tflops": flop / ms / 1e9, "frac_of_bf16_peak": flop / ms / 1e9 / tf_peak}
        z.zero_device_status(stream)
        res.update(ms=res["fused_optimizer"]["ms"], tflops=res["fused_optimizer"]["tflops"],
                   frac_of_bf16_peak=res["fused_optimizer"]["frac_of_bf16_peak"],
                   fused_optimizer_gain=res["separate_optimizer"]["ms"] / res["fused_optimizer"]["ms"] - 1.0,
                   gemm_flop_per_step=flop, workspace_bytes=wsb,
                   adam_bytes_per_step=MLP_UNITS * 3 * 30 * 4096 * 14336,
                   silu_backward_bytes_per_step=MLP_UNITS * 10 * nm * 14336,
                   note="tflops counts the GEMM flops over the whole step, which also holds each rank's Adam (fused "
                        "into the dW GEMMs' epilogues, or separate) and the SiLU-gate backward; every backward operand "
                        "is read in place (no transpose)")
    except Exception as e:  # the leg must not hide the step's line
        res["error"] = str(e)[:300]
    return res


def zero3_units(z, synth, dev, n, m, shapes=ZERO3_SHAPES):
    """A stack of FSDP units with the Mistral-7B MLP shapes (alternating 14336 x 4096 and
    4096 x 14336, each in n row shards), ZeRO-3 state, n ranks of m tokens."""
    import torch
    units = []
    nm = n * m
    for i, (R, K) in enumerate(shapes):
        w = torch.cat(synth.weight_shards(R, K, n, device=dev, seed_key=20 + i), 0).contiguous()
        units.append({"plan": z.zero_plan(R * K, n, "zero3", 50 * MIB), "w": w, "master": w.float().reshape(-1),
                      "m": torch.zeros(R * K, device=dev), "v": torch.zeros(R * K, device=dev),
                      "x": torch.empty(nm, K, dtype=torch.bfloat16, device=dev),
                      "dy": torch.empty(nm, R, dtype=torch.bfloat16, device=dev),
                      "dw": torch.empty(R, K, device=dev)})
    units[0]["x"].copy_(synth.activations(nm, shapes[0][1], device=dev))
    units[-1]["dy"].copy_(synth.upstream_grad(nm, shapes[-1][0], device=dev))
    return units


def zero3_leg(z, synth, dev, tf_peak, hbm_peak, stream):
    """One ZeRO-3 training step over 4 FSDP units with the Mistral-7B MLP shapes, N = 8
    ranks of 1024 tokens (8192 in all): forward, backward in reverse with each rank's Adam
    on its shard after the unit's backward (fused into the dW GEMM's epilogue, or its own
    launch). Timed serial (every gather fused into the GEMMs' loads), with each unit's Adam
    on a second stream beside the next units' GEMMs, and with the gathers materialised into
    a workspace slot, serially or with the next unit's gather prefetched on that stream."""
    import torch
    n, m = 8, 1024
    res = {"units": [list(s) for s in ZERO3_SHAPES], "n_ranks": n, "tokens_per_rank": m}
    try:
        units = zero3_units(z, synth, dev, n, m)
        nm = n * m
        y = torch.empty(nm, ZERO3_SHAPES[-1][0], dtype=torch.bfloat16, device=dev)
        dx = torch.empty(nm, ZERO3_SHAPES[0][1], dtype=torch.bfloat16, device=dev)
        side = torch.cuda.Stream()
        flop = sum(6.0 * nm * R * K for R, K in ZERO3_SHAPES)
        adam_bytes = sum(30 * R * K for R, K in ZERO3_SHAPES)
        res["gemm_flop_per_step"] = flop
        res["adam_bytes_per_step"] = adam_bytes
        P, O, G, S = (z.FSDP_BACKWARD_PREFETCH, z.FSDP_OVERLAP_OPTIMIZER, z.FSDP_GATHER_MATERIALIZE,
                      z.FSDP_SEPARATE_OPTIMIZER)
        # the fused optimizer (the default) writes no dW; the separate forms read it back
        no_dw = [{k: v for k, v in u.items() if k != "dw"} for u in units]
        for name, flags, pf in (("serial", 0, None), ("separate_optimizer", S, None),
                                ("overlap_optimizer", O, side), ("materialized_serial", G, None),
                                ("materialized_prefetch", G | P, side),
                                ("materialized_prefetch_overlap_optimizer", G | P | O, side)):
            wsb = z.fsdp_zero3_step_workspace(n, ZERO3_SHAPES, m, flags)
            ws = torch.empty(wsb, dtype=torch.uint8, device=dev) if wsb else None
            t = [0]
            us = units if flags & (S | O) else no_dw

            def step():
                t[0] += 1
                z.fsdp_zero3_step(us, m, HP, t[0], y_out=y, dx_out=dx, flags=flags, workspace=ws, stream=stream,
                                  prefetch_stream=pf)

            ms = time_launches(step, 10, stream)
            res[name] = {"ms": ms, "tflops": flop / ms / 1e9, "frac_of_bf16_peak": flop / ms / 1e9 / tf_peak,
                         "workspace_bytes": wsb}
            del ws
        z.zero_device_status(stream)
        res["fused_optimizer_gain"] = res["separate_optimizer"]["ms"] / res["serial"]["ms"] - 1.0
        res["overlap_optimizer_gain"] = res["serial"]["ms"] / res["overlap_optimizer"]["ms"] - 1.0
        res["materialized_prefetch_gain"] = (res["materialized_serial"]["ms"] / res["materialized_prefetch"]["ms"]
                                             - 1.0)
        res["note"] = ("tflops counts the 12 GEMMs' flops (6 N M R K per unit) over the whole step, which also holds "
                       "each rank's Adam (fused into the dW GEMMs' epilogues unless separate); every backward operand "
                       "is read in place (no transpose), the gathers fused into the loads unless materialised")
    except Exception as e:  # the leg must not hide the step's line
        res["error"] = str(e)[:300]
    return res


def fsdp_leg(z, synth, dev, tf_peak, peak_src, stream):
    """Mistral-7B MLP unit, N = 8 row shards: W_up, W_gate [14336, 4096] times X [8192,
    4096]; W_down [4096, 14336] times H [8192, 14336]; fp32 out. Gather fused into the
    GEMM's loads (no scratch) and, separately, materialised into a scratch W."""
    import torch
    n, M = 8, 8192
    X = synth.activations(M, 4096, device=dev)
    H = synth.activations(M, 14336, device=dev, seed_key=1)
    mats = {"up": (14336, 4096, X), "gate": (14336, 4096, X), "down": (4096, 14336, H)}
    res = {}
    try:
        total_ms, total_flop = 0.0, 0.0
        for name, (R, K, A) in mats.items():
            shards = synth.weight_shards(R, K, n, device=dev, seed_key={"up": 11, "gate": 12, "down": 13}[name])
            Y = torch.empty(M, R, device=dev)
            ms = time_launches(lambda: z.fsdp_unit_forward(shards, A, Y, stream=stream), 10, stream)
            flop = 2.0 * M * R * K
            res[name] = {"ms": ms, "tflops": flop / ms / 1e9}
            total_ms += ms
            total_flop += flop
            del shards, Y
        res["total_ms"] = total_ms
        res["tflops"] = total_flop / total_ms / 1e9
        res["roofline"] = {"bound": "tensor", "kernel": "fsdp_gemm_pair_kernel<false>", "achieved": res["tflops"],
                           "peak": tf_peak, "unit": "TFLOP/s", "frac": res["tflops"] / tf_peak,
                           "peak_source": f"{peak_src} bf16_tflops (burst)" if peak_src == "measured" else "fallback"}
        # the same W_up GEMM with a bf16-only output (Y = NULL): half the output bytes
        shards = synth.weight_shards(14336, 4096, n, device=dev, seed_key=11)
        Yb = torch.empty(M, 14336, dtype=torch.bfloat16, device=dev)
        ms = time_launches(lambda: z.fsdp_unit_forward(shards, X, None, Y_bf16=Yb, stream=stream), 10, stream)
        res["up_bf16_output"] = {"ms": ms, "tflops": 2.0 * M * 14336 * 4096 / ms / 1e9,
                                 "frac": 2.0 * M * 14336 * 4096 / ms / 1e9 / tf_peak,
                                 "note": "Y_bf16 only (no fp32 Y); not part of the unit's fp32-output roofline"}
        # the same W_up GEMM on the one-CTA kernel (zero_set_gemm_kernel(1)), same bits
        Y = torch.empty(M, 14336, device=dev)
        z.zero_set_gemm_kernel(1)
        try:
            ms = time_launches(lambda: z.fsdp_unit_forward(shards, X, Y, stream=stream), 10, stream)
        finally:
            z.zero_set_gemm_kernel(0)
        res["up_one_cta_kernel"] = {"ms": ms, "tflops": 2.0 * M * 14336 * 4096 / ms / 1e9,
                                    "frac": 2.0 * M * 14336 * 4096 / ms / 1e9 / tf_peak,
                                    "note": "fsdp_gemm_kernel<false>: one CTA per 128 x 256 tile, for comparison"}
        del shards, Yb, Y
        # row a6 on its own: the materialised all-gather of W_up's 8 row shards (4 B per
        # element) and the transposed gather of the same shards into W^T (4 B per element;
        # the backward's fallback path for shapes the in-place GEMMs do not take)
        hbm = peaks()[0]
        shards_up = synth.weight_shards(14336, 4096, n, device=dev, seed_key=11)
        wfull = torch.empty(14336, 4096, dtype=torch.bfloat16, device=dev)
        ms_g = time_launches(lambda: z.fsdp_gather_rows(shards_up, wfull, stream=stream), 20, stream)
        ms_t = time_launches(lambda: z.fsdp_transpose_cat(shards_up, wfull.view(4096, 14336), stream=stream), 20,
                             stream)
        # a plain device-to-device copy of the same bytes, timed the same way: at 2 x 117 MB
        # per launch, ramp-up and drain cap every copy below the long-copy peak
        src_up = torch.cat(shards_up, 0)
        ms_c = time_launches(lambda: wfull.copy_(src_up), 20, stream)
        b_gt = 4.0 * 14336 * 4096
        res["gather_rows_w_up"] = {"ms": ms_g, "gbs": b_gt / ms_g / 1e6, "frac": b_gt / ms_g / 1e6 / hbm,
                                   "frac_of_same_size_copy": ms_c / ms_g}
        res["transpose_cat_w_up"] = {"ms": ms_t, "gbs": b_gt / ms_t / 1e6, "frac": b_gt / ms_t / 1e6 / hbm,
                                     "frac_of_same_size_copy": ms_c / ms_t}
        res["copy_same_bytes_w_up"] = {"ms": ms_c, "gbs": b_gt / ms_c / 1e6, "frac": b_gt / ms_c / 1e6 / hbm,
                                       "note": "torch copy_ of W_up's 117 MB (not this library's code): what a "
                                               "plain copy of this size reaches, for the two rows above"}
        del shards_up, wfull, src_up
        # the full MLP unit: gate + up in one kernel with the SiLU-gate epilogue, then down
        gs_ = synth.weight_shards(14336, 4096, n, device=dev, seed_key=12)
        us_ = synth.weight_shards(14336, 4096, n, device=dev, seed_key=11)
        ds_ = synth.weight_shards(4096, 14336, n, device=dev, seed_key=13)
        Hb = torch.empty(M, 14336, dtype=torch.bfloat16, device=dev)
        Ym = torch.empty(M, 4096, device=dev)
        ms = time_launches(lambda: z.fsdp_mlp_forward(gs_, us_, ds_, X, Hb, Ym, stream=stream), 10, stream)
        flop = 3 * 2.0 * M * 14336 * 4096
        res["mlp_unit"] = {"ms": ms, "tflops": flop / ms / 1e9, "frac": flop / ms / 1e9 / tf_peak,
                           "note": "gate+up GEMM with silu(gate)*up epilogue (bf16 H) + down GEMM, fused gathers"}
        side = torch.cuda.Stream()
        sd = torch.empty(4096, 14336, dtype=torch.bfloat16, device=dev)
        ms2 = time_launches(lambda: z.fsdp_mlp_forward(gs_, us_, ds_, X, Hb, Ym, scratch_down=sd, stream=stream,
                                                       prefetch_stream=side), 10, stream)
        res["mlp_unit_prefetched_gather"] = {"ms": ms2, "tflops": flop / ms2 / 1e9,
                                             "note": "W_down gathered into scratch on a second stream during gate+up"}
        del gs_, us_, ds_, Hb, Ym, sd
        # backward of W_up for 8 ranks of 2048 tokens, every operand read where it lies: one
        # dX GEMM over all ranks with W's row shards as an MN-major operand (the backward
        # gather fused into the loads), one rank-reduced dW GEMM with dY and X as MN-major
        # operands; no workspace
        R, K, Mb = 14336, 4096, 2048
        shards = synth.weight_shards(R, K, n, device=dev, seed_key=11)
        A = [synth.activations(Mb, K, device=dev, seed_key=q) for q in range(n)]
        dY = [synth.upstream_grad(Mb, R, device=dev, seed_key=q) for q in range(n)]
        dX = [torch.empty(Mb, K, device=dev) for _ in range(n)]
        dW = torch.empty(R, K, device=dev)
        wsb = z.fsdp_unit_backward_workspace(n, R, K, Mb)
        ws = torch.empty(wsb, dtype=torch.uint8, device=dev) if wsb else None
        ms = time_launches(lambda: z.fsdp_unit_backward(shards, A, dY, dX, dW, ws, stream=stream), 5, stream)
        flop = 2.0 * (2.0 * n * Mb * R * K)
        res["backward_up"] = {"ms": ms, "tflops": flop / ms / 1e9, "frac": flop / ms / 1e9 / tf_peak,
                              "ranks": n, "tokens_per_rank": Mb,
                              "launches": 2, "workspace_bytes": wsb,
                              "note": "every operand read in place (CTA-pair kernel): dX over all ranks with W's "
                                      "shards as an MN-major operand; dW with dY and X as MN-major operands"}
        # the same call on the one-CTA kernel, for comparison
        z.zero_set_gemm_kernel(1)
        try:
            ms_1 = time_launches(lambda: z.fsdp_unit_backward(shards, A, dY, dX, dW, ws, stream=stream), 5, stream)
        finally:
            z.zero_set_gemm_kernel(0)
        res["backward_up_one_cta_kernel"] = {"ms": ms_1, "tflops": flop / ms_1 / 1e9,
                                             "frac": flop / ms_1 / 1e9 / tf_peak,
                                             "note": "the same in-place GEMMs on fsdp_gemm_kernel (one CTA per "
                                                     "128 x 256 tile)"}
        del shards, A, dY, dX, dW, ws
        # the same for W_down [4096, 14336] (X is the MLP's H)
        R, K = 4096, 14336
        shards = synth.weight_shards(R, K, n, device=dev, seed_key=13)
        A = [synth.activations(Mb, K, device=dev, seed_key=q) for q in range(n)]
        dY = [synth.upstream_grad(Mb, R, device=dev, seed_key=q) for q in range(n)]
        dX = [torch.empty(Mb, K, device=dev) for _ in range(n)]
        dW = torch.empty(R, K, device=dev)
        wsb = z.fsdp_unit_backward_workspace(n, R, K, Mb)
        ws = torch.empty(wsb, dtype=torch.uint8, device=dev) if wsb else None
        ms = time_launches(lambda: z.fsdp_unit_backward(shards, A, dY, dX, dW, ws, stream=stream), 5, stream)
        res["backward_down"] = {"ms": ms, "tflops": flop / ms / 1e9, "frac": flop / ms / 1e9 / tf_peak,
                                "ranks": n, "tokens_per_rank": Mb, "workspace_bytes": wsb,
                                "note": "every operand read in place, as backward_up"}
    except Exception as e:  # the GEMM leg must not hide the step's line
        res["error"] = str(e)[:300]
    return res


# ---------------------------------------------------------------------------------------
# the CPU oracle as baseline / reference arm
# ---------------------------------------------------------------------------------------

class OracleSample:
    """A bounded sample of a fused-step workload, generated once: n_params parameters with
    n_ranks bf16 gradient slices and fp32 master / m / v. chunks=True draws the slices as
    one rank's incoming chunks (the Mistral-7B rank view, synth.chunk_grads), otherwise as
    the ranks' flat gradient buffers (synth.rank_grads); both are the same distributions.
    step() runs one fused oracle step (reduce, Adam, cast in plain numpy) on the first
    `count` parameters and returns its seconds. With threads > 1 the same oracle call runs
    on `threads` contiguous ranges at once: the step is elementwise, so the split changes
    no result, and numpy releases the interpreter lock inside its array operations."""

    def __init__(self, n_params: int, n_ranks: int = 8, threads: int = 1, chunks: bool = False):
        import numpy as np
        import torch

        import synth
        from oracle import zero_oracle as O
        self.O = O
        self.n = n_params
        self.master = synth.master_params(n_params, n_params).numpy()
        self.m = np.zeros(n_params, np.float32)
        self.v = np.zeros(n_params, np.float32)
        if chunks:
            ch = synth.chunk_grads(n_params, n_ranks, 1).view(torch.int16).numpy().view(np.uint16)
            self.grads = [ch[q] for q in range(n_ranks)]
        else:
            self.grads = [synth.rank_grads(n_params, n_params, r, 1).view(torch.int16).numpy().view(np.uint16)
                          for r in range(n_ranks)]
        self.hp = O.AdamHyper()
        self.t = 0
        self.threads = max(1, int(threads))
        self._pool = None
        if self.threads > 1:
            from concurrent.futures import ThreadPoolExecutor
            self._pool = ThreadPoolExecutor(self.threads)

    def _range(self, lo: int, hi: int) -> None:
        w, m, v, _ = self.O.fused_step_elements([g[lo:hi] for g in self.grads], self.master[lo:hi],
                                                self.m[lo:hi], self.v[lo:hi], self.hp, self.t)
        self.master[lo:hi], self.m[lo:hi], self.v[lo:hi] = w, m, v

    def step(self, count: int) -> float:
        count = min(count, self.n)
        self.t += 1
        cuts = [count * i // self.threads for i in range(self.threads + 1)]
        t0 = time.perf_counter()
        if self._pool is None:
            self._range(0, count)
        else:
            list(self._pool.map(lambda i: self._range(cuts[i], cuts[i + 1]), range(self.threads)))
        return time.perf_counter() - t0


def _time_bounded(fn, budget_s: float):
    """Seconds per call of fn, over as many calls as fit in budget_s (at least one)."""
    fn()
    t0, k = time.perf_counter(), 0
    while True:
        fn()
        k += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            return el / k, k


def oracle_beside_legs(legs: dict, budget_s: float = 1.5):
    """The oracle as it stands, timed on the host beside each GPU leg on a bounded sample of
    that leg's workload; numpy with its BLAS pinned to one thread. Adds legs[k]["cpu_oracle"]."""
    import numpy as np
    import torch

    import synth
    from oracle import zero_oracle as O
    n_params, n = 4 * MIB, 8
    s = OracleSample(n_params)
    g = O.reduce_sum_scale(s.grads, 0, n_params)
    S = n_params // n
    g32 = [synth.rank_grads_f32(n_params, n_params, r, 1).numpy() for r in range(n)]
    elem = f"first {n_params:,} of the 124,356,864 GPT-2-small parameters, N = 8"

    def put(key, per_call, calls, value, unit, sample):
        if key in legs and isinstance(legs[key], dict):
            legs[key]["cpu_oracle"] = {"value": value, "unit": unit, "cores": 1, "kind": "oracle",
                                       "sample": f"{sample}; {calls} calls, {per_call * 1e3:.1f} ms each"}

    t, k = _time_bounded(lambda: O.reduce_sum_scale(s.grads, 0, n_params), budget_s)
    put("ddp_allreduce", t, k, n_params / t, "params/s", elem + " bf16 gradient slices, rank-order fp32 sum x 1/N")
    t, k = _time_bounded(lambda: O.adam_update(s.master, s.m, s.v, g, s.hp, 1), budget_s)
    put("adam_step", t, k, n_params / t, "params/s", elem + ", Adam on fp32 master / m / v")
    t, k = _time_bounded(lambda: O.f32_to_bf16(O.all_gather([s.master[i * S:(i + 1) * S] for i in range(n)])),
                         budget_s)
    put("allgather_params", t, k, n_params / t, "params/s", elem + ", bf16 cast and all-gather of 8 master shards")
    t, k = _time_bounded(lambda: O.fused_step_elements(g32, s.master, s.m, s.v, s.hp, 1), budget_s)
    put("megatron_fp32_grads", t, k, n_params / t, "params/s", elem + " fp32 gradient slices, fused step")
    fl = legs.get("fsdp_unit_forward")
    if isinstance(fl, dict):
        R, K, rows = 14336, 4096, 16
        shards = [x.view(torch.int16).numpy().view(np.uint16) for x in synth.weight_shards(R, K, n)]
        a = synth.activations(rows, K).view(torch.int16).numpy().view(np.uint16)
        dy = synth.upstream_grad(rows, R).view(torch.int16).numpy().view(np.uint16)
        t, k = _time_bounded(lambda: O.fsdp_linear_forward(a, shards), budget_s)
        for key in ("up", "gate"):
            if isinstance(fl.get(key), dict):
                fl[key]["cpu_oracle"] = {"value": 2.0 * rows * R * K / t / 1e12, "unit": "TFLOP/s", "cores": 1,
                                         "kind": "oracle", "sample": f"{rows} of 8192 token rows against the full "
                                         f"14336 x 4096 weight from 8 shards (float64); {k} calls"}
        if isinstance(fl.get("backward_up"), dict):
            t, k = _time_bounded(lambda: O.fsdp_linear_backward(a, shards, dy, n), budget_s)
            fl["backward_up"]["cpu_oracle"] = {
                "value": 4.0 * rows * R * K / t / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                "sample": f"one rank's {rows} of 2048 tokens: dX and dW against the full 14336 x 4096 weight "
                          f"(float64); {k} calls"}
    t_adam = n_params / legs["adam_step"]["cpu_oracle"]["value"] if isinstance(legs.get("adam_step"), dict) \
        and "cpu_oracle" in legs["adam_step"] else None
    z3 = legs.get("fsdp_zero3_step")
    if isinstance(z3, dict) and "serial" in z3:
        # one unit of the step, the oracle's way: forward, dX and dW on 16 token rows of one
        # rank against the full 14336 x 4096 weight; Adam from its 4M-parameter timing
        R, K, rows = 14336, 4096, 16
        shards = [x.view(torch.int16).numpy().view(np.uint16) for x in synth.weight_shards(R, K, n)]
        a = synth.activations(rows, K).view(torch.int16).numpy().view(np.uint16)
        dy = synth.upstream_grad(rows, R).view(torch.int16).numpy().view(np.uint16)
        t, k = _time_bounded(lambda: (O.fsdp_linear_forward(a, shards), O.fsdp_linear_backward(a, shards, dy, n)),
                             budget_s)
        z3["cpu_oracle"] = {"value": 6.0 * rows * R * K / t / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                            "adam_params_per_s": (n_params / t_adam) if t_adam else None,
                            "sample": f"one 14336 x 4096 unit from 8 shards: forward, dX and dW on {rows} token rows "
                                      f"of one rank (float64); {k} calls; Adam as in legs.adam_step"}
    zm = legs.get("fsdp_zero3_mlp_step")
    if isinstance(zm, dict) and "fused_optimizer" in zm:
        # one Mistral MLP unit's forward (gate, up, SiLU gate, down) and its SiLU-gate
        # backward on 16 token rows, the oracle's way
        D, F, rows = 4096, 14336, 16
        gs = [x.view(torch.int16).numpy().view(np.uint16) for x in synth.weight_shards(F, D, n, seed_key=1)]
        us = [x.view(torch.int16).numpy().view(np.uint16) for x in synth.weight_shards(F, D, n, seed_key=2)]
        ds = [x.view(torch.int16).numpy().view(np.uint16) for x in synth.weight_shards(D, F, n, seed_key=3)]
        x = synth.activations(rows, D).view(torch.int16).numpy().view(np.uint16)
        dh = synth.upstream_grad(rows, F).view(torch.int16).numpy().view(np.uint16)
        gu = synth.activations(rows, 2 * F).view(torch.int16).numpy().view(np.uint16)
        t, k = _time_bounded(lambda: (O.mlp_unit_forward(x, gs, us, ds),
                                      O.silu_gate_backward(dh, gu[:, :F], gu[:, F:])), budget_s)
        zm["cpu_oracle"] = {"value": 3 * 2.0 * rows * D * F / t / 1e12, "unit": "TFLOP/s", "cores": 1,
                            "kind": "oracle", "adam_params_per_s": (n_params / t_adam) if t_adam else None,
                            "sample": f"one Mistral MLP unit from 8 shards per weight: forward (gate, up, SiLU gate, "
                                      f"down) and the SiLU-gate backward on {rows} token rows (float64); {k} calls; "
                                      "Adam as in legs.adam_step"}


def host_info() -> dict:
    """The host the oracle was timed on: architecture, logical CPUs, CPU model if known."""
    import platform
    info = {"machine": platform.machine(), "nproc": os.cpu_count()}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.split(":")[0].strip() in ("model name", "CPU part", "Hardware"):
                    info["cpu"] = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    return info


MISTRAL_SHARD = 905_216_512


def cpu_baseline(budget_s: float = 12.0, one_core_s: float = 4.0):
    """The oracle on every host core (contiguous ranges of the sample, one thread each), and
    for context the same oracle on one core, on a sample of the bench workload: the first
    elements of the Mistral-7B rank's shard with its 8 incoming gradient chunks."""
    cores = os.cpu_count() or 1
    n_params = 16 * MIB
    s = OracleSample(n_params, threads=cores, chunks=True)
    el = s.step(n_params)
    reps = max(1, int(budget_s / max(el, 1e-3)))
    total = sum(s.step(n_params) for _ in range(reps))
    one = OracleSample(4 * MIB, chunks=True)
    one_el, one_reps = _time_bounded(lambda: one.step(4 * MIB), one_core_s)
    return {"value": n_params * reps / total, "unit": UNIT, "cores": cores, "kind": "oracle", "host": host_info(),
            "one_core_value": 4 * MIB / one_el,
            "sample": f"{n_params:,} of the {MISTRAL_SHARD:,} elements of the Mistral-7B rank's shard (N=8, ZeRO-3) "
                      f"with their 8 incoming bf16 gradient chunks, {reps} fused steps ({total:.1f} s), split into "
                      f"{cores} contiguous ranges run by {cores} threads (numpy elementwise); one_core_value: "
                      f"{4 * MIB:,} elements on one thread, {one_reps} steps"}


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import synth
    psi, n, stage, bb, S = synth.MISTRAL_7B_PSI, 8, "zero3", 50 * MIB, MISTRAL_SHARD
    cap = 16 * MIB
    cores = os.cpu_count() or 1
    s = OracleSample(cap, threads=cores, chunks=True)
    s.step(cap)
    rate = cap / s.step(cap)
    # size each step's sample so the whole run stays near args.ref_seconds
    per_step = args.ref_seconds / max(1, args.steps + args.warmup)
    count = int(min(cap, max(65536, rate * per_step)))
    for _ in range(args.warmup):
        s.step(count)
    t_total = sum(s.step(count) for _ in range(args.steps))
    value = count * args.steps / t_total
    cb = {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "host": host_info(),
          "sample": f"{count:,} of the {S:,} elements of the Mistral-7B rank's shard per step (N=8 incoming chunks), "
                    f"numpy elementwise, split into {cores} contiguous ranges run by {cores} threads"}
    out = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": 1e3 * S / value, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded; Mistral-7B parameter count and shard "
                                                        "layout)",
           "config": workload_config(psi, n, stage, bb, S), "impl": "reference", "cpu_baseline": cb,
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


# ---------------------------------------------------------------------------------------
# the 1.5B-parameter bandwidth sweep
# ---------------------------------------------------------------------------------------

def bucket_graph(z, plan, rank, args, n_streams):
    """A CUDA graph of one fused-step launch per bucket, bucket k on stream k % n_streams,
    captured on the current stream. The buckets are disjoint index ranges, so launches on
    different streams may overlap: the next bucket's ramp-up runs during this one's drain."""
    import torch
    g = torch.cuda.CUDAGraph()
    side = [torch.cuda.Stream() for _ in range(n_streams - 1)]
    with torch.cuda.graph(g, stream=torch.cuda.current_stream()):
        cur = torch.cuda.current_stream()
        fork = torch.cuda.Event()
        fork.record(cur)
        for s in side:
            s.wait_event(fork)
        streams = [cur] + side
        for k in range(plan.n_buckets):
            z.zero_fused_step_buckets(plan, rank, k, k + 1, *args, streams[k % n_streams])
        for s in side:
            join = torch.cuda.Event()
            join.record(s)
            cur.wait_event(join)
    return g


def run_sweep(args):
    """psi = 1.5e9, N in {2,4,8,16,64}, buckets {1,5,25,100} MiB. For each point: one launch
    over all buckets, and one launch per bucket (as DDP reduces each bucket once backward
    produced it) captured in a CUDA graph, on one stream and round-robin on four. All N ranks' shards (full simulation) whenever
    the (2N + 14) P bytes of gradients, state and parameters fit in free device memory with
    an 8 GiB margin (N = 64: 213 GB, which a GB300 holds); otherwise one rank's view (its N
    incoming chunks)."""
    import torch

    import fsdp_sharded_optimizer_zero_gb300 as z
    import synth
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream()
    hbm_peak, _, _, peak_src = peaks()
    psi = 1_500_000_000
    hp = {"lr": 1e-4, "beta1": 0.9, "beta2": 0.999, "eps": 1e-8, "weight_decay": 0.0}
    cores = os.cpu_count() or 1
    for n in (2, 4, 8, 16, 64):
        plan0 = z.zero_plan(psi, n, "zero2", MIB)
        P, S = plan0.psi_padded, plan0.shard_elems
        # the oracle on every host core over a 2^22-parameter sample of this N, extrapolated
        # to the sweep's 1.5e9 parameters (the step is elementwise: time grows in proportion)
        ns = 1 << 22
        sample = OracleSample(ns, n_ranks=n, threads=cores)
        t_or, reps_or = _time_bounded(lambda: sample.step(ns), 3.0)
        cpu_or = {"value": ns / t_or, "unit": UNIT, "cores": cores, "kind": "oracle", "extrapolated": True,
                  "ms_per_step_extrapolated": psi / (ns / t_or) * 1e3,
                  "sample": f"first {ns:,} parameters, N={n} gradient slices, {reps_or} fused steps on "
                            f"{cores} threads; extrapolated to {psi:,} parameters"}
        del sample
        torch.cuda.empty_cache()
        # all ranks when the step's buffers ((2N + 14) P bytes, as the library counts them)
        # fit in free device memory less an 8 GiB margin
        try:
            z.zero_plan_check_memory(plan0, z.ZERO_ALL_RANKS, max(1, torch.cuda.mem_get_info()[0] - (8 << 30)))
            full = True
        except z.ZeroError:
            full = False
        L = P if full else S
        if full:
            grads = [synth.rank_grads(psi, P, r, 1, device=dev) for r in range(n)]
        else:
            ch = synth.chunk_grads(S, n, 1, device=dev)
            grads = [ch[q] for q in range(n)]
        master = synth.master_params(L, L, device=dev)
        m = torch.zeros(L, device=dev)
        v = torch.zeros(L, device=dev)
        param = torch.empty(L, dtype=torch.bfloat16, device=dev)
        rank = z.ZERO_ALL_RANKS if full else z.ZERO_RANK_VIEW
        byts = L * (2 * n + 26)
        for bmib in (1, 5, 25, 100):
            plan = z.zero_plan(psi, n, "zero2", bmib * MIB)
            NB = plan.n_buckets
            with torch.cuda.stream(stream):
                one = time_launches(lambda: z.zero_fused_step(plan, rank, grads, master, m, v, param, hp, 1, stream),
                                    10, stream)
                g = bucket_graph(z, plan, rank, (grads, master, m, v, param, hp, 1), 1)
                per_bucket = time_launches(lambda: g.replay(), 10, stream)
                del g
                g = bucket_graph(z, plan, rank, (grads, master, m, v, param, hp, 1), 4)
                per_bucket_4 = time_launches(lambda: g.replay(), 10, stream)
            z.zero_device_status(stream)
            line = {"sweep": "fused step", "psi": psi, "n_ranks": n, "bucket_mib": bmib, "n_buckets": NB,
                    "mode": "all ranks" if full else "rank view", "bytes_per_step": byts,
                    "single_launch_ms": one, "single_launch_gbs": byts / one / 1e6,
                    "single_launch_frac": byts / one / 1e6 / hbm_peak,
                    "per_bucket_graph_ms": per_bucket, "per_bucket_graph_gbs": byts / per_bucket / 1e6,
                    "per_bucket_graph_frac": byts / per_bucket / 1e6 / hbm_peak,
                    "per_bucket_graph_4streams_ms": per_bucket_4,
                    "per_bucket_graph_4streams_gbs": byts / per_bucket_4 / 1e6,
                    "per_bucket_graph_4streams_frac": byts / per_bucket_4 / 1e6 / hbm_peak,
                    "state_bytes_per_rank": {s: z.zero_plan(psi, n, s, bmib * MIB).state_total_bytes
                                             for s in ("ddp", "zero1", "zero2", "zero3")},
                    "peak": hbm_peak, "peak_source": peak_src, "cpu_oracle": cpu_or}
            print(json.dumps(line), flush=True)
            del g
        del grads, master, m, v, param
        torch.cuda.empty_cache()


def run_case(args):
    """Small cases for ncu captures (a few launches, about 1 GB on the device, inputs larger
    than L2). fused_small: psi = 33,554,432 flat, N = 8, all ranks, 5 fused launches.
    gemm_small: Y[2048, 14336] = X W^T with W 14336 x 4096 in 8 row shards, 5 launches."""
    import torch

    import fsdp_sharded_optimizer_zero_gb300 as z
    import synth
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    out = {"case": args.case}
    if args.case in ("fused_small", "fused_tma_small"):
        # fused_tma_small: the same step on the TMA bulk-copy pipeline (zero_set_fused_kernel(1))
        psi, n = 1 << 25, 8
        plan = z.zero_plan(psi, n, "zero2", 25 * MIB)
        grads = [synth.rank_grads(psi, psi, r, 1, device=dev) for r in range(n)]
        master = synth.master_params(psi, psi, device=dev)
        m = torch.zeros(psi, device=dev)
        v = torch.zeros(psi, device=dev)
        param = torch.empty(psi, dtype=torch.bfloat16, device=dev)
        hp = {"lr": 1e-4, "beta1": 0.9, "beta2": 0.999, "eps": 1e-8, "weight_decay": 0.0}
        z.zero_set_fused_kernel(1 if args.case == "fused_tma_small" else 0)
        try:
            ms = time_launches(lambda: z.zero_fused_step(plan, z.ZERO_ALL_RANKS, grads, master, m, v, param, hp, 1,
                                                         stream), 4, stream)
        finally:
            z.zero_set_fused_kernel(0)
        out.update(psi=psi, n_ranks=n, ms=ms, bytes=plan.fused_step_bytes, gbs=plan.fused_step_bytes / ms / 1e6)
    elif args.case == "e2e_small":
        # the e2e kernel: psi = 33,554,432, N = 8, gradients and parameters in page-locked
        # host memory (537 MB in, 67 MB out over the host link), master / m / v on the device
        psi, n = 1 << 25, 8
        plan = z.zero_plan(psi, n, "zero2", 25 * MIB)
        host_grads = [synth.rank_grads(psi, psi, r, 1).pin_memory() for r in range(n)]
        host_param = torch.empty(psi, dtype=torch.bfloat16).pin_memory()
        master = synth.master_params(psi, psi, device=dev)
        m = torch.zeros(psi, device=dev)
        v = torch.zeros(psi, device=dev)
        hp = {"lr": 1e-4, "beta1": 0.9, "beta2": 0.999, "eps": 1e-8, "weight_decay": 0.0}
        ms = time_launches(lambda: z.zero_fused_step_host(plan, z.ZERO_ALL_RANKS, host_grads, master, m, v, host_param,
                                                          hp, 1, stream), 4, stream)
        link = psi * (2 * n + 2)
        out.update(psi=psi, n_ranks=n, ms=ms, host_link_bytes=link, host_link_gbs=link / ms / 1e6)
    elif args.case == "megatron_small":
        # the Megatron distributed optimizer's step: psi = 33,554,432, N = 8, fp32 gradients
        # (4N + 26 = 58 B per parameter, 1.95 GB per launch), 5 launches
        psi, n = 1 << 25, 8
        plan = z.zero_plan(psi, n, "megatron", 25 * MIB)
        grads = [synth.rank_grads_f32(psi, psi, r, 1, device=dev) for r in range(n)]
        master = synth.master_params(psi, psi, device=dev)
        m = torch.zeros(psi, device=dev)
        v = torch.zeros(psi, device=dev)
        param = torch.empty(psi, dtype=torch.bfloat16, device=dev)
        hp = {"lr": 1e-4, "beta1": 0.9, "beta2": 0.999, "eps": 1e-8, "weight_decay": 0.0}
        ms = time_launches(lambda: z.zero_fused_step_fp32_grads(plan, z.ZERO_ALL_RANKS, grads, master, m, v, param, hp,
                                                                1, stream), 4, stream)
        out.update(psi=psi, n_ranks=n, ms=ms, bytes=plan.fused_step_bytes, gbs=plan.fused_step_bytes / ms / 1e6)
    elif args.case in ("tiny", "mistral_rank_view", "rank_view_small"):
        # tiny: psi = 2^20, N = 4, every rank in one launch (35.7 MB: L2-resident, reported as
        # such). mistral_rank_view: one rank's shard of the Mistral-7B list at N = 8
        # (S = 905,216,512; its 8 incoming chunks, 14.5 GB), ZeRO-3, 50 MiB buckets.
        # rank_view_small: the same rank-view launch on 33,554,432-element chunks (1.41 GB
        # per launch, 11x the L2), sized for an ncu capture.
        hp = {"lr": 1e-4, "beta1": 0.9, "beta2": 0.999, "eps": 1e-8, "weight_decay": 0.0}
        hbm_peak = peaks()[0]
        if args.case == "tiny":
            psi, n = 1 << 20, 4
            plan = z.zero_plan(psi, n, "zero2", 25 * MIB)
            grads = [synth.rank_grads(psi, psi, r, 1, device=dev) for r in range(n)]
            L, rank = psi, z.ZERO_ALL_RANKS
        else:
            psi, n = (synth.MISTRAL_7B_PSI if args.case == "mistral_rank_view" else 8 << 25), 8
            plan = z.zero_plan(psi, n, "zero3", 50 * MIB)
            L, rank = plan.shard_elems, z.ZERO_RANK_VIEW
            ch = synth.chunk_grads(L, n, 1, device=dev)
            grads = [ch[q] for q in range(n)]
        master = synth.master_params(L, L, device=dev)
        m = torch.zeros(L, device=dev)
        v = torch.zeros(L, device=dev)
        param = torch.empty(L, dtype=torch.bfloat16, device=dev)
        ms = time_launches(lambda: z.zero_fused_step(plan, rank, grads, master, m, v, param, hp, 1, stream),
                           4 if args.case == "rank_view_small" else 20, stream)
        byts = L * (2 * n + 26)
        out.update(params_per_step=L, n_ranks=n, ms=ms, bytes=byts, gbs=byts / ms / 1e6,
                   frac=byts / ms / 1e6 / hbm_peak, params_per_s=L / ms * 1e3,
                   l2_resident=byts < 129e6)
    elif args.case in ("gemm_small", "gemm_w_up"):
        # gemm_small: 2048 tokens; gemm_w_up: the full Mistral W_up shape, 8192 tokens
        # (X 64 MB, W 117 MB in 8 row shards, Y 470 MB fp32: under 1 GB on the device)
        M, R, K, n = (2048 if args.case == "gemm_small" else 8192), 14336, 4096, 8
        X = synth.activations(M, K, device=dev)
        shards = synth.weight_shards(R, K, n, device=dev)
        Y = torch.empty(M, R, device=dev)
        ms = time_launches(lambda: z.fsdp_unit_forward(shards, X, Y, stream=stream), 4, stream)
        out.update(M=M, R=R, K=K, ms=ms, tflops=2.0 * M * R * K / ms / 1e9)
    elif args.case == "mlp_unit":
        # Mistral MLP unit at 8192 tokens: gate-up kernel (silu epilogue) + down GEMM
        M, n = 8192, 8
        X = synth.activations(M, 4096, device=dev)
        gs = synth.weight_shards(14336, 4096, n, device=dev, seed_key=1)
        us = synth.weight_shards(14336, 4096, n, device=dev, seed_key=2)
        ds = synth.weight_shards(4096, 14336, n, device=dev, seed_key=3)
        H = torch.empty(M, 14336, dtype=torch.bfloat16, device=dev)
        Y = torch.empty(M, 4096, device=dev)
        ms = time_launches(lambda: z.fsdp_mlp_forward(gs, us, ds, X, H, Y, stream=stream), 4, stream)
        out.update(M=M, ms=ms, tflops=3 * 2.0 * M * 14336 * 4096 / ms / 1e9)
    elif args.case == "legs_small":
        # the standalone step kernels on psi = 33,554,432 flat, N = 8, all ranks (1.1 GB of
        # inputs): DDP all-reduce (reduce_vec_kernel<8>), Adam with the bf16 cast
        # (adam_vec_kernel), the parameter all-gather (allgather_kernel); 3 launches each
        psi, n = 1 << 25, 8
        plan = z.zero_plan(psi, n, "ddp", 25 * MIB)
        S = plan.shard_elems
        grads = [synth.rank_grads(psi, psi, r, 1, device=dev) for r in range(n)]
        g = torch.empty(psi, device=dev)
        master = synth.master_params(psi, psi, device=dev)
        m = torch.zeros(psi, device=dev)
        v = torch.zeros(psi, device=dev)
        param = torch.empty(psi, dtype=torch.bfloat16, device=dev)
        hp = {"lr": 1e-4, "beta1": 0.9, "beta2": 0.999, "eps": 1e-8, "weight_decay": 0.0}
        ms_ar = time_launches(lambda: z.ddp_allreduce(plan, grads, g, stream), 2, stream)
        ms_ad = time_launches(lambda: z.zero_adam_step(plan, z.ZERO_ALL_RANKS, g, master, m, v, param, hp, 1, stream),
                              2, stream)
        ms_ag = time_launches(lambda: z.zero_allgather_params(plan, [master[r * S:(r + 1) * S] for r in range(n)],
                                                              param, stream), 2, stream)
        out.update(psi=psi, n_ranks=n, allreduce_ms=ms_ar, adam_ms=ms_ad, allgather_ms=ms_ag,
                   allreduce_bytes=psi * (2 * n + 4), adam_bytes=psi * 30, allgather_bytes=psi * 6)
    elif args.case == "gather_w_up":
        # W_up [14336, 4096] bf16 from 8 row shards: the materialised all-gather
        # (fsdp_gather_rows) and the transposed gather W^T (fsdp_transpose_cat, which the
        # backward's fallback path uses for shapes the in-place GEMMs do not take); 235 MB
        # moved per launch each, 3 launches each
        n, R, K = 8, 14336, 4096
        shards = synth.weight_shards(R, K, n, device=dev)
        W = torch.empty(R, K, dtype=torch.bfloat16, device=dev)
        Wt = torch.empty(K, R, dtype=torch.bfloat16, device=dev)
        ms_g = time_launches(lambda: z.fsdp_gather_rows(shards, W, stream=stream), 2, stream)
        ms_t = time_launches(lambda: z.fsdp_transpose_cat(shards, Wt, stream=stream), 2, stream)
        byts = 4 * R * K
        out.update(R=R, K=K, n_ranks=n, gather_ms=ms_g, transpose_ms=ms_t, bytes=byts,
                   gather_gbs=byts / ms_g / 1e6, transpose_gbs=byts / ms_t / 1e6)
    elif args.case in ("zero3_step", "zero3_unit_small"):
        # one ZeRO-3 step over the 4 Mistral-shaped units, N = 8 ranks x 1024 tokens, each
        # rank's Adam fused into the dW GEMMs (about 7 GB on the device), 3 steps;
        # zero3_unit_small: the second unit alone (W [4096, 14336], about 1.4 GB): per step
        # its forward GEMM, dX GEMM and fused dW GEMM
        n, m = 8, 1024
        shapes = ZERO3_SHAPES if args.case == "zero3_step" else ZERO3_SHAPES[1:2]
        units = zero3_units(z, synth, dev, n, m, shapes=shapes)
        flags = 0  # each rank's Adam fused into the dW GEMMs
        units = [{k: v for k, v in u.items() if k != "dw"} for u in units]
        wsb = z.fsdp_zero3_step_workspace(n, shapes, m, flags)
        ws = torch.empty(wsb, dtype=torch.uint8, device=dev) if wsb else None
        y = torch.empty(n * m, shapes[-1][0], dtype=torch.bfloat16, device=dev)
        dx = torch.empty(n * m, shapes[0][1], dtype=torch.bfloat16, device=dev)
        side = torch.cuda.Stream()
        hp = {"lr": 1e-4, "beta1": 0.9, "beta2": 0.999, "eps": 1e-8, "weight_decay": 0.0}
        ms = time_launches(lambda: z.fsdp_zero3_step(units, m, hp, 1, y_out=y, dx_out=dx, flags=flags, workspace=ws,
                                                     stream=stream, prefetch_stream=side), 2, stream)
        flop = sum(6.0 * n * m * R * K for R, K in shapes)
        out.update(n_ranks=n, tokens_per_rank=m, units=len(shapes), ms=ms, tflops=flop / ms / 1e9)
    elif args.case in ("zero3_mlp_step", "zero3_mlp_small"):
        # one ZeRO-3 step over 2 Mistral-7B MLP units, N = 8 ranks x 1024 tokens (about
        # 10 GB on the device), 3 steps; zero3_mlp_small: one unit, 8 x 256 tokens (2.7 GB)
        n, m, nu = (8, 1024, MLP_UNITS) if args.case == "zero3_mlp_step" else (8, 256, 1)
        units = zero3_mlp_units(z, synth, dev, n, m, n_units=nu)
        ws = torch.empty(z.fsdp_zero3_mlp_step_workspace(n, [(4096, 14336)] * nu, m), dtype=torch.uint8,
                         device=dev)
        y = torch.empty(n * m, 4096, dtype=torch.bfloat16, device=dev)
        dx = torch.empty(n * m, 4096, dtype=torch.bfloat16, device=dev)
        hp = {"lr": 1e-4, "beta1": 0.9, "beta2": 0.999, "eps": 1e-8, "weight_decay": 0.0}
        units = [{k: v for k, v in u.items() if k not in ("dw_gu", "dw_down")} for u in units]  # fused Adam
        ms = time_launches(lambda: z.fsdp_zero3_mlp_step(units, m, hp, 1, y_out=y, dx_out=dx, workspace=ws,
                                                         stream=stream), 2, stream)
        flop = nu * 9 * 2.0 * n * m * 4096 * 14336
        out.update(n_ranks=n, tokens_per_rank=m, units=nu, ms=ms, tflops=flop / ms / 1e9)
    elif args.case == "backward_up":
        # FSDP unit backward of W_up [14336, 4096] in 8 row shards, 2048 tokens per rank
        # (dY 470 MB, X 134 MB, dX 268 MB, dW 235 MB, no workspace): 2 launches (dX GEMM,
        # dW GEMM) per call, 4 calls
        n, R, K, M = 8, 14336, 4096, 2048
        shards = synth.weight_shards(R, K, n, device=dev, seed_key=11)
        A = [synth.activations(M, K, device=dev, seed_key=q) for q in range(n)]
        dY = [synth.upstream_grad(M, R, device=dev, seed_key=q) for q in range(n)]
        dX = [torch.empty(M, K, device=dev) for _ in range(n)]
        dW = torch.empty(R, K, device=dev)
        ws = torch.empty(z.fsdp_unit_backward_workspace(n, R, K, M), dtype=torch.uint8, device=dev)
        ms = time_launches(lambda: z.fsdp_unit_backward(shards, A, dY, dX, dW, ws, stream=stream), 3, stream)
        out.update(n_ranks=n, R=R, K=K, M=M, ms=ms, tflops=4.0 * n * M * R * K / ms / 1e9,
                   workspace_bytes=ws.numel())
    else:
        raise SystemExit(f"unknown case {args.case}")
    z.zero_device_status(stream)
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--case", default=None,
                    help="one measured case: fused_small | fused_tma_small | megatron_small | e2e_small | legs_small | gather_w_up | gemm_small | gemm_w_up | mlp_unit | "
                         "backward_up | rank_view_small | zero3_step | zero3_unit_small (ncu-sized) | zero3_mlp_step | "
                         "zero3_mlp_small (ncu-sized) | "
                         "tiny | mistral_rank_view")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-seconds", type=float, default=60.0)
    ap.add_argument("--no-legs", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--leg-idle-s", type=float, default=2.0,
                    help="seconds the GPU idles before each tensor-core leg group")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours" and not args.sweep:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
        return
    import __graft_entry__ as g
    g.build()
    if args.case:
        run_case(args)
    elif args.sweep:
        run_sweep(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
