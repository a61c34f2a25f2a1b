"""Seeded random cases of the step, every element compared bit for bit with the oracle:
psi, N (1..64), stage, bucket size, rank mode, misaligned buffers, steps and starting
moments drawn from a fixed generator, plus four long launches (tens of millions of
elements, odd psi): N = 2 and 17 on the 4-CTA-per-SM grid (N = 17 through the generic-N
load groups, which serve N > 16), N = 3 and 5 on the full grid."""
import numpy as np
import pytest

from test_step_parity import compare, gpu_run, make_inputs, oracle_run, z  # noqa: F401  (z: fixture)

pytestmark = pytest.mark.gpu

MODES = ("all", "all_buckets", "ranks", "buckets", "rank_view", "unfused", "unfused_ag", "ddp")
STAGES = ("ddp", "zero1", "zero2", "zero3")


def draw(i):
    rng = np.random.default_rng(1000 + i)
    n = int(rng.choice([1, 2, 3, 4, 5, 7, 8, 12, 16, 31, 64]))
    psi = int(rng.integers(1, 300_000))
    stage = str(rng.choice(STAGES))
    mode = str(rng.choice(MODES))
    S = -(-psi // n)
    # bucket: anywhere from one element per rank to more than the shard, but keep the number
    # of per-bucket launches bounded
    lo = max(2 * n, (2 * n * S) // 300 if mode in ("all_buckets", "buckets") else 2 * n)
    hi = max(lo + 1, 4 * n * S + 2 * n)
    bb = int(np.exp(rng.uniform(np.log(lo), np.log(hi))))  # log-uniform
    return dict(psi=psi, n=n, stage=stage, mode=mode, bb=bb, misalign=bool(rng.random() < 0.15),
                steps=int(rng.integers(1, 3)), moments=bool(rng.random() < 0.5), seed=i)


@pytest.mark.parametrize("i", range(24))
def test_random_step_bit_exact(z, i):
    c = draw(i)
    master0, m0, v0, grads = make_inputs(c["psi"], c["n"], c["steps"], seed=c["seed"], moments=c["moments"])
    want = oracle_run(c["stage"], c["psi"], c["n"], c["bb"], master0, m0, v0, grads)
    got = gpu_run(z, c["stage"], c["mode"], c["psi"], c["n"], c["bb"], master0, m0, v0, grads,
                  misalign=c["misalign"])
    compare(got, want, str(c))


@pytest.mark.parametrize("psi,n", [(20_000_001, 2), (21_000_003, 3), (19_999_997, 5), (20_000_017, 17)])
def test_long_launch_bit_exact(z, psi, n):
    master0, m0, v0, grads = make_inputs(psi, n, 1, seed=psi % 97)
    want = oracle_run("zero2", psi, n, 25 << 20, master0, m0, v0, grads)
    got = gpu_run(z, "zero2", "all", psi, n, 25 << 20, master0, m0, v0, grads)
    compare(got, want, f"long launch psi={psi} N={n}")
