"""The C ABI from plain C: tests/c_abi_plan.c includes include/zero.h, is compiled as C99
with every warning an error, links against the built library and calls its host-side
entry points (plan, query, bucket ranges, argument errors). Its printed layouts must equal
the oracle's. CPU only: nothing here launches a kernel."""
import shutil
import subprocess
from pathlib import Path

import pytest

from oracle import zero_oracle as O

ROOT = Path(__file__).resolve().parents[1]
STAGES = {0: "ddp", 1: "zero1", 2: "zero2", 3: "zero3", 4: "megatron"}


@pytest.fixture(scope="module")
def z():
    import __graft_entry__ as g
    g.build()
    import fsdp_sharded_optimizer_zero_gb300 as z
    return z


@pytest.fixture(scope="module")
def c_output(z, tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib_dir = Path(z.library()._name).parent
    exe = tmp_path_factory.mktemp("c_abi") / "c_abi_plan"
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", str(ROOT / "include"),
           str(ROOT / "tests" / "c_abi_plan.c"), "-o", str(exe), "-L", str(lib_dir), "-lzero_gb300",
           f"-Wl,-rpath,{lib_dir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    return r.stdout.splitlines()


def test_c_program_sees_the_oracle_layout(c_output):
    plans = [ln for ln in c_output if ln.startswith("plan ")]
    assert len(plans) == 5
    for ln in plans:
        head, body, buckets = ln.split("|")
        psi, n, stage, bb = (int(x) for x in head.split()[1:])
        f = [int(x) for x in body.split()]
        lay = O.make_layout(psi, n, bb)
        assert f[:5] == [lay.psi, lay.psi_padded, lay.shard, lay.bucket_elems, lay.n_buckets]
        mb = O.model_state_bytes(STAGES[stage], lay)
        assert f[5:11] == [mb["param"], mb["grad"], mb["master"], mb["m"], mb["v"], mb["total"]]
        c = O.comm_elements(STAGES[stage], lay)
        assert f[11:15] == [c["reduce_scatter"], c["all_gather_fwd"], c["all_gather_bwd"], c["total"]]
        assert f[15] == O.ring_sent_elements(c["total"], n)
        assert f[16] == lay.psi_padded * ((4 if stage == 4 else 2) * n + 26)
        # first and last bucket of the last rank: [r S + k C, r S + min((k + 1) C, S))
        r, S, C, nb = n - 1, lay.shard, lay.bucket_elems, lay.n_buckets
        want = [r * S, r * S + min(C, S), r * S + (nb - 1) * C, r * S + min(nb * C, S)]
        assert [int(x) for x in buckets.split()] == want


def test_c_program_gets_error_codes_and_messages(c_output):
    errs = [ln for ln in c_output if ln.startswith("error ")]
    assert len(errs) == 5
    assert all(ln.split()[1] == "-1" and len(ln.split()) > 2 for ln in errs)
    assert any("n_ranks 0" in ln for ln in errs) and any("NULL" in ln for ln in errs)
