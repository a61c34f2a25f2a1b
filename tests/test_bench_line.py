"""bench.py's JSON line (GPU): a short run prints one line with the keys the measurement
contract asks for, and a roofline whose numbers are consistent with each other."""
import json
import subprocess
import sys
from pathlib import Path

import pytest

pytestmark = pytest.mark.gpu
ROOT = Path(__file__).resolve().parents[1]


def test_bench_prints_one_complete_line():
    r = subprocess.run([sys.executable, str(ROOT / "bench.py"), "--steps", "5", "--warmup", "3", "--no-legs",
                        "--no-cpu-baseline", "--e2e-steps", "2"], capture_output=True, text=True, timeout=900,
                       cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "clocks", "gpu_launches", "e2e"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3 and d["gpu_launches"] == 5
    assert d["value"] > 0 and d["higher_is_better"] is True and d["scaling"] == "weak"
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    # the Mistral-7B rank view at N = 8: a 905,216,512-element shard, 2N + 26 bytes each
    S = 905_216_512
    assert d["config"]["shard_elems"] == S and d["config"]["n_ranks"] == 8 and d["config"]["stage"] == "zero3"
    assert rf["algorithmic_bytes_per_launch"] == S * (2 * 8 + 26)
    assert d["ms_per_step"] * 1e-3 * d["value"] == pytest.approx(S, rel=1e-9)
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(d["clocks"])
    e2e = d["e2e"]
    assert e2e["unit"] == d["unit"] and e2e["value"] > 0
    L = e2e["elems_per_step"]
    assert 0 < L <= S and e2e["whole_shard"] == (L == S)
    assert e2e["h2d_bytes_per_step"] == 8 * L * 2 and e2e["d2h_bytes_per_step"] == L * 2
