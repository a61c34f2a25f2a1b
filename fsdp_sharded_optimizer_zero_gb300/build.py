"""Build libzero_gb300.so in-tree: nvcc for sm_103a, one object per translation unit
compiled in parallel, then one shared-library link. No CMake, no torch extension (the C
ABI carries no torch types). Rebuilds only when a source, header or flag changed."""
from __future__ import annotations

import fcntl
import hashlib
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
BUILD = PKG / "_build"
LIB = PKG / "libzero_gb300.so"
SOURCES = ["capi.cu", "fused_step.cu", "step_kernels.cu", "fsdp_gemm.cu", "fsdp_unit.cu", "fsdp_zero3.cu",
           "fsdp_static_scratch.cu"]
HEADERS = ["internal.h", "device_common.cuh", "step_common.cuh", "tcgen05.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = [
    "-O3", "-std=c++17", "-lineinfo", *ARCH,
    # IEEE fp32 everywhere: no contraction into FMA, correctly rounded div / sqrt, no FTZ
    "-fmad=false", "-prec-div=true", "-prec-sqrt=true", "-ftz=false",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-ffp-contract=off", "-Xcompiler", "-fvisibility=hidden",
    "-I", str(ROOT / "include"),
]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and Path(c).exists():
            return c
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libzero_gb300.so")


def _digest() -> str:
    h = hashlib.sha256()
    for name in SOURCES + HEADERS:
        p = CSRC / name
        if p.exists():
            h.update(name.encode())
            h.update(p.read_bytes())
    h.update((ROOT / "include" / "zero.h").read_bytes())
    h.update(" ".join(FLAGS).encode())
    h.update(os.uname().machine.encode())
    return h.hexdigest()


def build(verbose: bool = False, force: bool = False) -> Path:
    digest = _digest()
    stamp = BUILD / "stamp"
    if not force and LIB.exists() and stamp.exists() and stamp.read_text() == digest:
        return LIB
    BUILD.mkdir(exist_ok=True)
    # one builder at a time (several ranks of one job may call build() together)
    with open(BUILD / "lock", "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        try:
            if not force and LIB.exists() and stamp.exists() and stamp.read_text() == digest:
                return LIB
            return _build_locked(digest, stamp, verbose)
        finally:
            fcntl.flock(lock, fcntl.LOCK_UN)


def _build_locked(digest: str, stamp: Path, verbose: bool) -> Path:
    cc = nvcc()

    def compile_one(src: str) -> Path:
        obj = BUILD / (src + ".o")
        cmd = [cc, *FLAGS, "-c", str(CSRC / src), "-o", str(obj)]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB.with_suffix(".so.tmp")
    r = subprocess.run([cc, "-shared", *ARCH, "-o", str(tmp), *map(str, objs)], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    stamp.write_text(digest)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
