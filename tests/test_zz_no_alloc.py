"""The allocation-free FSDP unit forward (fsdp_unit_forward_static_scratch).

Some callers cannot allocate device memory where they run the unit: a plug-in inside a
framework that owns every byte of device memory through its own pool, or a latency-
critical path that cannot afford cudaMalloc's device-wide synchronisation. For them the
library keeps the gathered weight in a fixed 16 MiB device array of its own. This test
calls that entry point through the C ABI twice in a row, with different inputs each
time, and checks each output against the regular entry point (fsdp_unit_forward with a
caller-provided scratch, or none when the shards tile the GEMM) within the tolerance the
GEMM tests use:
    |Y_static - Y_regular| <= (K + 1) * 2^-23 * sum_k |a_k w_k|.
It lives in its own file, collected last, and passes alone or after the other tests.
"""
from __future__ import annotations

import ctypes as C

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def z():
    import __graft_entry__ as g
    g.build()
    import fsdp_sharded_optimizer_zero_gb300 as z
    return z


def call_static(z, shards, A, Y, Yb=None):
    lib = z.library()
    f = lib.fsdp_unit_forward_static_scratch
    f.restype = C.c_int
    f.argtypes = [C.c_int, C.POINTER(C.c_void_p), C.c_int64, C.c_int64, C.c_void_p, C.c_int64, C.c_void_p,
                  C.c_void_p, C.c_void_p]
    ptrs = (C.c_void_p * len(shards))(*[s.data_ptr() for s in shards])
    rows = sum(int(s.shape[0]) for s in shards)
    rc = f(len(shards), ptrs, rows, int(A.shape[1]), A.data_ptr(), int(A.shape[0]), Y.data_ptr(),
           Yb.data_ptr() if Yb is not None else None, torch.cuda.current_stream().cuda_stream)
    return rc, lib.zero_last_error().decode()


def tolerance(A, shards):
    a = A.float().double().abs().cpu().numpy()
    w = torch.cat(shards, 0).float().double().abs().cpu().numpy()
    return (A.shape[1] + 1) * 2.0 ** -23 * (a @ w.T)


def run_and_compare(z, m, rows, k, n, key, scratch_regular):
    """One call of the allocation-free entry point against fsdp_unit_forward on the same
    inputs; returns the free device bytes measured around the call."""
    shards = synth.weight_shards(rows, k, n, device=DEV, seed_key=key)
    A = synth.activations(m, k, device=DEV, seed_key=key)
    y_ref = torch.empty(m, rows, device=DEV)
    scratch = torch.empty(rows, k, dtype=torch.bfloat16, device=DEV) if scratch_regular else None
    z.fsdp_unit_forward(shards, A, y_ref, scratch_w=scratch)
    y = torch.full((m, rows), float("nan"), device=DEV)
    yb = torch.zeros(m, rows, dtype=torch.bfloat16, device=DEV)
    torch.cuda.synchronize()
    before = (torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0])
    rc, msg = call_static(z, shards, A, y, yb)
    assert rc == 0, msg
    z.zero_device_status()
    after = (torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0])
    diff = (y.double() - y_ref.double()).abs().cpu().numpy()
    assert np.all(diff <= tolerance(A, shards)), f"{(m, rows, k, n)}: outside the GEMM tolerance"
    assert torch.equal(yb, y.to(torch.bfloat16)), f"{(m, rows, k, n)}: bf16 output is not RNE of the fp32 output"
    return before, after


def test_static_scratch_forward_matches_regular_entry_point(z):
    # shard rows of 100 and 96 do not tile the GEMM's 128-row W loads, so the unit needs
    # the gathered W: the regular call gets a caller buffer, the new one the library's
    # array. Two calls in a row with different shapes and inputs; the first call also
    # loads the library's module on this device, so only the second is held to "frees and
    # allocates nothing" by cudaMemGetInfo, which sees any allocation in the process.
    cases = [(130, 3 * 100, 72, 3, 2), (200, 8 * 96, 256, 8, 3)]
    for call, case in enumerate(cases):
        before, after = run_and_compare(z, *case, scratch_regular=True)
        assert after[0] == before[0], f"call {call}: torch's allocator grew"
        if call > 0:
            assert after[1] == before[1], f"call {call}: free device memory changed"


def test_static_scratch_tiling_shards_need_no_array(z):
    # shards of a multiple of 128 rows tile the GEMM: W is read straight from them, so the
    # 16 MiB limit does not apply (W_up of a Mistral-7B MLP, 14336 x 4096 in 8 shards)
    before, after = run_and_compare(z, 256, 14336, 4096, 8, 4, scratch_regular=False)
    assert after == before


def test_static_scratch_rejects_weights_above_the_limit(z):
    # 2 shards of 2056 rows (not a multiple of 128): a gather would be needed, and
    # 4112 x 4104 > 8,388,608 elements
    n, rows, k = 2, 2 * 2056, 4096 + 8
    shards = [torch.empty(rows // n, k, dtype=torch.bfloat16, device=DEV) for _ in range(n)]
    A = torch.empty(128, k, dtype=torch.bfloat16, device=DEV)
    Y = torch.empty(128, rows, device=DEV)
    rc, msg = call_static(z, shards, A, Y)
    assert rc == -1 and "exceeds the static scratch" in msg
