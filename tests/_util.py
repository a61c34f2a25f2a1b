"""Helpers shared by the test files (comparison of raw bits, tensor <-> numpy)."""
from __future__ import annotations

import numpy as np
import torch


def bits16(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy().astype(np.float32, copy=False)


def from_bits16(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16).copy()).view(torch.bfloat16).to(device)


def assert_f32_identical(got: np.ndarray, want: np.ndarray, what: str):
    """Bit-identical fp32, with any NaN accepted for NaN (NaN payloads are not unique)."""
    got = np.ascontiguousarray(got, dtype=np.float32)
    want = np.ascontiguousarray(want, dtype=np.float32)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    same = (got.view(np.uint32) == want.view(np.uint32)) | (np.isnan(got) & np.isnan(want))
    if not same.all():
        bad = np.flatnonzero(~same)
        i = bad[0]
        raise AssertionError(f"{what}: {bad.size} of {got.size} differ; first at {i}: got {got.flat[i]!r} "
                             f"want {want.flat[i]!r}")


def assert_bf16_identical(got: np.ndarray, want: np.ndarray, what: str):
    got = np.ascontiguousarray(got, dtype=np.uint16)
    want = np.ascontiguousarray(want, dtype=np.uint16)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    gn = ((got & 0x7F80) == 0x7F80) & ((got & 0x007F) != 0)
    wn = ((want & 0x7F80) == 0x7F80) & ((want & 0x007F) != 0)
    same = (got == want) | (gn & wn)
    if not same.all():
        bad = np.flatnonzero(~same)
        i = bad[0]
        raise AssertionError(f"{what}: {bad.size} of {got.size} differ; first at {i}: got {got.flat[i]:#06x} "
                             f"want {want.flat[i]:#06x}")
