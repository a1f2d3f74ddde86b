"""Shared helpers of the GPU parity tests: ulp distances and the tolerance of
the fused step against the oracle (2 fp32 ulp on master / m / v, 1 fp16 ulp
on the gathered parameters; NaN matches NaN)."""
from __future__ import annotations

import numpy as np

F32_ULP_TOL = 2
F16_ULP_TOL = 1


# Floats mapped to integers in value order, one step per representable value,
# with -0 one step below +0: a distance of 0 then means identical bits (NaN
# payloads aside), so a zero of the wrong sign is caught.
def _ordered32(x: np.ndarray) -> np.ndarray:
    i = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.int64)
    mag = i & 0x7FFFFFFF
    return np.where(i & 0x80000000, -mag - 1, mag)


def _ordered16(codes: np.ndarray) -> np.ndarray:
    i = np.ascontiguousarray(codes).view(np.uint16).astype(np.int64)
    mag = i & 0x7FFF
    return np.where(i & 0x8000, -mag - 1, mag)


def ulp32(a: np.ndarray, b: np.ndarray) -> int:
    """Largest distance in binary32 ulps between a and b (NaN == NaN)."""
    a = np.asarray(a, np.float32).ravel()
    b = np.asarray(b, np.float32).ravel()
    if a.size == 0:
        return 0
    na, nb = np.isnan(a), np.isnan(b)
    if np.any(na != nb):
        return 1 << 40
    keep = ~na
    if not keep.any():
        return 0
    return int(np.max(np.abs(_ordered32(a[keep]) - _ordered32(b[keep]))))


def ulp16(a: np.ndarray, b: np.ndarray) -> int:
    """Largest distance in binary16 ulps between two code arrays (NaN == NaN)."""
    a = np.asarray(a).view(np.uint16).ravel()
    b = np.asarray(b).view(np.uint16).ravel()
    if a.size == 0:
        return 0
    na = ((a & 0x7C00) == 0x7C00) & ((a & 0x3FF) != 0)
    nb = ((b & 0x7C00) == 0x7C00) & ((b & 0x3FF) != 0)
    if np.any(na != nb):
        return 1 << 40
    keep = ~na
    if not keep.any():
        return 0
    return int(np.max(np.abs(_ordered16(a[keep]) - _ordered16(b[keep]))))


def assert_close(gpu_state, ref_state, what=""):
    """gpu_state / ref_state: (master, m, v, params codes) as numpy arrays."""
    names = ("master", "m", "v")
    for name, g, r in zip(names, gpu_state[:3], ref_state[:3]):
        d = ulp32(g, r)
        assert d <= F32_ULP_TOL, f"{what} {name}: {d} fp32 ulp"
    d = ulp16(gpu_state[3], ref_state[3])
    assert d <= F16_ULP_TOL, f"{what} params: {d} fp16 ulp"


def max_ulps(gpu_state, ref_state):
    return (max(ulp32(g, r) for g, r in zip(gpu_state[:3], ref_state[:3])),
            ulp16(gpu_state[3], ref_state[3]))
