"""CPU oracle for the ZeRO partitioned mixed-precision Adam step.

TEST INFRASTRUCTURE ONLY.  Only the test-suite, ``__graft_entry__.smoke()`` and
the benchmark's CPU-baseline leg may import this package.  It shares no code
with the CUDA library (``zero_sharded_mixed_shard_gb300``) and never imports
it.

* :mod:`oracle.adam_oracle` (``adam_oracle.c``) -- the per-element step in
  plain C: binary16 conversion written from the format's definition, the
  gradient mean, the three Adam readings and the cast, each one IEEE binary32
  operation in a fixed order.  Built with ``gcc -ffp-contract=off``.
* :mod:`oracle.layout` -- the ceil partition, the shard/tensor segment table
  and the per-rank memory and communication accounting, in plain Python.

numpy-level wrappers are below; they take and return numpy arrays only.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

from . import layout  # noqa: F401  (re-export)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "adam_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-Wall",
           "-fPIC", "-shared", "-pthread"]

_lib = None


def build(force: bool = False) -> str:
    """Compile ``adam_oracle.c`` into ``oracle/_build/liboracle.so`` with gcc."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_BUILD_DIR)
    os.close(fd)
    cmd = ["gcc", *_CFLAGS, _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    # ZERO_ORACLE_LIB points the pins at another build of adam_oracle.c (the
    # mutation test plants mistakes in copies of it to show the pins fail)
    lib = ctypes.CDLL(os.environ.get("ZERO_ORACLE_LIB") or build())
    i64, i32, f32, f64, vp = (ctypes.c_int64, ctypes.c_int32, ctypes.c_float,
                              ctypes.c_double, ctypes.c_void_p)
    lib.oracle_half_to_float.argtypes = [ctypes.c_uint16]
    lib.oracle_half_to_float.restype = f32
    lib.oracle_float_to_half.argtypes = [f32]
    lib.oracle_float_to_half.restype = ctypes.c_uint16
    lib.oracle_half_to_float_array.argtypes = [vp, vp, i64]
    lib.oracle_float_to_half_array.argtypes = [vp, vp, i64]
    lib.oracle_adam_elems.argtypes = [vp, i64, i32, vp, vp, vp, vp, i64, i64,
                                      f32, f32, f32, f32, i32, i32]
    lib.oracle_adam_elems.restype = ctypes.c_int
    lib.oracle_zero_step.argtypes = [vp, i64, i32, i64, vp, vp, vp, vp, i64,
                                     f32, f32, f32, f32, i32, i32]
    lib.oracle_zero_step.restype = ctypes.c_int
    lib.oracle_offload_elems.argtypes = [vp, i64, i32, vp, vp, vp, vp, vp, i64, i64,
                                         f32, f32, f32, f32, i32]
    lib.oracle_offload_elems.restype = ctypes.c_int
    lib.oracle_adam_elems_f64.argtypes = [vp, i64, i32, vp, vp, vp, i64, i64,
                                          f64, f64, f64, f64, i32]
    lib.oracle_adam_elems_f64.restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _as_u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    assert a.dtype == np.uint16
    return a


def half_to_float(h) -> np.ndarray:
    """binary16 codes (uint16 or float16 array) -> float32 values."""
    h = _as_u16(h)
    out = np.empty(h.shape, np.float32)
    _load().oracle_half_to_float_array(_ptr(h), _ptr(out), h.size)
    return out


def float_to_half(f) -> np.ndarray:
    """float32 values -> binary16 codes (uint16), round to nearest even."""
    f = np.ascontiguousarray(f, dtype=np.float32)
    out = np.empty(f.shape, np.uint16)
    _load().oracle_float_to_half_array(_ptr(f), _ptr(out), f.size)
    return out


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what} failed with status {rc}")


def adam_elems(grads, rank_stride: int, P: int, master: np.ndarray, m: np.ndarray,
               v: np.ndarray, t: int, lr: float, b1: float, b2: float, eps: float,
               mode: int, threads: int = 1, params_out: np.ndarray | None = None
               ) -> np.ndarray:
    """Elementwise step over ``n = master.size`` elements, in place on
    master / m / v.  ``grads`` is a flat uint16 array holding rank r's n codes
    at ``r * rank_stride``.  Returns the fp16 codes of the new weights."""
    g = _as_u16(grads).reshape(-1)
    n = master.size
    for a in (master, m, v):
        assert a.dtype == np.float32 and a.size == n and a.flags["C_CONTIGUOUS"]
    assert P >= 1 and (n == 0 or g.size >= (P - 1) * rank_stride + n)
    out = params_out if params_out is not None else np.empty(n, np.uint16)
    assert out.dtype == np.uint16 and out.size == n
    rc = _load().oracle_adam_elems(_ptr(g), rank_stride, P, _ptr(master), _ptr(m),
                                   _ptr(v), _ptr(out), n, t, lr, b1, b2, eps, mode,
                                   threads)
    _check(rc, "adam_elems")
    return out


def zero_step(grads, rank_stride: int, P: int, N: int, master: np.ndarray,
              m: np.ndarray, v: np.ndarray, params: np.ndarray, t: int, lr: float,
              b1: float, b2: float, eps: float, mode: int, threads: int = 1) -> None:
    """Whole ZeRO step (reduce-scatter, shard update, cast, all-gather) over N
    parameters, in place on master / m / v / params (uint16 codes)."""
    g = _as_u16(grads).reshape(-1)
    assert rank_stride >= N and g.size >= (P - 1) * rank_stride + N
    for a in (master, m, v):
        assert a.dtype == np.float32 and a.size == N and a.flags["C_CONTIGUOUS"]
    assert params.dtype == np.uint16 and params.size == N
    rc = _load().oracle_zero_step(_ptr(g), rank_stride, P, N, _ptr(master), _ptr(m),
                                  _ptr(v), _ptr(params), t, lr, b1, b2, eps, mode,
                                  threads)
    _check(rc, "zero_step")


def adam_elems_f64(grads, rank_stride: int, P: int, w: np.ndarray, m: np.ndarray,
                   v: np.ndarray, t: int, lr: float, b1: float, b2: float, eps: float,
                   mode: int) -> None:
    """The same formulas in double precision (state in float64, in place)."""
    g = _as_u16(grads).reshape(-1)
    n = w.size
    for a in (w, m, v):
        assert a.dtype == np.float64 and a.size == n and a.flags["C_CONTIGUOUS"]
    rc = _load().oracle_adam_elems_f64(_ptr(g), rank_stride, P, _ptr(w), _ptr(m),
                                       _ptr(v), n, t, lr, b1, b2, eps, mode)
    _check(rc, "adam_elems_f64")


def offload_elems(grads, rank_stride: int, P: int, master: np.ndarray, m: np.ndarray,
                  v: np.ndarray, t: int, lr: float, b1: float, b2: float, eps: float,
                  mode: int) -> tuple[np.ndarray, np.ndarray]:
    """ZeRO-Offload's elementwise step (gradient mean crosses to the CPU as
    fp16), in place on master / m / v.  Returns (fp16 codes of the new
    weights, fp16 codes of the gradient that crossed)."""
    g = _as_u16(grads).reshape(-1)
    n = master.size
    for a in (master, m, v):
        assert a.dtype == np.float32 and a.size == n and a.flags["C_CONTIGUOUS"]
    assert P >= 1 and (n == 0 or g.size >= (P - 1) * rank_stride + n)
    out = np.empty(n, np.uint16)
    g16 = np.empty(n, np.uint16)
    rc = _load().oracle_offload_elems(_ptr(g), rank_stride, P, _ptr(master), _ptr(m), _ptr(v),
                                      _ptr(out), _ptr(g16), n, t, lr, b1, b2, eps, mode)
    _check(rc, "offload_elems")
    return out, g16
