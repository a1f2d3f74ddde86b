"""Python binding of the fused ZeRO step library (``libzero_step.so``).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels (or, for the layout table, in its host C++).  The functions carry the
C-ABI's names; tensors are torch tensors on the current CUDA device (or raw
integer addresses), streams are torch streams (default: the current one).

The library is built in-tree by :func:`build` (nvcc, sm_103a).  There is no
fallback: if the library is missing, :func:`lib` raises.
"""
from __future__ import annotations

import ctypes
import os

from ._build import LIB as _LIB_PATH
from ._build import build  # noqa: F401  (re-export)

ZERO_OK = 0
ZERO_EINVAL = -1
ZERO_EALIGN = -2
ZERO_EOVERLAP = -3
ZERO_ECUDA = -4
ZERO_ENOMEM = -5
ZERO_MAX_RANKS = 1024
ZERO_KERNEL_BULK = 1
ZERO_KERNEL_VECTOR = 2

MODE_STANDARD = 0
MODE_FOLDED_LITERAL = 1
MODE_FOLDED_STORAGE = 2
MODE_SGD = 3
MODE_MOMENTUM = 4

# every symbol include/zero_step.h declares
EXPORTED = ("zero_init_layout", "zero_free_layout", "zero_shard_range", "zero_memory_bytes",
            "zero_adam_step", "zero_adam_step_shard", "zero_plan_buckets", "zero_adam_step_range",
            "zero_adam_step_bucketed", "zero_set_step_max_sms", "zero_step_plan",
            "zero_reduce_scatter_fp16", "zero_cpu_adam",
            "zero_offload_step", "zero_mlp4_loss", "zero_mlp4_layer_grads",
            "zero_mlp4_zero3_step", "zero_mlp4_zero3_step_noalloc", "zero_device_timeouts",
            "zero_selftest_wait_timeout", "zero_selftest_mean_division", "zero_strerror",
            "zero_last_cuda_error", "zero_last_cuda_error_string")


class ZeroError(RuntimeError):
    def __init__(self, code: int, what: str):
        msg = f"{what}: {_strerror(code)} (status {code})"
        if code == ZERO_ECUDA:
            msg += f" [{lib().zero_last_cuda_error_string().decode()}]"
        super().__init__(msg)
        self.code = code


class zero_segment_t(ctypes.Structure):
    _fields_ = [("tensor_id", ctypes.c_int64), ("tensor_offset", ctypes.c_int64),
                ("shard_offset", ctypes.c_int64), ("len", ctypes.c_int64)]


class zero_bucket_t(ctypes.Structure):
    _fields_ = [("begin", ctypes.c_int64), ("end", ctypes.c_int64),
                ("first_tensor", ctypes.c_int32), ("last_tensor", ctypes.c_int32)]


class zero_layout_t(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int64), ("M", ctypes.c_int64), ("P", ctypes.c_int32),
                ("stage", ctypes.c_int32), ("n_tensors", ctypes.c_int32),
                ("reserved", ctypes.c_int32),
                ("shard_begin", ctypes.POINTER(ctypes.c_int64)),
                ("shard_end", ctypes.POINTER(ctypes.c_int64)),
                ("seg_offsets", ctypes.POINTER(ctypes.c_int64)),
                ("segs", ctypes.POINTER(zero_segment_t)),
                ("n_segs", ctypes.c_int64),
                ("bytes_per_rank_mixed", ctypes.c_double),
                ("floats_per_rank_p1", ctypes.c_double),
                ("comm_elems_per_rank", ctypes.c_double)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"{_LIB_PATH} is missing: build it with "
                           "zero_sharded_mixed_shard_gb300.build() (needs nvcc)")
    L = ctypes.CDLL(_LIB_PATH)
    i64, i32, f32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_void_p
    L.zero_init_layout.argtypes = [ctypes.POINTER(ctypes.c_int64), i32, i32, i32,
                                   ctypes.POINTER(zero_layout_t)]
    L.zero_init_layout.restype = ctypes.c_int
    L.zero_free_layout.argtypes = [ctypes.POINTER(zero_layout_t)]
    L.zero_free_layout.restype = None
    L.zero_shard_range.argtypes = [i64, i32, i32, ctypes.POINTER(ctypes.c_int64),
                                   ctypes.POINTER(ctypes.c_int64)]
    L.zero_shard_range.restype = ctypes.c_int
    L.zero_memory_bytes.argtypes = [i64, i32, i32, ctypes.POINTER(ctypes.c_double),
                                    ctypes.POINTER(ctypes.c_double),
                                    ctypes.POINTER(ctypes.c_double)]
    L.zero_memory_bytes.restype = ctypes.c_int
    L.zero_adam_step.argtypes = [vp, i64, vp, vp, vp, vp, i64, i32, i32, i64,
                                 f32, f32, f32, f32, i32, vp]
    L.zero_adam_step.restype = ctypes.c_int
    L.zero_adam_step_shard.argtypes = [vp, i64, i64, i32, vp, vp, vp, vp, i64, i32, i32, i64,
                                       f32, f32, f32, f32, i32, vp]
    L.zero_adam_step_shard.restype = ctypes.c_int
    L.zero_plan_buckets.argtypes = [ctypes.POINTER(ctypes.c_int64), i32, i64, i32,
                                    ctypes.POINTER(zero_bucket_t), i32, ctypes.POINTER(ctypes.c_int32)]
    L.zero_plan_buckets.restype = ctypes.c_int
    L.zero_adam_step_range.argtypes = [vp, i64, i64, i64, vp, vp, vp, vp, i64, i32, i32, i64,
                                       f32, f32, f32, f32, i32, vp]
    L.zero_adam_step_range.restype = ctypes.c_int
    L.zero_adam_step_bucketed.argtypes = [vp, i64, vp, vp, vp, vp, i64, i32, i32, i64,
                                          f32, f32, f32, f32, i32, ctypes.POINTER(zero_bucket_t),
                                          i32, ctypes.POINTER(ctypes.c_void_p), vp]
    L.zero_adam_step_bucketed.restype = ctypes.c_int
    L.zero_step_plan.argtypes = [vp, i64, vp, vp, vp, vp, i64, i32, i32, i32,
                                 ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32),
                                 ctypes.POINTER(ctypes.c_int64)]
    L.zero_step_plan.restype = ctypes.c_int
    L.zero_set_step_max_sms.argtypes = [i32, ctypes.POINTER(ctypes.c_int32)]
    L.zero_set_step_max_sms.restype = ctypes.c_int
    L.zero_reduce_scatter_fp16.argtypes = [vp, i64, i64, i32, i64, vp, vp]
    L.zero_reduce_scatter_fp16.restype = ctypes.c_int
    L.zero_cpu_adam.argtypes = [vp, vp, vp, vp, vp, i64, i64, f32, f32, f32, f32, i32, i32]
    L.zero_cpu_adam.restype = ctypes.c_int
    L.zero_offload_step.argtypes = [vp, i64, vp, vp, vp, vp, vp, vp, i64, i32, i32, i64,
                                    f32, f32, f32, f32, i32, i32, vp]
    L.zero_offload_step.restype = ctypes.c_int
    L.zero_mlp4_loss.argtypes = [vp, vp, i32, i32, vp, vp]
    L.zero_mlp4_loss.restype = ctypes.c_int
    L.zero_mlp4_layer_grads.argtypes = [i32, vp, vp, i32, i32, vp, i64, vp]
    L.zero_mlp4_layer_grads.restype = ctypes.c_int
    L.zero_mlp4_zero3_step.argtypes = [vp, i32, i32, vp, vp, vp, vp, vp, vp, i64, vp, i64,
                                       f32, f32, f32, f32, i32, i32, vp, vp]
    L.zero_mlp4_zero3_step.restype = ctypes.c_int
    L.zero_mlp4_zero3_step_noalloc.argtypes = [vp, i32, i32, vp, vp, vp, vp, vp, i64, f32, f32,
                                               f32, f32, i32, vp]
    L.zero_mlp4_zero3_step_noalloc.restype = ctypes.c_int
    L.zero_selftest_wait_timeout.argtypes = [vp, i64, vp, vp, vp, vp, i64, i32, i32, i64,
                                             f32, f32, f32, f32, i32, vp]
    L.zero_selftest_wait_timeout.restype = ctypes.c_int
    L.zero_selftest_mean_division.argtypes = [i32, i32, ctypes.POINTER(ctypes.c_int64),
                                              ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_float)]
    L.zero_selftest_mean_division.restype = ctypes.c_int
    L.zero_device_timeouts.argtypes = [ctypes.POINTER(ctypes.c_int64), i32]
    L.zero_device_timeouts.restype = ctypes.c_int
    L.zero_strerror.argtypes = [ctypes.c_int]
    L.zero_strerror.restype = ctypes.c_char_p
    L.zero_last_cuda_error.argtypes = []
    L.zero_last_cuda_error.restype = ctypes.c_int
    L.zero_last_cuda_error_string.argtypes = []
    L.zero_last_cuda_error_string.restype = ctypes.c_char_p
    _lib = L
    return L


def _strerror(code: int) -> str:
    return lib().zero_strerror(code).decode()


def zero_strerror(code: int) -> str:
    return _strerror(code)


def _addr(x) -> int | None:
    """Address of a torch tensor or numpy array (or pass an int / None through)."""
    if x is None or isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    return x.__array_interface__["data"][0]


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def zero_shard_range(N: int, P: int, k: int) -> tuple[int, int]:
    b, e = ctypes.c_int64(), ctypes.c_int64()
    rc = lib().zero_shard_range(N, P, k, ctypes.byref(b), ctypes.byref(e))
    if rc:
        raise ZeroError(rc, "zero_shard_range")
    return b.value, e.value


def zero_memory_bytes(N: int, P: int, stage: int) -> tuple[float, float, float]:
    """(model-state bytes per rank, float count per rank, elements moved per rank)."""
    b, f, c = ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
    rc = lib().zero_memory_bytes(N, P, stage, ctypes.byref(b), ctypes.byref(f), ctypes.byref(c))
    if rc:
        raise ZeroError(rc, "zero_memory_bytes")
    return b.value, f.value, c.value


def zero_init_layout(tensor_numel, P: int, stage: int) -> dict:
    """Layout table as plain Python data (the C table is freed before
    returning): N, M, P, stage, shard bounds, per-shard segments and the
    accounting figures."""
    n = len(tensor_numel)
    arr = (ctypes.c_int64 * max(n, 1))(*tensor_numel)
    t = zero_layout_t()
    rc = lib().zero_init_layout(arr, n, P, stage, ctypes.byref(t))
    if rc:
        raise ZeroError(rc, "zero_init_layout")
    try:
        segs = []
        for k in range(t.P):
            lo, hi = t.seg_offsets[k], t.seg_offsets[k + 1]
            segs.append([(t.segs[j].tensor_id, t.segs[j].tensor_offset,
                          t.segs[j].shard_offset, t.segs[j].len) for j in range(lo, hi)])
        return {
            "N": t.N, "M": t.M, "P": t.P, "stage": t.stage,
            "shards": [(t.shard_begin[k], t.shard_end[k]) for k in range(t.P)],
            "segments": segs,
            "n_segs": t.n_segs,
            "bytes_per_rank_mixed": t.bytes_per_rank_mixed,
            "floats_per_rank_p1": t.floats_per_rank_p1,
            "comm_elems_per_rank": t.comm_elems_per_rank,
        }
    finally:
        lib().zero_free_layout(ctypes.byref(t))


def zero_adam_step(grads, rank_stride: int, master, m, v, params, N: int, P: int, stage: int,
                   t: int, lr: float, beta1: float, beta2: float, eps: float, mode: int,
                   stream=None) -> None:
    """Enqueue one whole-vector ZeRO step (see include/zero_step.h)."""
    rc = lib().zero_adam_step(_addr(grads), rank_stride, _addr(master), _addr(m), _addr(v),
                              _addr(params), N, P, stage, t, lr, beta1, beta2, eps, mode,
                              _stream(stream))
    if rc:
        raise ZeroError(rc, "zero_adam_step")


def zero_adam_step_shard(grads, rank_stride: int, grad_offset: int, k: int, master_s, m_s,
                         v_s, params_out, N: int, P: int, stage: int, t: int, lr: float,
                         beta1: float, beta2: float, eps: float, mode: int,
                         stream=None) -> None:
    """Enqueue shard k's step (see include/zero_step.h)."""
    rc = lib().zero_adam_step_shard(_addr(grads), rank_stride, grad_offset, k, _addr(master_s),
                                    _addr(m_s), _addr(v_s), _addr(params_out), N, P, stage, t,
                                    lr, beta1, beta2, eps, mode, _stream(stream))
    if rc:
        raise ZeroError(rc, "zero_adam_step_shard")


def zero_set_step_max_sms(max_sms: int) -> int:
    """Cap the SMs a fused step occupies (0 = all); returns the previous cap."""
    prev = ctypes.c_int32()
    rc = lib().zero_set_step_max_sms(max_sms, ctypes.byref(prev))
    if rc:
        raise ZeroError(rc, "zero_set_step_max_sms")
    return prev.value


def zero_step_plan(grads, rank_stride: int, master, m, v, params, N: int, P: int, stage: int,
                   mode: int) -> dict:
    """The kernel zero_adam_step would launch: {"kernel": "bulk" | "vector",
    "vector_width": V, "ctas": C} (nothing is launched)."""
    k, vw, c = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int64()
    rc = lib().zero_step_plan(_addr(grads), rank_stride, _addr(master), _addr(m), _addr(v),
                              _addr(params), N, P, stage, mode, ctypes.byref(k), ctypes.byref(vw),
                              ctypes.byref(c))
    if rc:
        raise ZeroError(rc, "zero_step_plan")
    return {"kernel": "bulk" if k.value == ZERO_KERNEL_BULK else "vector",
            "vector_width": vw.value, "ctas": c.value}


def zero_selftest_mean_division(p_lo: int, p_hi: int) -> tuple:
    """(mismatches, first P, first sum) of the fast mean against the correctly
    rounded divide for rank counts p_lo..p_hi (see include/zero_step.h)."""
    n, fp, fs = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_float()
    rc = lib().zero_selftest_mean_division(p_lo, p_hi, ctypes.byref(n), ctypes.byref(fp), ctypes.byref(fs))
    if rc:
        raise ZeroError(rc, "zero_selftest_mean_division")
    return n.value, fp.value, fs.value


def zero_device_timeouts(reset: bool = False) -> int:
    """Bounded waits that gave up on the current device (0 in a correct run);
    synchronises with the device."""
    n = ctypes.c_int64()
    rc = lib().zero_device_timeouts(ctypes.byref(n), 1 if reset else 0)
    if rc:
        raise ZeroError(rc, "zero_device_timeouts")
    return n.value


def zero_selftest_wait_timeout(grads, rank_stride: int, master, m, v, params, N: int, P: int,
                               stage: int, t: int, lr: float, beta1: float, beta2: float,
                               eps: float, mode: int, stream=None) -> None:
    """Enqueue the bounded-wait diagnostic (see include/zero_step.h)."""
    rc = lib().zero_selftest_wait_timeout(_addr(grads), rank_stride, _addr(master), _addr(m),
                                          _addr(v), _addr(params), N, P, stage, t, lr, beta1,
                                          beta2, eps, mode, _stream(stream))
    if rc:
        raise ZeroError(rc, "zero_selftest_wait_timeout")


def zero_plan_buckets(tensor_numel, bucket_elems: int, backward_order: bool = True) -> list:
    """Buckets of consecutive tensors as (begin, end, first_tensor, last_tensor)."""
    n = len(tensor_numel)
    arr = (ctypes.c_int64 * max(n, 1))(*tensor_numel)
    count = ctypes.c_int32()
    rc = lib().zero_plan_buckets(arr, n, bucket_elems, 1 if backward_order else 0, None, 0,
                                 ctypes.byref(count))
    if rc:
        raise ZeroError(rc, "zero_plan_buckets")
    out = (zero_bucket_t * max(count.value, 1))()
    rc = lib().zero_plan_buckets(arr, n, bucket_elems, 1 if backward_order else 0, out,
                                 count.value, ctypes.byref(count))
    if rc:
        raise ZeroError(rc, "zero_plan_buckets")
    return [(b.begin, b.end, b.first_tensor, b.last_tensor) for b in out[:count.value]]


def zero_adam_step_range(grads, rank_stride: int, begin: int, end: int, master, m, v, params,
                         N: int, P: int, stage: int, t: int, lr: float, beta1: float,
                         beta2: float, eps: float, mode: int, stream=None) -> None:
    """Enqueue the step of flat elements [begin, end) (see include/zero_step.h)."""
    rc = lib().zero_adam_step_range(_addr(grads), rank_stride, begin, end, _addr(master),
                                    _addr(m), _addr(v), _addr(params), N, P, stage, t, lr,
                                    beta1, beta2, eps, mode, _stream(stream))
    if rc:
        raise ZeroError(rc, "zero_adam_step_range")


def zero_adam_step_bucketed(grads, rank_stride: int, master, m, v, params, N: int, P: int,
                            stage: int, t: int, lr: float, beta1: float, beta2: float,
                            eps: float, mode: int, buckets, ready_events=None,
                            stream=None) -> None:
    """Enqueue the step bucket by bucket; bucket b waits for ready_events[b]
    (torch.cuda.Event or None) on ``stream`` (see include/zero_step.h)."""
    nb = len(buckets)
    arr = (zero_bucket_t * max(nb, 1))()
    for i, b in enumerate(buckets):
        arr[i].begin, arr[i].end = int(b[0]), int(b[1])
        arr[i].first_tensor = int(b[2]) if len(b) > 2 else -1
        arr[i].last_tensor = int(b[3]) if len(b) > 3 else -1
    evs = None
    if ready_events is not None:
        evs = (ctypes.c_void_p * max(nb, 1))()
        for i, e in enumerate(ready_events):
            evs[i] = None if e is None else (e if isinstance(e, int) else e.cuda_event)
    rc = lib().zero_adam_step_bucketed(_addr(grads), rank_stride, _addr(master), _addr(m),
                                       _addr(v), _addr(params), N, P, stage, t, lr, beta1,
                                       beta2, eps, mode, arr, nb, evs, _stream(stream))
    if rc:
        raise ZeroError(rc, "zero_adam_step_bucketed")


def zero_reduce_scatter_fp16(grads, rank_stride: int, grad_offset: int, P: int, n: int, out,
                             stream=None) -> None:
    """Enqueue the fp16 gradient mean of n elements into ``out`` (device or
    page-locked host memory; see include/zero_step.h)."""
    rc = lib().zero_reduce_scatter_fp16(_addr(grads), rank_stride, grad_offset, P, n, _addr(out),
                                        _stream(stream))
    if rc:
        raise ZeroError(rc, "zero_reduce_scatter_fp16")


def zero_cpu_adam(grad16, master, m, v, params16, n: int, t: int, lr: float, beta1: float,
                  beta2: float, eps: float, mode: int, threads: int = 0) -> None:
    """ZeRO-Offload's host update on host buffers (numpy arrays, page-locked
    torch tensors or addresses); runs synchronously."""
    rc = lib().zero_cpu_adam(_addr(grad16), _addr(master), _addr(m), _addr(v), _addr(params16), n,
                             t, lr, beta1, beta2, eps, mode, threads)
    if rc:
        raise ZeroError(rc, "zero_cpu_adam")


def zero_offload_step(grads, rank_stride: int, master_host, m_host, v_host, grad16_host,
                      params16_host, params, N: int, P: int, stage: int, t: int, lr: float,
                      beta1: float, beta2: float, eps: float, mode: int, cpu_threads: int = 0,
                      stream=None) -> None:
    """Enqueue one ZeRO-Offload step (see include/zero_step.h)."""
    rc = lib().zero_offload_step(_addr(grads), rank_stride, _addr(master_host), _addr(m_host),
                                 _addr(v_host), _addr(grad16_host), _addr(params16_host),
                                 _addr(params), N, P, stage, t, lr, beta1, beta2, eps, mode,
                                 cpu_threads, _stream(stream))
    if rc:
        raise ZeroError(rc, "zero_offload_step")


def zero_mlp4_loss(params16, x, P: int, n: int, loss, stream=None) -> None:
    rc = lib().zero_mlp4_loss(_addr(params16), _addr(x), P, n, _addr(loss), _stream(stream))
    if rc:
        raise ZeroError(rc, "zero_mlp4_loss")


def zero_mlp4_layer_grads(layer: int, params16, x, P: int, n: int, grads16, rank_stride: int,
                          stream=None) -> None:
    rc = lib().zero_mlp4_layer_grads(layer, _addr(params16), _addr(x), P, n, _addr(grads16),
                                     rank_stride, _stream(stream))
    if rc:
        raise ZeroError(rc, "zero_mlp4_layer_grads")


def zero_mlp4_zero3_step(x, P: int, n: int, gathered16, master, m, v, shard16, grads16,
                         rank_stride: int, loss, t: int, lr: float, beta1: float, beta2: float,
                         eps: float, mode: int, pipelined: bool = True, main_stream=None,
                         step_stream=None) -> None:
    """Enqueue one layer-pipelined ZeRO-3 step of the 4-layer scalar MLP
    (see include/zero_step.h)."""
    rc = lib().zero_mlp4_zero3_step(_addr(x), P, n, _addr(gathered16), _addr(master), _addr(m),
                                    _addr(v), _addr(shard16), _addr(grads16), rank_stride,
                                    _addr(loss), t, lr, beta1, beta2, eps, mode,
                                    1 if pipelined else 0, _stream(main_stream),
                                    _stream(step_stream) if step_stream is not None else None)
    if rc:
        raise ZeroError(rc, "zero_mlp4_zero3_step")


def zero_mlp4_zero3_step_noalloc(x, P: int, n: int, master, m, v, shard16, loss, t: int,
                                 lr: float, beta1: float, beta2: float, eps: float, mode: int,
                                 stream=None) -> None:
    """The ZeRO-3 MLP step for callers that cannot allocate device memory:
    its scratch lives inside the library (at most 8 ranks; calls that
    overlap on the GPU race on it; see include/zero_step.h)."""
    rc = lib().zero_mlp4_zero3_step_noalloc(_addr(x), P, n, _addr(master), _addr(m), _addr(v),
                                            _addr(shard16), _addr(loss), t, lr, beta1, beta2, eps,
                                            mode, _stream(stream))
    if rc:
        raise ZeroError(rc, "zero_mlp4_zero3_step_noalloc")
