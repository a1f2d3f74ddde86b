"""The C ABI without a GPU: the library loads, exports every function its
header declares, and rejects bad arguments on the host before any CUDA call.

The rejection cases pass made-up device addresses; they run only where no
GPU is visible, so a case that wrongly passed validation could never reach a
kernel.  The same checks with real device buffers are in the GPU tests."""
import ctypes
import math
import os
import re

import pytest

from conftest import cuda_available

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
           if f.endswith(".h")]


def declared_functions():
    names = set()
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names.update(re.findall(r"^\s*(?:const\s+)?\w+\s*\**\s*(zero_\w+)\s*\(", text, flags=re.M))
    return names


def test_header_declares_the_step_api():
    names = declared_functions()
    assert {"zero_init_layout", "zero_free_layout", "zero_memory_bytes", "zero_adam_step",
            "zero_adam_step_shard", "zero_strerror"} <= names


def test_library_exports_every_declared_symbol(zlib):
    L = zlib.lib()
    for name in declared_functions():
        assert hasattr(L, name), name
    assert set(zlib.EXPORTED) == declared_functions()


def test_status_codes_match_header(zlib):
    text = "".join(open(h).read() for h in HEADERS)
    for name in ("ZERO_OK", "ZERO_EINVAL", "ZERO_EALIGN", "ZERO_EOVERLAP", "ZERO_ECUDA",
                 "ZERO_ENOMEM", "ZERO_MAX_RANKS", "ZERO_KERNEL_BULK", "ZERO_KERNEL_VECTOR"):
        m = re.search(r"#define\s+%s\s+\(?(-?\d+)\)?" % name, text)
        assert m and int(m.group(1)) == getattr(zlib, name), name
    for code in (0, -1, -2, -3, -4, -5):
        assert zlib.zero_strerror(code)
    assert "unknown" in zlib.zero_strerror(-99)


no_gpu = pytest.mark.skipif(cuda_available(), reason="made-up device addresses: CPU-only check")

A = 1 << 40                    # made-up, 256-byte aligned addresses, far apart
G, W, MM, V, PP = A, 2 * A, 3 * A, 4 * A, 5 * A
GOOD = dict(grads=G, rank_stride=1000, master=W, m=MM, v=V, params=PP, N=1000, P=4, stage=2,
            t=1, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, mode=0)


def _call(zlib, **kw):
    a = dict(GOOD, **kw)
    return zlib.lib().zero_adam_step(a["grads"], a["rank_stride"], a["master"], a["m"], a["v"],
                                     a["params"], a["N"], a["P"], a["stage"], a["t"], a["lr"],
                                     a["beta1"], a["beta2"], a["eps"], a["mode"], 0)


@no_gpu
@pytest.mark.parametrize("kw,code", [
    (dict(grads=None), -1), (dict(master=None), -1), (dict(m=None), -1), (dict(v=None), -1),
    (dict(params=None), -1), (dict(N=0), -1), (dict(N=-5), -1), (dict(P=0), -1),
    (dict(P=1025), -1), (dict(stage=4), -1), (dict(stage=-1), -1), (dict(mode=7), -1),
    (dict(mode=-1), -1), (dict(mode=5), -1), (dict(t=0), -1), (dict(lr=math.nan), -1), (dict(lr=math.inf), -1),
    (dict(beta1=1.0), -1), (dict(beta2=-0.5), -1), (dict(eps=-1e-8), -1),
    (dict(eps=math.inf), -1), (dict(rank_stride=999), -1),
    (dict(master=W + 2), -2), (dict(v=V + 1), -2), (dict(params=PP + 1), -2),
    (dict(grads=G + 1), -2),
    (dict(m=W + 3996), -3), (dict(v=MM), -3), (dict(params=W + 100), -3),
    (dict(master=G + 2 * 3000), -3), (dict(params=G + 2 * 3999), -3),
])
def test_step_rejects(zlib, kw, code):
    assert _call(zlib, **kw) == code
    # the diagnostic entry point validates exactly like the step
    a = dict(GOOD, **kw)
    assert zlib.lib().zero_selftest_wait_timeout(
        a["grads"], a["rank_stride"], a["master"], a["m"], a["v"], a["params"], a["N"], a["P"],
        a["stage"], a["t"], a["lr"], a["beta1"], a["beta2"], a["eps"], a["mode"], 0) == code


@no_gpu
def test_shard_rejects_and_empty_shard(zlib):
    L = zlib.lib()

    def shard(k=0, off=0, N=1000, P=4, stride=250, w=W, m=MM, v=V, p=PP, g=G):
        return L.zero_adam_step_shard(g, stride, off, k, w, m, v, p, N, P, 2, 1, 1e-3, 0.9,
                                      0.999, 1e-8, 0, 0)

    assert shard(k=4) == -1
    assert shard(k=-1) == -1
    assert shard(off=-1) == -1
    assert shard(stride=249) == -1          # rank slices would overlap
    assert shard(g=None) == -1
    assert shard(w=W + 1) == -2
    assert shard(p=W) == -3
    # N = 5, P = 4: shard 3 owns nothing, returns success without any CUDA call,
    # even with no buffers at all; its scalars are still checked
    assert shard(k=3, N=5, stride=2) == 0
    assert shard(k=3, N=5, stride=2, g=None, w=None, m=None, v=None, p=None) == 0
    assert L.zero_adam_step_shard(None, 2, 0, 3, None, None, None, None, 5, 4, 2, 0, 1e-3, 0.9,
                                  0.999, 1e-8, 0, 0) == -1   # t = 0


@no_gpu
def test_range_and_bucketed_reject(zlib):
    L = zlib.lib()

    def rng_(b, e, N=1000):
        return L.zero_adam_step_range(G, 1000, b, e, W, MM, V, PP, N, 4, 2, 1, 1e-3, 0.9, 0.999,
                                      1e-8, 0, 0)

    for b, e in [(-1, 10), (10, 10), (20, 10), (0, 1001)]:
        assert rng_(b, e) == zlib.ZERO_EINVAL
    assert rng_(0, 10, N=0) == zlib.ZERO_EINVAL

    def bucketed(pairs, n=None):
        arr = (zlib.zero_bucket_t * max(len(pairs), 1))()
        for i, (b, e) in enumerate(pairs):
            arr[i].begin, arr[i].end = b, e
        return L.zero_adam_step_bucketed(G, 1000, W, MM, V, PP, 1000, 4, 2, 1, 1e-3, 0.9, 0.999,
                                         1e-8, 0, arr, len(pairs) if n is None else n, None, 0)

    assert bucketed([(0, 500), (400, 1000)]) == zlib.ZERO_EINVAL     # overlap
    assert bucketed([(500, 1000), (0, 501)]) == zlib.ZERO_EINVAL     # overlap, unsorted
    assert bucketed([(0, 500), (500, 1001)]) == zlib.ZERO_EINVAL     # past N
    assert bucketed([(5, 5)]) == zlib.ZERO_EINVAL                    # empty
    assert bucketed([(0, 10)], n=0) == zlib.ZERO_EINVAL
    # valid buckets on a misaligned master pointer are refused before any launch
    arr = (zlib.zero_bucket_t * 1)()
    arr[0].begin, arr[0].end = 0, 1000
    assert L.zero_adam_step_bucketed(G, 1000, W + 2, MM, V, PP, 1000, 4, 2, 1, 1e-3, 0.9, 0.999,
                                     1e-8, 0, arr, 1, None, 0) == zlib.ZERO_EALIGN


@no_gpu
def test_unused_state_may_be_null_but_used_state_may_not(zlib):
    # SGD (mode 3) uses neither m nor v; momentum (mode 4) uses m; Adam both.
    # Only the rejected calls are made here: nothing reaches a kernel.
    assert _call(zlib, mode=4, m=None) == zlib.ZERO_EINVAL
    assert _call(zlib, mode=0, v=None) == zlib.ZERO_EINVAL
    assert _call(zlib, mode=3, master=None) == zlib.ZERO_EINVAL
    # an unused buffer is not checked for alignment or overlap either: the
    # first failing check is then on a used one
    assert _call(zlib, mode=3, m=W + 1, v=W, params=PP + 1) == zlib.ZERO_EALIGN
    assert _call(zlib, mode=4, v=MM + 1, m=W + 8) == zlib.ZERO_EOVERLAP


def test_step_max_sms_setting(zlib):
    """Host-only: the cap is stored, returned as the previous value, and a
    negative cap is refused without changing it."""
    prev = zlib.zero_set_step_max_sms(12)
    try:
        assert zlib.zero_set_step_max_sms(0) == 12
        with pytest.raises(zlib.ZeroError) as e:
            zlib.zero_set_step_max_sms(-1)
        assert e.value.code == zlib.ZERO_EINVAL
        assert zlib.zero_set_step_max_sms(0) == 0
    finally:
        zlib.zero_set_step_max_sms(prev)


def test_mean_division_check_rejects_bad_ranges(zlib):
    """Host-side argument checks of the mean-division diagnostic (no CUDA call)."""
    for lo, hi in ((0, 5), (5, 4), (1, zlib.ZERO_MAX_RANKS + 1)):
        with pytest.raises(zlib.ZeroError) as e:
            zlib.zero_selftest_mean_division(lo, hi)
        assert e.value.code == zlib.ZERO_EINVAL


# the 4-layer MLP steps: made-up buffers, 4 KiB apart unless a case moves one
X_, GATH, MST, MOM, VAR, SHD, GRD, LOSS = (A + (i << 12) for i in range(8))
MLP_GOOD = dict(x=X_, P=4, n=16, gathered=GATH, master=MST, m=MOM, v=VAR, shard=SHD, grads=GRD,
                rank_stride=8, loss=LOSS, t=1, lr=1e-2, beta1=0.9, beta2=0.999, eps=1e-8, mode=0)


def _mlp_regular(zlib, **kw):
    a = dict(MLP_GOOD, **kw)
    return zlib.lib().zero_mlp4_zero3_step(a["x"], a["P"], a["n"], a["gathered"], a["master"],
                                           a["m"], a["v"], a["shard"], a["grads"],
                                           a["rank_stride"], a["loss"], a["t"], a["lr"],
                                           a["beta1"], a["beta2"], a["eps"], a["mode"], 0, 0, 0)


def _mlp_noalloc(zlib, **kw):
    a = dict(MLP_GOOD, **kw)
    return zlib.lib().zero_mlp4_zero3_step_noalloc(a["x"], a["P"], a["n"], a["master"], a["m"],
                                                   a["v"], a["shard"], a["loss"], a["t"],
                                                   a["lr"], a["beta1"], a["beta2"], a["eps"],
                                                   a["mode"], 0)


MLP_BAD_BOTH = [
    (dict(P=0), -1), (dict(P=9), -1), (dict(n=0), -1), (dict(t=0), -1), (dict(mode=5), -1),
    (dict(lr=math.nan), -1), (dict(beta1=1.0), -1), (dict(eps=-1.0), -1),
    (dict(x=None), -1), (dict(master=None), -1), (dict(m=None), -1), (dict(loss=None), -1),
    (dict(master=MST + 2), -2), (dict(m=MOM + 1), -2), (dict(v=VAR + 2), -2),
    (dict(loss=LOSS + 2), -2), (dict(x=X_ + 2), -2), (dict(shard=SHD + 1), -2),
    # whole 8-element buffers that overlap, though no one shard's pieces would
    (dict(m=MST + 8), -3), (dict(v=MOM + 28), -3), (dict(shard=VAR + 16), -3),
    (dict(loss=MST + 28), -3), (dict(master=X_ + 4 * 63), -3),
]


@no_gpu
@pytest.mark.parametrize("kw,code", MLP_BAD_BOTH + [
    (dict(gathered=None), -1), (dict(grads=None), -1), (dict(rank_stride=7), -1),
    (dict(gathered=GATH + 1), -2), (dict(grads=GRD + 1), -2),
    (dict(gathered=SHD + 14), -3), (dict(grads=LOSS - 2 * 3 * 8 - 14), -3),
    (dict(rank_stride=2048, loss=GRD + 2 * 2048 + 4), -3),
])
def test_mlp4_step_rejects_before_enqueueing(zlib, kw, code):
    """Every argument check of the MLP step comes before its first CUDA call:
    with made-up device addresses and no GPU, a rejected call returns its
    status instead of a CUDA error from a copy or a launch."""
    assert _mlp_regular(zlib, **kw) == code


@no_gpu
@pytest.mark.parametrize("kw,code", MLP_BAD_BOTH)
def test_mlp4_noalloc_step_rejects_before_enqueueing(zlib, kw, code):
    assert _mlp_noalloc(zlib, **kw) == code


@no_gpu
@pytest.mark.parametrize("kw,code", [
    (dict(mode=3), -1), (dict(cpu_threads=-1), -1), (dict(rank_stride=999), -1), (dict(g16=None), -1),
    (dict(master=W + 2), -2), (dict(g16=7 * A + 1), -2), (dict(grads=G + 1), -2), (dict(params=PP + 1), -2),
    (dict(g16=G + 2 * 2000), -3),
])
def test_offload_step_rejects_before_enqueueing(zlib, kw, code):
    """The offload step checks every buffer before its first CUDA call."""
    a = dict(grads=G, rank_stride=1000, master=W, m=MM, v=V, g16=7 * A, p16=8 * A, params=PP, N=1000,
             P=4, mode=0, cpu_threads=0)
    a.update(kw)
    assert zlib.lib().zero_offload_step(a["grads"], a["rank_stride"], a["master"], a["m"], a["v"], a["g16"],
                                        a["p16"], a["params"], a["N"], a["P"], 2, 1, 1e-3, 0.9, 0.999, 1e-8,
                                        a["mode"], a["cpu_threads"], 0) == code
