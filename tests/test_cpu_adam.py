"""ZeRO-Offload's host update (the library's C++ CPU Adam, no GPU needed)
against the oracle's offload step: given the fp16 gradient that crossed to the
host (the oracle's own output), the update must equal the oracle's bit for
bit, in every reading, with any thread split, on special values too."""
import numpy as np
import pytest

from zero_sharded_mixed_shard_gb300 import synth

LR, B1, B2, EPS = 1e-3, 0.9, 0.999, 1e-8


def _same32(a, b):
    nan = np.isnan(b)
    return np.array_equal(np.isnan(a), nan) and np.array_equal(a[~nan].view(np.uint32),
                                                               b[~nan].view(np.uint32))


def _same16(a, b):
    nan = ((b & 0x7C00) == 0x7C00) & ((b & 0x3FF) != 0)
    nan_a = ((a & 0x7C00) == 0x7C00) & ((a & 0x3FF) != 0)
    return np.array_equal(nan, nan_a) and np.array_equal(a[~nan], b[~nan])


def _check(zlib, oracle_mod, codes, stride, P, w, m, v, t, mode, threads):
    n = w.size
    ref = [w.copy(), m.copy(), v.copy()]
    p_ref, g16 = oracle_mod.offload_elems(codes, stride, P, *ref, t, LR, B1, B2, EPS, mode)
    p = np.empty(n, np.uint16)
    zlib.zero_cpu_adam(g16, w, m, v, p, n, t, LR, B1, B2, EPS, mode, threads)
    for got, exp in zip((w, m, v), ref):
        assert _same32(got, exp), (mode, threads, t)
    assert _same16(p, p_ref), (mode, threads, t)


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("threads", [1, 3, 0])
def test_cpu_adam_matches_oracle(zlib, oracle_mod, mode, threads):
    n, P = 300_001, 4
    w, m, v, _ = synth.np_state(n, 9)
    for t in (1, 2, 3):
        codes = synth.np_grads(P, n, n, 1e-3, 10 * mode + threads + t, heavy_tail_frac=0.01)
        _check(zlib, oracle_mod, codes, n, P, w, m, v, t, mode, threads)


def test_cpu_adam_special_values(zlib, oracle_mod):
    n, P = 70_000, 2
    rng = np.random.default_rng(3)
    specials16 = np.array([0x0000, 0x8000, 0x0001, 0x8001, 0x7BFF, 0xFBFF, 0x7C00, 0xFC00,
                           0x3C00], np.uint16)
    codes = (rng.standard_normal(P * n) * 1e-3).astype(np.float16).view(np.uint16)
    pick = rng.random(P * n) < 0.2
    codes[pick] = rng.choice(specials16, int(pick.sum()))
    # a tiny negative mean that rounds to -0 on the fp16 edge: (-2^-24 + 0) / 2
    codes[:8] = 0x8001
    codes[n:n + 8] = 0x0000
    sp = np.array([np.inf, -np.inf, 0.0, -0.0, 3e38, 1e-45, 1e-38], np.float32)

    def sprinkle(x):
        k = rng.random(n) < 0.2
        x[k] = rng.choice(sp, int(k.sum()))
        return x

    w = sprinkle(rng.standard_normal(n).astype(np.float32))
    m = sprinkle((rng.standard_normal(n) * 1e-3).astype(np.float32))
    v = np.abs(sprinkle((rng.random(n) * 1e-6).astype(np.float32)))
    for mode in (0, 1, 2):
        _check(zlib, oracle_mod, codes, n, P, w.copy(), m.copy(), v.copy(), 4, mode, 4)
    # the -0 gradient did cross
    _, g16 = oracle_mod.offload_elems(codes[:], n, P, w.copy(), m.copy(), v.copy(), 4, LR, B1,
                                      B2, EPS, 0)
    assert np.all(g16[:8] == 0x8000)


def test_cpu_adam_rejects(zlib):
    a = np.zeros(4, np.float32)
    h = np.zeros(4, np.uint16)
    for kw in (dict(t=0), dict(mode=3), dict(threads=-1), dict(beta1=1.0), dict(lr=float("nan"))):
        args = dict(t=1, mode=0, threads=1, beta1=B1, lr=LR)
        args.update(kw)
        with pytest.raises(zlib.ZeroError):
            zlib.zero_cpu_adam(h, a, a.copy(), a.copy(), h.copy(), 4, args["t"], args["lr"],
                               args["beta1"], B2, EPS, args["mode"], args["threads"])
    with pytest.raises(zlib.ZeroError):
        zlib.zero_cpu_adam(None, a, a, a, h, 4, 1, LR, B1, B2, EPS, 0, 1)
    zlib.zero_cpu_adam(None, None, None, None, None, 0, 1, LR, B1, B2, EPS, 0, 1)  # n = 0


def test_cpu_adam_concurrent_callers_share_the_pool(zlib, oracle_mod):
    """The host threads are a pool kept between calls; calls from several
    threads at once queue on it and each still matches the oracle bit for
    bit (ctypes releases the GIL for the duration of each call)."""
    import threading

    n, P = 200_003, 4
    cases = []
    for k in range(6):
        w, m, v, _ = synth.np_state(n, 50 + k)
        codes = synth.np_grads(P, n, n, 1e-3, 60 + k)
        ref = [w.copy(), m.copy(), v.copy()]
        p_ref, g16 = oracle_mod.offload_elems(codes, n, P, *ref, 2, LR, B1, B2, EPS, k % 3)
        cases.append((w, m, v, np.empty(n, np.uint16), g16, ref, p_ref, k % 3, (0, 1, 2, 5)[k % 4]))
    errors = []

    def run(case):
        w, m, v, p, g16, _, _, mode, threads = case
        try:
            for _ in range(3):   # same inputs each time: the last call's bytes are checked
                w2, m2, v2 = w.copy(), m.copy(), v.copy()
                zlib.zero_cpu_adam(g16, w2, m2, v2, p, n, 2, LR, B1, B2, EPS, mode, threads)
            w[:], m[:], v[:] = w2, m2, v2
        except Exception as e:   # pragma: no cover - reported below
            errors.append(e)

    ths = [threading.Thread(target=run, args=(c,)) for c in cases]
    for th in ths:
        th.start()
    for th in ths:
        th.join()
    assert not errors
    for w, m, v, p, _, ref, p_ref, mode, threads in cases:
        for got, exp in zip((w, m, v), ref):
            assert _same32(got, exp), (mode, threads)
        assert _same16(p, p_ref), (mode, threads)


def test_cpu_adam_more_threads_than_cpus(zlib, oracle_mod):
    """A thread count above the CPUs available is capped, not an error."""
    n, P = 100_000, 2
    w, m, v, _ = synth.np_state(n, 77)
    codes = synth.np_grads(P, n, n, 1e-3, 78)
    _check(zlib, oracle_mod, codes, n, P, w, m, v, 1, 0, 1024)
