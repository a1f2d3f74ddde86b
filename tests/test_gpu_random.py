"""A seeded random sweep of the fused step through every entry point that
launches it (whole vector, one shard, a flat range), against the oracle bit
for bit: random N and P, rank strides padded or not, each buffer starting at
its own element offset (so the head length, the vector width and the kernel
vary), all five modes, and the SM cap on or off.  The cases that take the
bulk pipeline and the vector kernel are both counted, so the sweep is known
to cover both."""
import numpy as np
import pytest

import oracle
from _helpers import max_ulps
from zero_sharded_mixed_shard_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

LR, B1, B2, EPS = 1e-3, 0.9, 0.999, 1e-8
CASES = 160


@pytest.fixture(scope="module")
def z(zlib, oracle_mod):
    if not torch.cuda.is_available():
        pytest.fail("the GPU tests need a CUDA device")
    return zlib


def _dev_at(arr: np.ndarray, off: int, dtype):
    """A device copy of `arr` starting `off` elements into a fresh buffer."""
    buf = torch.zeros(arr.size + off + 8, dtype=dtype, device="cuda")
    view = buf[off:off + arr.size]
    view.copy_(torch.from_numpy(arr.view(np.int16) if dtype == torch.int16 else arr))
    return view


def _case(rng, sms):
    big = rng.random() < 0.3
    P = int(rng.choice([1, 2, 3, 4, 5, 8, 12, 16, 33])) if big else int(rng.integers(1, 41))
    N = int(sms * 2048 * 4 + rng.integers(0, 50_000)) if big else int(rng.integers(1, 120_000))
    aligned = rng.random() < 0.6       # every buffer on one 16-byte phase
    stride = synth.round_up(N, 8) + 8 * int(rng.integers(0, 3)) if aligned else N + int(rng.integers(0, 9))
    offs = [0] * 5 if aligned else [int(x) for x in rng.integers(0, 8, size=5)]
    return dict(P=P, N=N, stride=stride, offs=offs, mode=int(rng.integers(0, 5)),
                api=str(rng.choice(["whole", "shard", "range"])), cap=int(rng.choice([0, 0, 7, 40])),
                seed=int(rng.integers(0, 2**31)))


def test_random_sweep(z):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rng = np.random.default_rng(20261202)
    kernels = {"bulk": 0, "vector": 0}
    for i in range(CASES):
        c = _case(rng, sms)
        P, N, stride, mode = c["P"], c["N"], c["stride"], c["mode"]
        codes = synth.np_grads(P, N, stride, 1e-3, c["seed"], heavy_tail_frac=0.01, zero_frac=0.02)
        w0, m0, v0, p0 = synth.np_state(N, c["seed"])
        m0 = (np.random.default_rng(c["seed"]).standard_normal(N) * 1e-4).astype(np.float32)
        v0 = np.abs(m0) * np.float32(1e-3)
        og, ow, om, ov, op = c["offs"]
        g = _dev_at(codes, og, torch.int16).view(torch.float16)
        s = [_dev_at(w0, ow, torch.float32), _dev_at(m0, om, torch.float32),
             _dev_at(v0, ov, torch.float32), _dev_at(p0, op, torch.int16).view(torch.float16)]
        # the range of the vector this call updates
        if c["api"] == "whole":
            b, e = 0, N
        elif c["api"] == "shard":
            M = -(-N // P)
            k = int(rng.integers(0, P))
            b, e = min(k * M, N), min((k + 1) * M, N)
        else:
            b = int(rng.integers(0, N))
            e = int(rng.integers(b + 1, N + 1))
        prev = z.zero_set_step_max_sms(c["cap"])
        try:
            if e > b:
                plan = z.zero_step_plan(g[b:], stride, *[x[b:] for x in s], e - b, P, 2, mode)
                kernels[plan["kernel"]] += 1
            t = 1 + i % 3
            if c["api"] == "whole":
                z.zero_adam_step(g, stride, *s, N, P, 2, t, LR, B1, B2, EPS, mode)
            elif c["api"] == "shard":
                z.zero_adam_step_shard(g, stride, b, k, *[x[b:e] for x in s], N, P, 3, t,
                                       LR, B1, B2, EPS, mode)
            else:
                z.zero_adam_step_range(g, stride, b, e, *s, N, P, 2, t, LR, B1, B2, EPS, mode)
        finally:
            z.zero_set_step_max_sms(prev)
        ref = [w0.copy(), m0.copy(), v0.copy()]
        ref_p = p0.copy()
        if e > b:
            win = codes.reshape(P, stride)[:, b:e].copy().reshape(-1)
            sub = [r[b:e].copy() for r in ref]
            ref_p[b:e] = oracle.adam_elems(win, e - b, P, *sub, t, LR, B1, B2, EPS, mode, threads=8)
            for r, x in zip(ref, sub):
                r[b:e] = x
        got = [s[0].cpu().numpy(), s[1].cpu().numpy(), s[2].cpu().numpy(),
               s[3].view(torch.int16).cpu().numpy().view(np.uint16)]
        # elements outside [b, e) are untouched, inside equal the oracle
        assert max_ulps(got, ref + [ref_p]) == (0, 0), c
    assert kernels["bulk"] >= 10 and kernels["vector"] >= 30, kernels
    assert z.zero_device_timeouts() == 0
