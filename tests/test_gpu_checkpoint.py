"""Checkpoint and resume of the optimizer state.

A run is stopped after step j: the fp32 master / m / v shards and the
number of the last step t = j are written to a file (the fp16 parameters
are not: they are the rounding of master, and the next step rewrites every
one of them).  Fresh device buffers are filled from the file and the run goes
on with steps j+1..T.  The resumed run must equal both the uninterrupted run
and the oracle bit for bit, in every Adam reading and on both kernels.  The
folded readings divide by 1 - beta^t, so a resume that lost or shifted t
would show here (深度学习专题：模型训练的数据并行（三） §（一）Adam 优化器:
the bias correction is folded into the stored m and v).
"""
import numpy as np
import pytest

import oracle
from zero_sharded_mixed_shard_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

LR, B1, B2, EPS = 1e-3, 0.9, 0.999, 1e-8


@pytest.fixture(scope="module")
def z(zlib, oracle_mod):
    if not torch.cuda.is_available():
        pytest.fail("the GPU tests need a CUDA device")
    return zlib


def _u16(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _grads(P, N, stride, t):
    return synth.np_grads(P, N, stride, 1e-3, 5000 + t, heavy_tail_frac=0.01, zero_frac=0.05)


def _dev(codes):
    return torch.from_numpy(codes.view(np.int16)).cuda().view(torch.float16)


def _save(path, state, t):
    np.savez(path, master=state[0].cpu().numpy(), m=state[1].cpu().numpy(),
             v=state[2].cpu().numpy(), t=np.int64(t))


def _load(path, N):
    f = np.load(path)
    params = torch.full((N,), synth.SENTINEL_HALF, dtype=torch.int16, device="cuda").view(torch.float16)
    return [torch.from_numpy(f["master"]).cuda(), torch.from_numpy(f["m"]).cuda(),
            torch.from_numpy(f["v"]).cuda(), params], int(f["t"])


# (N, P, kernel): 1.5 M elements at P = 8 is more than 4 tiles per SM (the
# bulk-copy pipeline); 100,003 at P = 3 takes the vector kernel
CASES = [(1_500_000, 8, "bulk"), (100_003, 3, "vector")]


@pytest.mark.parametrize("N,P,kernel", CASES)
@pytest.mark.parametrize("mode", [0, 1, 2])
def test_resume_from_checkpoint_equals_uninterrupted_run(z, tmp_path, N, P, kernel, mode):
    T, j = 6, 3
    stride = synth.round_up(N, 8)
    w0, m0, v0, p0 = synth.np_state(N, 77 + P)
    codes = [_grads(P, N, stride, t) for t in range(1, T + 1)]

    # the oracle, uninterrupted
    ref = [w0.copy(), m0.copy(), v0.copy()]
    ref_p = None
    for t in range(1, T + 1):
        ref_p = oracle.adam_elems(codes[t - 1], stride, P, *ref, t, LR, B1, B2, EPS, mode, threads=8)

    def fresh():
        return [torch.from_numpy(w0.copy()).cuda(), torch.from_numpy(m0.copy()).cuda(),
                torch.from_numpy(v0.copy()).cuda(),
                torch.from_numpy(p0.view(np.int16).copy()).cuda().view(torch.float16)]

    # the device, uninterrupted
    a = fresh()
    plan = z.zero_step_plan(_dev(codes[0]), stride, *a, N, P, 2, mode)
    assert plan["kernel"] == kernel, plan
    for t in range(1, T + 1):
        z.zero_adam_step(_dev(codes[t - 1]), stride, *a, N, P, 2, t, LR, B1, B2, EPS, mode)

    # the device, stopped after step j, saved, reloaded into new buffers, resumed
    b = fresh()
    for t in range(1, j + 1):
        z.zero_adam_step(_dev(codes[t - 1]), stride, *b, N, P, 2, t, LR, B1, B2, EPS, mode)
    path = tmp_path / "zero_state.npz"
    _save(path, b, j)
    del b
    torch.cuda.empty_cache()
    c, t_last = _load(path, N)
    assert t_last == j
    for t in range(t_last + 1, T + 1):
        z.zero_adam_step(_dev(codes[t - 1]), stride, *c, N, P, 2, t, LR, B1, B2, EPS, mode)
    torch.cuda.synchronize()

    for name, x, y, r in zip(("master", "m", "v"), c[:3], a[:3], ref):
        xb = x.cpu().numpy().view(np.uint32)
        assert np.array_equal(xb, y.cpu().numpy().view(np.uint32)), f"{name}: resumed vs uninterrupted"
        assert np.array_equal(xb, r.view(np.uint32)), f"{name}: resumed vs oracle"
    assert np.array_equal(_u16(c[3]), _u16(a[3])) and np.array_equal(_u16(c[3]), ref_p)


def test_resume_with_a_wrong_step_count_differs(z, tmp_path):
    """The check above has teeth: resuming the folded reading with t off by
    one gives other bytes."""
    N, P, mode = 100_003, 3, 2
    stride = synth.round_up(N, 8)
    w0, m0, v0, p0 = synth.np_state(N, 91)
    s = [torch.from_numpy(x.copy()).cuda() for x in (w0, m0, v0)] + [
        torch.from_numpy(p0.view(np.int16).copy()).cuda().view(torch.float16)]
    for t in (1, 2):
        z.zero_adam_step(_dev(_grads(P, N, stride, t)), stride, *s, N, P, 2, t, LR, B1, B2, EPS, mode)
    _save(tmp_path / "s.npz", s, 2)
    good, t_last = _load(tmp_path / "s.npz", N)
    bad, _ = _load(tmp_path / "s.npz", N)
    g3 = _dev(_grads(P, N, stride, 3))
    z.zero_adam_step(g3, stride, *good, N, P, 2, t_last + 1, LR, B1, B2, EPS, mode)
    z.zero_adam_step(g3, stride, *bad, N, P, 2, t_last, LR, B1, B2, EPS, mode)
    assert not torch.equal(good[1], bad[1])
