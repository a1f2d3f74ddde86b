"""The no-allocation variant of the ZeRO-3 MLP step.

Some callers cannot allocate device memory: a host program that reserved
all of the GPU's memory for its own allocator at start-up, or a service that
may not allocate while it runs, has no way to hand the library the scratch
buffers zero_mlp4_zero3_step needs between its kernels.  For them,
zero_mlp4_zero3_step_noalloc keeps that scratch in an array inside the
library.  Its results must be those of the oracle's training loop and of the
regular entry point, bit for bit, on every step: both run the same kernels
in the same order, so any difference -- a stale scratch entry left by an
earlier call, a wrong rank stride inside the array -- is a bug.

This file is collected last on purpose: the first call on a device looks the
array up, and the test must pass both alone in a fresh process and after
every other test."""
import numpy as np
import pytest

import oracle
from oracle import mlp4

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

LR, B1, B2, EPS = 1e-2, 0.9, 0.999, 1e-8


@pytest.fixture(scope="module")
def z(zlib, oracle_mod):
    if not torch.cuda.is_available():
        pytest.fail("the GPU tests need a CUDA device")
    return zlib


def _master0(rng):
    return np.array([rng.uniform(0.6, 1.2) if i % 2 == 0 else rng.uniform(0.0, 0.2)
                     for i in range(8)], np.float32)


def _state(master0, P, dev="cuda"):
    return [torch.from_numpy(master0.copy()).to(dev), torch.zeros(8, device=dev),
            torch.zeros(8, device=dev), torch.from_numpy(master0.astype(np.float16)).to(dev),
            torch.zeros(P, device=dev)]          # master, m, v, owners' fp16 shards, loss


def _oracle_steps(master0, xs, P, mode):
    """The oracle's training loop: each rank's fp16 local gradients, then the
    ZeRO step of the 8 parameters; the state after every step."""
    om, omm, ov = master0.copy(), np.zeros(8, np.float32), np.zeros(8, np.float32)
    op16 = master0.astype(np.float16).view(np.uint16).copy()
    out = []
    for t, x in enumerate(xs, start=1):
        codes, loss = mlp4.local_grads(op16, x)
        oracle.zero_step(codes.reshape(-1), 8, P, 8, om, omm, ov, op16, t, LR, B1, B2, EPS, mode)
        out.append((om.copy(), omm.copy(), ov.copy(), op16.copy(), loss.copy()))
    return out


def _bits(s):
    """Bit patterns of (master, m, v, fp16 shards, loss) on the host."""
    return (s[0].cpu().numpy().view(np.uint32), s[1].cpu().numpy().view(np.uint32),
            s[2].cpu().numpy().view(np.uint32), s[3].view(torch.int16).cpu().numpy().view(np.uint16),
            s[4].cpu().numpy().view(np.uint32))


def _ref_bits(r):
    return (r[0].view(np.uint32), r[1].view(np.uint32), r[2].view(np.uint32), r[3], r[4].view(np.uint32))


@pytest.mark.parametrize("P", [1, 3, 4, 8])
@pytest.mark.parametrize("mode", [0, 1, 2, 3, 4])
def test_no_alloc_step_matches_oracle_and_regular_step(z, P, mode):
    rng = np.random.default_rng(100 * P + mode)
    n, T = 24, 12
    master0 = _master0(rng)
    xs = [rng.uniform(0.1, 1.0, (P, n)).astype(np.float32) for _ in range(T)]
    ref = _oracle_steps(master0, xs, P, mode)
    a = _state(master0, P)     # the no-allocation entry point
    b = _state(master0, P)     # the regular one, with its scratch provided here
    gathered = torch.zeros(8, dtype=torch.float16, device="cuda")
    grads = torch.zeros((P, 8), dtype=torch.float16, device="cuda")
    x = torch.zeros((P, n), device="cuda")
    for t in range(1, T + 1):  # calls in a row: the array keeps the last call's contents
        x.copy_(torch.from_numpy(xs[t - 1]))
        z.zero_mlp4_zero3_step_noalloc(x, P, n, *a, t, LR, B1, B2, EPS, mode)
        z.zero_mlp4_zero3_step(x, P, n, gathered, b[0], b[1], b[2], b[3], grads, 8, b[4], t,
                               LR, B1, B2, EPS, mode, pipelined=True)
        torch.cuda.synchronize()
        got, reg, want = _bits(a), _bits(b), _ref_bits(ref[t - 1])
        for i, name in enumerate(("master", "m", "v", "shards", "loss")):
            assert np.array_equal(got[i], want[i]), f"P={P} mode={mode} t={t}: {name} vs oracle"
            assert np.array_equal(got[i], reg[i]), f"P={P} mode={mode} t={t}: {name} vs regular"
    assert z.zero_device_timeouts() == 0


def test_leftover_scratch_of_a_wider_call_is_never_read(z):
    """A call at P = 8 fills every rank's row of the array; the P = 3 calls
    that follow must read only what they wrote themselves."""
    rng = np.random.default_rng(7)
    n = 16
    wide = _state(_master0(rng), 8)
    xw = torch.from_numpy(rng.uniform(0.1, 1.0, (8, n)).astype(np.float32)).cuda()
    for t in (1, 2):
        z.zero_mlp4_zero3_step_noalloc(xw, 8, n, *wide, t, LR, B1, B2, EPS, 0)
    master0 = _master0(rng)
    xs = [rng.uniform(0.1, 1.0, (3, n)).astype(np.float32) for _ in range(4)]
    ref = _oracle_steps(master0, xs, 3, 0)
    s = _state(master0, 3)
    for t, x in enumerate(xs, start=1):
        z.zero_mlp4_zero3_step_noalloc(torch.from_numpy(x).cuda(), 3, n, *s, t, LR, B1, B2, EPS, 0)
        torch.cuda.synchronize()
        for g, w in zip(_bits(s), _ref_bits(ref[t - 1])):
            assert np.array_equal(g, w), t


def test_no_alloc_step_refuses_more_ranks_than_its_scratch_holds(z):
    x = torch.zeros((9, 4), device="cuda")
    s = _state(np.ones(8, np.float32), 9)
    with pytest.raises(z.ZeroError) as e:
        z.zero_mlp4_zero3_step_noalloc(x, 9, 4, *s, 1, LR, B1, B2, EPS, 0)
    assert e.value.code == z.ZERO_EINVAL


def test_rejected_no_alloc_call_writes_nothing(z):
    """A misaligned master is refused before anything is enqueued: the loss,
    the state and the shards keep their bytes."""
    x = torch.rand((4, 8), device="cuda")
    s = _state(np.ones(8, np.float32), 4)
    s[4].fill_(123.0)
    raw = torch.zeros(9, device="cuda")
    before = [t.clone() for t in s]
    with pytest.raises(z.ZeroError) as e:
        z.zero_mlp4_zero3_step_noalloc(x, 4, 8, raw.data_ptr() + 2, s[1], s[2], s[3], s[4], 1, LR,
                                       B1, B2, EPS, 0)
    assert e.value.code == z.ZERO_EALIGN
    torch.cuda.synchronize()
    for t, u in zip(s, before):
        assert torch.equal(t.view(torch.int16) if t.dtype == torch.float16 else t.view(torch.int32),
                           u.view(torch.int16) if u.dtype == torch.float16 else u.view(torch.int32))
