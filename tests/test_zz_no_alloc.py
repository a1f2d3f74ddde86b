"""The no-allocation variant of the ZeRO-3 MLP step.

Some callers cannot allocate device memory: a host program that reserved
all of the GPU's memory for its own allocator at start-up, or a service that
may not allocate while it runs, has no way to hand the library the scratch
buffers zero_mlp4_zero3_step needs between its kernels.  For them,
zero_mlp4_zero3_step_noalloc keeps that scratch in an array inside the
library.  Here two calls in a row must give what the regular entry point
gives on the same inputs, within the tolerance the other tests use (2 fp32
ulp on master / m / v and the loss, 1 fp16 ulp on the parameters).

This file is collected last on purpose: the first call on a device looks the
array up, and the test must pass both alone in a fresh process and after
every other test."""
import numpy as np
import pytest

from _helpers import ulp16, ulp32

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

LR, B1, B2, EPS = 1e-2, 0.9, 0.999, 1e-8


@pytest.fixture(scope="module")
def z(zlib):
    if not torch.cuda.is_available():
        pytest.fail("the GPU tests need a CUDA device")
    return zlib


def _state(master0, dev="cuda"):
    return [torch.from_numpy(master0.copy()).to(dev), torch.zeros(8, device=dev),
            torch.zeros(8, device=dev), torch.from_numpy(master0.astype(np.float16)).to(dev),
            torch.zeros(8, device=dev)]          # master, m, v, owners' fp16 shards, loss (>= P)


@pytest.mark.parametrize("P,mode", [(4, 0), (8, 2), (3, 4)])
def test_no_alloc_step_matches_the_regular_step(z, P, mode):
    rng = np.random.default_rng(P + 10 * mode)
    n = 24
    master0 = np.array([rng.uniform(0.6, 1.2) if i % 2 == 0 else rng.uniform(0.0, 0.2)
                        for i in range(8)], np.float32)
    xs = [torch.from_numpy(rng.uniform(0.1, 1.0, (P, n)).astype(np.float32)).cuda()
          for _ in range(2)]
    a = _state(master0)     # the no-allocation entry point
    b = _state(master0)     # the regular one, with its scratch provided here
    gathered = torch.zeros(8, dtype=torch.float16, device="cuda")
    grads = torch.zeros((P, 8), dtype=torch.float16, device="cuda")
    for t in (1, 2):        # two calls in a row: the array keeps the last call's contents
        z.zero_mlp4_zero3_step_noalloc(xs[t - 1], P, n, a[0], a[1], a[2], a[3], a[4], t, LR, B1,
                                       B2, EPS, mode)
        z.zero_mlp4_zero3_step(xs[t - 1], P, n, gathered, b[0], b[1], b[2], b[3], grads, 8, b[4],
                               t, LR, B1, B2, EPS, mode, pipelined=True)
        torch.cuda.synchronize()
        for x, y in zip(a[:3] + [a[4]], b[:3] + [b[4]]):
            assert ulp32(x.cpu().numpy(), y.cpu().numpy()) <= 2, (P, mode, t)
        assert ulp16(a[3].view(torch.int16).cpu().numpy().view(np.uint16),
                     b[3].view(torch.int16).cpu().numpy().view(np.uint16)) <= 1, (P, mode, t)


def test_no_alloc_step_refuses_more_ranks_than_its_scratch_holds(z):
    x = torch.zeros((9, 4), device="cuda")
    s = _state(np.ones(8, np.float32))
    with pytest.raises(z.ZeroError) as e:
        z.zero_mlp4_zero3_step_noalloc(x, 9, 4, s[0], s[1], s[2], s[3], s[4], 1, LR, B1, B2, EPS, 0)
    assert e.value.code == z.ZERO_EINVAL
