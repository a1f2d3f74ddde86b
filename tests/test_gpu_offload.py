"""ZeRO-Offload on the GPU machine (ZeRO 技术原理：进阶与 Offload §2.2, §2.3): the
GPU reduces the ranks' gradients and sends the fp16 mean to page-locked host
memory; host functions run the CPU Adam of each piece (a group of shards)
as its gradients arrive; the fp16 weights are copied back into the gathered
device vector while the next piece is updated.  Checked
against the oracle's offload step bit for bit."""
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


def _dev16(codes):
    return torch.from_numpy(np.ascontiguousarray(codes).view(np.int16)).cuda().view(torch.float16)


def _pinned(shape, dtype):
    return torch.empty(shape, dtype=dtype, pin_memory=True)


@pytest.mark.parametrize("P,N,stride,off", [(1, 5, 5, 0), (4, 100_003, 100_008, 0),
                                            (8, 1_000_000, 1_000_008, 8),
                                            (13, 65_537, 65_541, 3), (64, 20_001, 20_008, 0)])
def test_reduce_to_fp16_mean(z, P, N, stride, off):
    codes = synth.np_grads(P, N + off, stride, 1e-3, P + N, heavy_tail_frac=0.01)
    g = _dev16(codes)
    _, g16_ref = oracle.offload_elems(codes[off:], stride, P, *synth.np_state(N, 1)[:3], 1, LR,
                                      B1, B2, EPS, 0)
    out_dev = torch.empty(N, dtype=torch.float16, device="cuda")
    z.zero_reduce_scatter_fp16(g, stride, off, P, N, out_dev)
    out_host = _pinned(N, torch.float16)
    z.zero_reduce_scatter_fp16(g, stride, off, P, N, out_host)
    torch.cuda.synchronize()
    assert np.array_equal(out_dev.view(torch.int16).cpu().numpy().view(np.uint16), g16_ref)
    assert np.array_equal(out_host.view(torch.int16).numpy().view(np.uint16), g16_ref)


@pytest.mark.parametrize("P,N,mode", [(4, 1_000_003, 0), (8, 1_000_003, 1), (13, 1_000_003, 2),
                                      (8, 6_000_011, 0), (33, 9_000_007, 2)])
def test_offload_step_matches_oracle(z, P, N, mode):
    """One piece (N below 2^20 per piece) and pipelines of several pieces:
    6 pieces of uneven shard groups (P = 8), 9 pieces of 3-4 shards each
    with a short last shard (P = 33)."""
    stride = synth.round_up(N, 8)
    w0, m0, v0, p0 = synth.np_state(N, 20 + P)
    master, m, v = (_pinned(N, torch.float32) for _ in range(3))
    master.numpy()[:], m.numpy()[:], v.numpy()[:] = w0, m0, v0
    g16_h, p16_h = _pinned(N, torch.float16), _pinned(N, torch.float16)
    params = _dev16(p0)
    ref = [w0.copy(), m0.copy(), v0.copy()]
    for t in (1, 2, 3):
        codes = synth.np_grads(P, N, stride, 1e-3, 100 * t + P, zero_frac=0.05)
        z.zero_offload_step(_dev16(codes), stride, master, m, v, g16_h, p16_h, params, N, P, 2,
                            t, LR, B1, B2, EPS, mode, cpu_threads=8)
        torch.cuda.synchronize()
        p_ref, _ = oracle.offload_elems(codes, stride, P, *ref, t, LR, B1, B2, EPS, mode)
        for got, exp in zip((master.numpy(), m.numpy(), v.numpy()), ref):
            assert np.array_equal(got.view(np.uint32), exp.view(np.uint32)), t
        assert np.array_equal(params.view(torch.int16).cpu().numpy().view(np.uint16), p_ref)
    # every shard's weights reached the gathered device vector
    assert not bool((params.view(torch.int16) == synth.SENTINEL_HALF).any())


def test_offload_step_rejects(z):
    N, P = 1000, 4
    g = torch.zeros((P, N), dtype=torch.float16, device="cuda")
    h32 = [_pinned(N, torch.float32) for _ in range(3)]
    h16 = [_pinned(N, torch.float16) for _ in range(2)]
    params = torch.zeros(N, dtype=torch.float16, device="cuda")
    for kw in (dict(t=0), dict(mode=5), dict(cpu_threads=-2), dict(stride=N - 1)):
        a = dict(t=1, mode=0, cpu_threads=1, stride=N)
        a.update(kw)
        with pytest.raises(z.ZeroError):
            z.zero_offload_step(g, a["stride"], *h32, *h16, params, N, P, 2, a["t"], LR, B1, B2,
                                EPS, a["mode"], a["cpu_threads"])
    with pytest.raises(z.ZeroError):
        z.zero_reduce_scatter_fp16(g, N, 0, P, N, g.view(-1)[5:])   # output inside the gradients
