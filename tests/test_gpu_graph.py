"""The fused step inside a CUDA graph: zero_adam_step enqueues one kernel
launch and nothing else, so after one call on the device outside capture
(which does the kernel's one-time set-up) a sequence of steps can be
captured and replayed.  Three steps t = 1, 2, 3 are captured once and the
graph is replayed twice; the buffers must then equal the oracle after the
six steps 1, 2, 3, 1, 2, 3 bit for bit, on both kernels."""
import numpy as np
import pytest

import oracle
from _helpers import max_ulps
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


@pytest.mark.parametrize("kernel", ["vector", "bulk"])
def test_steps_captured_in_a_graph(z, kernel):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    P = 8
    N = 300_007 if kernel == "vector" else sms * 2048 * 4 + 1001
    stride = synth.round_up(N, 8)
    codes = synth.np_grads(P, N, stride, 1e-3, 61, heavy_tail_frac=0.01)
    g = torch.from_numpy(codes.view(np.int16)).cuda().view(torch.float16)
    w0, m0, v0, p0 = synth.np_state(N, 62)
    s = [torch.from_numpy(a.copy()).cuda() for a in (w0, m0, v0)]
    s.append(torch.from_numpy(p0.view(np.int16).copy()).cuda().view(torch.float16))
    assert z.zero_step_plan(g, stride, *s, N, P, 2, 0)["kernel"] == kernel

    # one call outside capture sets the kernel up on this device; it runs
    # on scratch copies so the captured sequence starts from the initial state
    scratch = [x.clone() for x in s]
    z.zero_adam_step(g, stride, *scratch, N, P, 2, 1, LR, B1, B2, EPS, 0)
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            for t in (1, 2, 3):
                z.zero_adam_step(g, stride, *s, N, P, 2, t, LR, B1, B2, EPS, 0, side)
    torch.cuda.synchronize()
    # capture ran nothing: the state is still the initial one
    assert np.array_equal(s[0].cpu().numpy().view(np.uint32), w0.view(np.uint32))
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()

    ref = [w0.copy(), m0.copy(), v0.copy()]
    for t in (1, 2, 3, 1, 2, 3):
        p_ref = oracle.adam_elems(codes, stride, P, *ref, t, LR, B1, B2, EPS, 0, threads=8)
    got = [s[0].cpu().numpy(), s[1].cpu().numpy(), s[2].cpu().numpy(), _u16(s[3])]
    assert max_ulps(got, ref + [p_ref]) == (0, 0)
    assert z.zero_device_timeouts() == 0
