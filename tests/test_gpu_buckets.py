"""Bucketed, stream-overlapped steps (ZeRO 技术原理：进阶与 Offload §1.5: gradients
are sent bucket by bucket while the backward pass goes on; §1.6.7: separate
CUDA streams for communication and computation).

A producer stream stands in for the backward pass: it fills the gradient
buckets in backward order, each after a deliberate delay, and records one
event per bucket; the step stream waits for each event before that bucket's
fused step.  The gradient buffers start out as NaN, so a step that ran
before its bucket was ready would differ from the whole-vector step."""
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


def _host(s):
    return [s[0].cpu().numpy(), s[1].cpu().numpy(), s[2].cpu().numpy(),
            s[3].view(torch.int16).cpu().numpy().view(np.uint16)]


def _tensors(total, rng):
    sizes = []
    while sum(sizes) < total:
        sizes.append(int(rng.integers(1, 400_000)))
    sizes[-1] -= sum(sizes) - total
    return sizes


@pytest.mark.parametrize("P,mode", [(4, 0), (8, 2), (13, 1)])
def test_bucketed_step_waits_for_each_bucket(z, P, mode):
    rng = np.random.default_rng(P)
    N = 3_000_011
    stride = synth.round_up(N, 8)
    numel = _tensors(N, rng)
    buckets = z.zero_plan_buckets(numel, 500_000, backward_order=True)
    assert len(buckets) >= 4
    codes = synth.np_grads(P, N, stride, 1e-3, 40 + P)
    final = torch.from_numpy(codes.view(np.int16)).cuda().view(torch.float16).view(P, stride)
    w0, m0, v0, p0 = synth.np_state(N, P)

    grads = torch.full((P, stride), float("nan"), dtype=torch.float16, device="cuda")
    producer = torch.cuda.Stream()
    stepper = torch.cuda.Stream()
    s = [torch.from_numpy(a.copy()).cuda() for a in (w0, m0, v0)] + \
        [torch.from_numpy(p0.view(np.int16).copy()).cuda().view(torch.float16)]
    torch.cuda.synchronize()
    events = []
    with torch.cuda.stream(producer):
        for (b, e, _, _) in buckets:
            torch.cuda._sleep(2_000_000)          # a slow "backward" for this bucket
            grads[:, b:e].copy_(final[:, b:e])
            ev = torch.cuda.Event()
            ev.record(producer)
            events.append(ev)
    z.zero_adam_step_bucketed(grads, stride, *s, N, P, 2, 3, LR, B1, B2, EPS, mode, buckets,
                              ready_events=events, stream=stepper)
    torch.cuda.synchronize()

    ref = [w0.copy(), m0.copy(), v0.copy()]
    p_ref = oracle.adam_elems(codes, stride, P, *ref, 3, LR, B1, B2, EPS, mode, threads=8)
    assert max_ulps(_host(s), ref + [p_ref]) == (0, 0)
    assert z.zero_device_timeouts() == 0


def test_range_steps_equal_whole_step(z):
    """Cuts at odd offsets: the ranges take the vector kernel and, for the
    longest one (about 6 tiles per SM, starting off a 16-byte boundary), the
    bulk pipeline with a head of elements done one by one."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    P, N = 8, sms * 2048 * 12 + 77
    stride = synth.round_up(N, 8)
    g = synth.torch_grads(P, N, stride, 1e-3, 3, "cuda")
    base = synth.torch_state(N, 3, "cuda")
    whole = [x.clone() for x in base]
    z.zero_adam_step(g, stride, *whole, N, P, 2, 2, LR, B1, B2, EPS, 0)
    parts = [x.clone() for x in base]
    cuts = sorted({0, N, 1, 12_345, 12_346, N // 3, N // 3 + 5, N // 2 + 1, N - 9})
    kernels = set()
    for b, e in zip(cuts, cuts[1:]):
        plan = z.zero_step_plan(g[:, b:], stride, *[x[b:] for x in parts], e - b, P, 2, 0)
        kernels.add(plan["kernel"])
        z.zero_adam_step_range(g, stride, b, e, *parts, N, P, 2, 2, LR, B1, B2, EPS, 0)
    assert kernels == {"bulk", "vector"}
    for x, y in zip(whole, parts):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
