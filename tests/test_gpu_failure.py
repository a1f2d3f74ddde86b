"""Failure detection without a GPU fault: the fused kernel's waits on its own
bulk copies are bounded.  The diagnostic entry point tells one barrier to
expect 16 bytes that never arrive; the wait must run out after ~2 s, count
itself, let the other copies land and return -- and the context must stay
usable for the next step."""
import time

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


def _dev(codes):
    return torch.from_numpy(np.ascontiguousarray(codes).view(np.int16)).cuda().view(torch.float16)


# P = 8: a compile-time instance, copies issued by one thread; 13 and 33: the
# run-time-P instance (peeled first / middle / last chunks), copies issued by
# the lanes of warp 0
@pytest.mark.parametrize("P", [8, 13, 33])
def test_bounded_wait_runs_out_and_the_context_survives(z, P):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    N = sms * 2048 * 4 + 3
    stride = synth.round_up(N, 8)
    codes = synth.np_grads(P, N, stride, 1e-3, 12)
    g = _dev(codes)
    w0, m0, v0, p0 = synth.np_state(N, 12)
    s = [torch.from_numpy(a.copy()).cuda() for a in (w0, m0, v0)] + [_dev(p0)]
    z.zero_device_timeouts(reset=True)
    torch.cuda.synchronize()
    t0 = time.monotonic()
    z.zero_selftest_wait_timeout(g, stride, *s, N, P, 2, 1, LR, B1, B2, EPS, 0)
    torch.cuda.synchronize()
    elapsed = time.monotonic() - t0
    assert z.zero_device_timeouts(reset=True) == 1
    assert 1.5 < elapsed < 60, elapsed

    # the context still works: a normal step from fresh state matches the oracle
    s = [torch.from_numpy(a.copy()).cuda() for a in (w0, m0, v0)] + [_dev(p0)]
    z.zero_adam_step(g, stride, *s, N, P, 2, 1, LR, B1, B2, EPS, 0)
    ref = [w0.copy(), m0.copy(), v0.copy()]
    p_ref = oracle.adam_elems(codes, stride, P, *ref, 1, LR, B1, B2, EPS, 0, threads=8)
    got = [s[0].cpu().numpy(), s[1].cpu().numpy(), s[2].cpu().numpy(),
           s[3].view(torch.int16).cpu().numpy().view(np.uint16)]
    assert max_ulps(got, ref + [p_ref]) == (0, 0)
    assert z.zero_device_timeouts() == 0


def test_diagnostic_refuses_problems_off_the_bulk_path(z):
    P, N = 4, 10_000                       # far fewer tiles than SMs
    g = torch.zeros((P, N), dtype=torch.float16, device="cuda")
    s = [torch.zeros(N, device="cuda") for _ in range(3)] + \
        [torch.zeros(N, dtype=torch.float16, device="cuda")]
    with pytest.raises(z.ZeroError) as e:
        z.zero_selftest_wait_timeout(g, N, *s, N, P, 2, 1, LR, B1, B2, EPS, 0)
    assert e.value.code == z.ZERO_EINVAL
    assert z.zero_device_timeouts() == 0
