"""The limits of the boundary on the GPU, checked against the oracle bit for
bit: the most ranks the library takes (ZERO_MAX_RANKS = 1024) on both
kernels, and a whole-vector step of more than 2^31 elements, where every
stream's element offsets pass 32 bits.

Elements never interact, so where an array is too large for the host oracle
the oracle runs on windows of it (the step's result on a window equals the
whole problem's result there)."""
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
    yield zlib
    torch.cuda.empty_cache()


def _u16(t) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _state_np(s, b=0, e=None):
    return [s[0][b:e].cpu().numpy(), s[1][b:e].cpu().numpy(), s[2][b:e].cpu().numpy(), _u16(s[3][b:e])]


@pytest.mark.parametrize("kernel", ["vector", "bulk"])
def test_most_ranks_the_library_takes(z, kernel):
    """P = ZERO_MAX_RANKS = 1024 (128 chunks of 8 ranks on the bulk path),
    whole arrays compared after each of two steps."""
    P = z.ZERO_MAX_RANKS
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    N = 5003 if kernel == "vector" else sms * 2048 * 4 + 77
    stride = synth.round_up(N, 8)
    mode = 2 if kernel == "vector" else 0
    s = list(synth.torch_state(N, 31, "cuda"))
    ref = _state_np(s)[:3]
    for t in (1, 2):
        g = synth.torch_grads(P, N, stride, 1e-3, 40 + t, "cuda", heavy_tail_frac=0.01)
        plan = z.zero_step_plan(g, stride, *s, N, P, 2, mode)
        assert plan["kernel"] == kernel, plan
        z.zero_adam_step(g, stride, *s, N, P, 2, t, LR, B1, B2, EPS, mode)
        codes = _u16(g).reshape(-1)
        del g
        p_ref = oracle.adam_elems(codes, stride, P, *ref, t, LR, B1, B2, EPS, mode, threads=8)
        assert max_ulps(_state_np(s), ref + [p_ref]) == (0, 0), (kernel, t)
    assert z.zero_device_timeouts() == 0


def test_more_than_2_31_elements(z):
    """One rank, N = 2^31 + 4099 elements (34 GB of device memory): two
    steps on the bulk path, compared on windows at the start, across the
    2^31 boundary, at the end and at random places."""
    P, N = 1, 2**31 + 4099
    stride = synth.round_up(N, 8)
    s = list(synth.torch_state(N, 5, "cuda"))
    g = torch.empty((P, stride), dtype=torch.float16, device="cuda")
    plan = z.zero_step_plan(g, stride, *s, N, P, 2, 0)
    assert plan["kernel"] == "bulk", plan
    rng = np.random.default_rng(9)
    wins = [(0, 4096), (2**31 - 4096, 2**31 + 4096), (N - 5000, N)]
    wins += [(int(b), int(b) + 65536) for b in rng.integers(0, N - 65536, size=6)]
    refs = {w: _state_np(s, *w)[:3] for w in wins}
    for t in (1, 2):
        synth.torch_grads(P, N, stride, 1e-3, 70 + t, "cuda", heavy_tail_frac=0.01, out=g)
        wg = {(b, e): _u16(g[:, b:e]).reshape(-1) for b, e in wins}
        z.zero_adam_step(g, stride, *s, N, P, 2, t, LR, B1, B2, EPS, 0)
        for (b, e) in wins:
            ref = refs[(b, e)]
            p_ref = oracle.adam_elems(wg[(b, e)], e - b, P, *ref, t, LR, B1, B2, EPS, 0)
            assert max_ulps(_state_np(s, b, e), ref + [p_ref]) == (0, 0), (b, e, t)
    assert z.zero_device_timeouts() == 0
    del g, s
