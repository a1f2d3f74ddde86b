"""The four full-size workloads, run through the same C-ABI calls the
benchmark times, checked against the oracle.

The GPT-2-small workload (124 M elements) is compared on whole arrays at
every checked step.  The larger ones are compared on windows: elements never
interact, so the oracle's result on a window of the flat vector equals the
full problem's result there.  Windows: the first and last 4,096 elements of
every shard, +-256 elements around every tensor boundary of the structured
vector, the first tile (2,048 elements) of every CTA's last tile of the
bulk-copy pipeline -- the far end of each CTA's walk -- and 64 random
windows of 2^20 elements.  The oracle carries its own window state from step
to step; gradients are redrawn on the device every step.
"""
import os

import numpy as np
import pytest

import oracle
from _helpers import assert_close, max_ulps
from _windows import windows
from zero_sharded_mixed_shard_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
THREADS = max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1))


@pytest.fixture(scope="module")
def z(zlib, oracle_mod):
    if not torch.cuda.is_available():
        pytest.fail("the GPU tests need a CUDA device")
    yield zlib
    torch.cuda.empty_cache()


def host_u16(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def run_workload(z, wl, mode, steps, check_steps, padded=True, kernel="bulk", whole=False):
    """Run the workload's steps; check the windows (or, with ``whole``, every
    element) against the oracle at the steps in ``check_steps``."""
    dev = "cuda"
    E, P = wl.elems, wl.P
    stride = wl.rank_stride(padded)
    g = torch.empty((P, stride), dtype=torch.float16, device=dev)
    master, m, v, params = synth.torch_state(E, wl.seed, dev, wl.master_sigma)
    # the full-size workloads run the bulk-copy pipeline, as in the benchmark
    # (an unpadded rank stride puts the ranks off the 16-byte phase: vector kernel)
    plan = z.zero_step_plan(g, stride, master, m, v, params, E, P, wl.stage, mode)
    assert plan["kernel"] == kernel, (wl.name, plan)
    wins = [(0, E)] if whole else windows(wl, wl.seed, ctas=plan["ctas"] if plan["kernel"] == "bulk" else None)
    ref = {w: [master[w[0]:w[1]].cpu().numpy(), m[w[0]:w[1]].cpu().numpy(),
               v[w[0]:w[1]].cpu().numpy()] for w in wins}
    worst = (0, 0)
    for t in range(1, steps + 1):
        synth.torch_grads(P, E, stride, wl.grad_sigma, wl.seed, dev, wl.heavy_tail_frac,
                          wl.zero_frac, step=t, out=g)
        if whole:
            wg = {(0, E): g[:, :E].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)}
        else:
            wg = {w: g[:, w[0]:w[1]].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
                  for w in wins}
        if wl.shard is None:
            z.zero_adam_step(g, stride, master, m, v, params, wl.N, P, wl.stage, t, wl.lr,
                             wl.b1, wl.b2, wl.eps, mode)
        else:
            z.zero_adam_step_shard(g, stride, 0, wl.shard, master, m, v, params, wl.N, P,
                                   wl.stage, t, wl.lr, wl.b1, wl.b2, wl.eps, mode)
        for (b, e) in wins:
            p_ref = oracle.adam_elems(wg[(b, e)].reshape(-1), e - b, P, *ref[(b, e)], t, wl.lr,
                                      wl.b1, wl.b2, wl.eps, mode, threads=THREADS)
            if t in check_steps:
                got = [master[b:e].cpu().numpy(), m[b:e].cpu().numpy(), v[b:e].cpu().numpy(),
                       host_u16(params[b:e])]
                assert_close(got, ref[(b, e)] + [p_ref], f"{wl.name} mode={mode} t={t} [{b},{e})")
                u = max_ulps(got, ref[(b, e)] + [p_ref])
                worst = (max(worst[0], u[0]), max(worst[1], u[1]))
    # every element of the gathered output was written at least once
    assert not bool((params.view(torch.int16) == synth.SENTINEL_HALF).any())
    out = (master, m, v, params)
    del g
    return worst, out


def test_gpt2s_workload(z):
    wl = synth.WORKLOADS["gpt2s"]
    worst, _ = run_workload(z, wl, 0, wl.steps, check_steps={1, 2, 5, 10, wl.steps}, whole=True)
    assert worst == (0, 0)
    torch.cuda.empty_cache()


def test_gpt2s_shards_equal_whole_step_bit_for_bit(z):
    """Full size: the P per-shard calls (full-gradient layout, grad_offset =
    k*M, writes into the gathered vector) give the same bytes as the one
    whole-vector launch."""
    wl = synth.WORKLOADS["gpt2s"]
    stride = wl.rank_stride(True)
    g = synth.torch_grads(wl.P, wl.N, stride, wl.grad_sigma, wl.seed, "cuda",
                          wl.heavy_tail_frac, step=1)
    a = synth.torch_state(wl.N, wl.seed, "cuda")
    b = [x.clone() for x in a]
    for t in (1, 2):
        z.zero_adam_step(g, stride, *a, wl.N, wl.P, wl.stage, t, wl.lr, wl.b1, wl.b2, wl.eps, 0)
        for k in range(wl.P):
            lo, hi = z.zero_shard_range(wl.N, wl.P, k)
            z.zero_adam_step_shard(g, stride, lo, k, b[0][lo:], b[1][lo:], b[2][lo:],
                                   b[3][lo:], wl.N, wl.P, wl.stage, t, wl.lr, wl.b1, wl.b2,
                                   wl.eps, 0)
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    del g, a, b
    torch.cuda.empty_cache()


def test_transformer_1p3b_workload(z):
    wl = synth.WORKLOADS["tf1p3b"]
    worst, _ = run_workload(z, wl, 0, wl.steps, check_steps=set(range(1, wl.steps + 1)))
    assert worst == (0, 0)
    torch.cuda.empty_cache()


def test_shard_of_7p5b_workload(z):
    wl = synth.WORKLOADS["shard7p5b"]
    assert wl.elems == 117_187_500 and wl.rank_stride(True) == 117_187_504
    worst, _ = run_workload(z, wl, 0, wl.steps, check_steps=set(range(1, wl.steps + 1)))
    assert worst == (0, 0)
    torch.cuda.empty_cache()


def test_shard_of_7p5b_unpadded_layout(z):
    """The packed receive buffer without padding: rank stride M = 117,187,500
    (4 mod 8), so the ranks' rows sit on alternating 8-byte phases and the
    step takes the vector kernel at width 4; two steps on sampled windows."""
    wl = synth.WORKLOADS["shard7p5b"]
    assert wl.rank_stride(False) == 117_187_500
    worst, _ = run_workload(z, wl, 0, 2, check_steps={1, 2}, padded=False, kernel="vector")
    assert worst == (0, 0)
    torch.cuda.empty_cache()


@pytest.mark.parametrize("mode", [1, 2])
def test_folded_workload_50_steps(z, mode):
    wl = synth.WORKLOADS["folded"]
    checks = {1, 2, 3, 5, 10, 20, 22, 25, 30, 40, 50}
    worst, (master, m, v, params) = run_workload(z, wl, mode, wl.steps, check_steps=checks)
    assert worst == (0, 0)
    assert not bool(torch.isnan(master).any())
    if mode == 1:
        # the literal reading's v passes the largest fp32 within the 50 steps
        assert bool(torch.isinf(v).any())
    else:
        assert bool(torch.isfinite(v).all())
    del master, m, v, params
    torch.cuda.empty_cache()
