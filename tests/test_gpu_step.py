"""Parity of the fused CUDA step (through the C ABI) with the CPU oracle.

Tolerance (the bar for the step): 2 fp32 ulp on master / m / v and 1 fp16 ulp
on the gathered parameters, NaN matching NaN.  Shard indexing and the
gathered layout are compared bit for bit.  Both sides perform the same IEEE
binary32 operations in the same order, so the measured distance is 0 ulp.
"""
import numpy as np
import pytest

import oracle
from _helpers import assert_close, max_ulps
from zero_sharded_mixed_shard_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

LR, B1, B2, EPS = 1e-3, 0.9, 0.999, 1e-8


@pytest.fixture(scope="module")
def z(zlib, oracle_mod):
    if not torch.cuda.is_available():
        pytest.fail("the GPU tests need a CUDA device")
    return zlib


def dev_u16(codes: np.ndarray):
    """uint16 codes -> fp16 device tensor holding the same bits."""
    return torch.from_numpy(np.ascontiguousarray(codes).view(np.int16)).cuda().view(torch.float16)


def host_u16(t) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def dev_state(master, m, v, params):
    return [torch.from_numpy(master.copy()).cuda(), torch.from_numpy(m.copy()).cuda(),
            torch.from_numpy(v.copy()).cuda(), dev_u16(params)]


def host_state(s):
    return [s[0].cpu().numpy(), s[1].cpu().numpy(), s[2].cpu().numpy(), host_u16(s[3])]


def gpu_step(z, g_dev, stride, s, N, P, t, mode, stage=2):
    z.zero_adam_step(g_dev, stride, s[0], s[1], s[2], s[3], N, P, stage, t, LR, B1, B2, EPS, mode)


# ---------------------------------------------------------------------------
# small problems: whole arrays compared
# ---------------------------------------------------------------------------

SMALL = [(1, 1), (1, 4), (2, 3), (7, 4), (8, 8), (9, 4), (15, 16), (16, 1), (17, 5), (63, 64),
         (64, 64), (65, 8), (1000, 3), (4099, 4), (4099, 64), (65541, 8), (65541, 13),
         (300_007, 16), (300_007, 33), (131_072, 32), (1_000_003, 4)]


@pytest.mark.parametrize("N,P", SMALL)
def test_small_matches_oracle(z, N, P):
    worst = (0, 0)
    for padded in (True, False):
        stride = synth.round_up(N, 8) if padded else N
        for mode in (0, 1, 2):
            w0, m0, v0, p0 = synth.np_state(N, 40 + N + P)
            ref = [w0.copy(), m0.copy(), v0.copy()]
            s = dev_state(w0, m0, v0, p0)
            for t in range(1, 4):
                codes = synth.np_grads(P, N, stride, 1e-3, 7 * t + P, heavy_tail_frac=0.01,
                                       zero_frac=0.05)
                gpu_step(z, dev_u16(codes), stride, s, N, P, t, mode)
                p_ref = oracle.adam_elems(codes, stride, P, *ref, t, LR, B1, B2, EPS, mode)
                got = host_state(s)
                assert_close(got, ref + [p_ref], f"N={N} P={P} stride={stride} mode={mode} t={t}")
                u = max_ulps(got, ref + [p_ref])
                worst = (max(worst[0], u[0]), max(worst[1], u[1]))
    assert worst == (0, 0), f"max ulp {worst}: expected bit-exact agreement"


def test_tiny_workload_ten_steps(z):
    """N = 1,000,003 (P does not divide N), P = 4, ZeRO-2, 10 steps, both with
    a padded and an unpadded rank stride; whole arrays compared every step."""
    wl = synth.WORKLOADS["tiny"]
    for stride in (wl.rank_stride(True), wl.rank_stride(False)):
        w0, m0, v0, p0 = synth.np_state(wl.N, wl.seed, wl.master_sigma)
        ref = [w0.copy(), m0.copy(), v0.copy()]
        s = dev_state(w0, m0, v0, p0)
        for t in range(1, wl.steps + 1):
            codes = synth.np_grads(wl.P, wl.N, stride, wl.grad_sigma, wl.seed * 100 + t)
            z.zero_adam_step(dev_u16(codes), stride, *s, wl.N, wl.P, wl.stage, t, wl.lr, wl.b1,
                             wl.b2, wl.eps, 0)
            p_ref = oracle.adam_elems(codes, stride, wl.P, *ref, t, wl.lr, wl.b1, wl.b2, wl.eps,
                                      0, threads=8)
            got = host_state(s)
            assert max_ulps(got, ref + [p_ref]) == (0, 0), (stride, t)
        # every element of the gathered vector was written
        assert not np.any(host_u16(s[3]) == synth.SENTINEL_HALF)


def test_special_values(z):
    """Gradients holding +-0, subnormal halves, the largest half, +-inf and NaN,
    and state holding huge and tiny values: NaN and inf propagate the same way
    on both sides."""
    P, N = 4, 4096
    rng = np.random.default_rng(2)
    specials = np.array([0x0000, 0x8000, 0x0001, 0x8001, 0x03FF, 0x7BFF, 0xFBFF, 0x7C00, 0xFC00,
                         0x7E00, 0x3C00, 0x0400], np.uint16)
    codes = (rng.standard_normal(P * N) * 1e-3).astype(np.float16).view(np.uint16)
    pick = rng.random(P * N) < 0.2
    codes[pick] = rng.choice(specials, size=int(pick.sum()))
    w0 = (rng.standard_normal(N) * np.exp(rng.uniform(-30, 30, N))).astype(np.float32)
    m0 = (rng.standard_normal(N) * 1e-3).astype(np.float32)
    v0 = (rng.random(N) * 1e-6).astype(np.float32)
    for mode in (0, 1, 2):
        for t in (1, 2, 7):
            ref = [w0.copy(), m0.copy(), v0.copy()]
            s = dev_state(w0, m0, v0, np.zeros(N, np.uint16))
            _assert_path(z, "vector", dev_u16(codes), N, s, N, P, mode)
            gpu_step(z, dev_u16(codes), N, s, N, P, t, mode)
            p_ref = oracle.adam_elems(codes, N, P, *ref, t, LR, B1, B2, EPS, mode)
            assert_close(host_state(s), ref + [p_ref], f"mode={mode} t={t}")


@pytest.mark.parametrize("big", [False, True])
def test_special_state_values(z, big):
    """master / m / v holding +-inf, NaN, +-0, huge and tiny values (on both
    the vector path and the bulk pipeline): infinities and NaN go through the
    divides and the square root exactly as IEEE 754 says, on both sides."""
    P = 4
    N = (torch.cuda.get_device_properties(0).multi_processor_count * 2048 * 4 + 8) if big else 4096
    rng = np.random.default_rng(8)
    codes = synth.np_grads(P, N, N, 1e-3, 8)
    specials = np.array([np.inf, -np.inf, np.nan, 0.0, -0.0, 3e38, -3e38, 1e-45, 1e-38, 1.0],
                        np.float32)

    def sprinkle(x):
        # specials only in [N/3, N/2): on the bulk pipeline the warps that
        # hold one take the guarded branch, all others the plain one
        pick = rng.random(N) < 0.3
        pick[: N // 3] = False
        pick[N // 2:] = False
        x[pick] = rng.choice(specials, size=int(pick.sum()))
        return x

    w0 = sprinkle(rng.standard_normal(N).astype(np.float32))
    m0 = sprinkle((rng.standard_normal(N) * 1e-3).astype(np.float32))
    v0 = sprinkle((rng.random(N) * 1e-6).astype(np.float32))
    for mode in (0, 1, 2):
        for t in (1, 3):
            ref = [w0.copy(), m0.copy(), v0.copy()]
            s = dev_state(w0, m0, v0, np.zeros(N, np.uint16))
            _assert_path(z, "bulk" if big else "vector", dev_u16(codes), N, s, N, P, mode)
            gpu_step(z, dev_u16(codes), N, s, N, P, t, mode)
            p_ref = oracle.adam_elems(codes, N, P, *ref, t, LR, B1, B2, EPS, mode, threads=8)
            assert_close(host_state(s), ref + [p_ref], f"mode={mode} t={t} big={big}")


@pytest.mark.parametrize("stride", [10_004, 10_008])
@pytest.mark.parametrize("offs", [(0, 0, 0, 0, 0), (3, 3, 3, 3, 3), (1, 1, 1, 1, 1),
                                  (0, 4, 0, 0, 0), (2, 0, 2, 2, 0), (5, 1, 7, 3, 2),
                                  (4, 4, 0, 4, 4), (6, 2, 2, 6, 6), (7, 7, 7, 7, 7)])
def test_alignment_paths_and_guard_bands(z, offs, stride):
    """Buffers offset by 0..7 elements from 16-byte boundaries select the 8-,
    4-, 2- and 1-element paths (with a head of up to 7 elements done one by
    one); every byte outside the range keeps its sentinel."""
    og, ow, om, ov, op = offs
    P, N = 8, 10_001
    guard = 64
    rng = np.random.default_rng(sum(offs))
    codes = (rng.standard_normal(P * stride) * 1e-3).astype(np.float16).view(np.uint16)
    g_buf = torch.full((P * stride + 2 * guard,), 0, dtype=torch.int16, device="cuda")
    g_buf[guard + og: guard + og + P * stride] = torch.from_numpy(codes.view(np.int16)).cuda()
    g = g_buf.view(torch.float16)[guard + og:]
    w0, m0, v0, _ = synth.np_state(N, 5)
    bufs = []
    for arr, off in ((w0, ow), (m0, om), (v0, ov)):
        b = torch.full((N + 2 * guard,), -7.25, dtype=torch.float32, device="cuda")
        b[guard + off: guard + off + N] = torch.from_numpy(arr).cuda()
        bufs.append((b, off))
    p_buf = torch.full((N + 2 * guard,), 0x5555, dtype=torch.int16, device="cuda")
    for mode in (0, 2):
        s = [b[guard + off: guard + off + N] for b, off in bufs] + \
            [p_buf.view(torch.float16)[guard + op: guard + op + N]]
        # a stride of 10,004 is a multiple of 4 but not of 8: the 8-element
        # path can never serve every rank there
        z.zero_adam_step(g, stride, *s, N, P, 2, 1, LR, B1, B2, EPS, mode)
        ref = [w0.copy(), m0.copy(), v0.copy()]
        p_ref = oracle.adam_elems(codes, stride, P, *ref, 1, LR, B1, B2, EPS, mode)
        assert_close(host_state(s), ref + [p_ref], f"offsets={offs} mode={mode}")
        # restore the inputs for the next mode
        for (b, off), arr in zip(bufs, (w0, m0, v0)):
            b[guard + off: guard + off + N] = torch.from_numpy(arr).cuda()
    for b, off in bufs:
        h = b.cpu().numpy()
        assert np.all(h[:guard + off] == -7.25) and np.all(h[guard + off + N:] == -7.25)
    h = p_buf.cpu().numpy()
    assert np.all(h[:guard + op] == 0x5555) and np.all(h[guard + op + N:] == 0x5555)


@pytest.mark.parametrize("stride_pad", [0, 4, 8])
def test_alignment_of_rank_stride(z, stride_pad):
    """Rank strides of N, N + 4 and N + 8 for N = 8 * 1237 (16-byte aligned
    rows only in the last case)."""
    P, N = 16, 8 * 1237
    stride = N + stride_pad
    codes = synth.np_grads(P, N, stride, 1e-3, 77)
    w0, m0, v0, p0 = synth.np_state(N, 77)
    s = dev_state(w0, m0, v0, p0)
    gpu_step(z, dev_u16(codes), stride, s, N, P, 1, 0)
    ref = [w0.copy(), m0.copy(), v0.copy()]
    p_ref = oracle.adam_elems(codes, stride, P, *ref, 1, LR, B1, B2, EPS, 0)
    assert max_ulps(host_state(s), ref + [p_ref]) == (0, 0)


# ---------------------------------------------------------------------------
# sharding invariance and stages
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("N,P", [(1, 1), (5, 4), (9, 4), (64, 64), (63, 8), (1000, 7),
                                 (100_003, 16), (65_536, 64), (250_001, 3)])
def test_shard_calls_concatenate_to_whole_step(z, N, P):
    stride = synth.round_up(N, 8)
    codes = synth.np_grads(P, N, stride, 1e-3, N + P)
    w0, m0, v0, p0 = synth.np_state(N, N)
    g = dev_u16(codes)
    whole = dev_state(w0, m0, v0, p0)
    gpu_step(z, g, stride, whole, N, P, 3, 2)
    # full per-rank gradients, full-vector state, writes into the full vector
    full = dev_state(w0, m0, v0, p0)
    for k in range(P):
        b, e = z.zero_shard_range(N, P, k)
        z.zero_adam_step_shard(g, stride, b, k, full[0][b:], full[1][b:], full[2][b:],
                               full[3][b:], N, P, 2, 3, LR, B1, B2, EPS, 2)
    for x, y in zip(whole, full):
        assert torch.equal(x.view(torch.int8) if x.dtype == torch.float16 else x.view(torch.int32),
                           y.view(torch.int8) if y.dtype == torch.float16 else y.view(torch.int32))
    # ZeRO-3: packed receive buffers of the shard only and shard-local
    # buffers; the all-gather of the shard outputs equals the whole step
    gathered = torch.empty(N, dtype=torch.float16, device="cuda")
    M = -(-N // P)
    for k in range(P):
        b, e = z.zero_shard_range(N, P, k)
        n = e - b
        if n == 0:
            # an empty shard is accepted and writes nothing
            z.zero_adam_step_shard(g, stride, 0, k, whole[0], whole[1], whole[2], gathered, N, P,
                                   3, 3, LR, B1, B2, EPS, 2)
            continue
        for pad in (0, 3):   # an unaligned packed stride too
            mpad = M + pad
            packed = torch.zeros((P, mpad), dtype=torch.float16, device="cuda")
            packed[:, :n] = g.view(P, stride)[:, b:e]
            st = [torch.from_numpy(a[b:e].copy()).cuda() for a in (w0, m0, v0)]
            p_local = torch.empty(n, dtype=torch.float16, device="cuda")
            z.zero_adam_step_shard(packed, mpad, 0, k, *st, p_local, N, P, 3, 3, LR, B1, B2,
                                   EPS, 2)
            for x, y in zip(st, whole[:3]):
                assert torch.equal(x.view(torch.int32), y[b:e].view(torch.int32))
            gathered[b:e] = p_local
    assert torch.equal(gathered.view(torch.int16), whole[3].view(torch.int16))


def test_stages_compute_identical_bytes(z):
    P, N = 8, 50_000
    stride = N
    codes = synth.np_grads(P, N, stride, 1e-3, 3)
    g = dev_u16(codes)
    w0, m0, v0, p0 = synth.np_state(N, 3)
    outs = []
    for stage in range(4):
        s = dev_state(w0, m0, v0, p0)
        for t in (1, 2):
            gpu_step(z, g, stride, s, N, P, t, 0, stage=stage)
        outs.append(host_state(s))
    for o in outs[1:]:
        for x, y in zip(o, outs[0]):
            assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


def test_repeatable(z):
    P, N = 16, 123_457
    codes = synth.np_grads(P, N, N, 1e-3, 9)
    g = dev_u16(codes)
    w0, m0, v0, p0 = synth.np_state(N, 9)
    outs = []
    for _ in range(3):
        s = dev_state(w0, m0, v0, p0)
        gpu_step(z, g, N, s, N, P, 5, 0)
        outs.append(host_state(s))
    for o in outs[1:]:
        for x, y in zip(o, outs[0]):
            assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


def test_validation_with_device_buffers(z):
    P, N = 4, 1000
    g = torch.zeros((P, N), dtype=torch.float16, device="cuda")
    s = dev_state(*synth.np_state(N, 1))
    before = host_state(s)
    bad = [dict(N=0), dict(P=0), dict(t=0), dict(mode=5), dict(stage=7), dict(beta1=1.0),
           dict(eps=-1.0), dict(rank_stride=N - 1)]
    for kw in bad:
        a = dict(rank_stride=N, N=N, P=P, stage=2, t=1, beta1=B1, eps=EPS, mode=0)
        a.update(kw)
        with pytest.raises(z.ZeroError) as e:
            z.zero_adam_step(g, a["rank_stride"], *s, a["N"], a["P"], a["stage"], a["t"], LR,
                             a["beta1"], B2, a["eps"], a["mode"])
        assert e.value.code == z.ZERO_EINVAL
    with pytest.raises(z.ZeroError) as e:      # m aliases master
        z.zero_adam_step(g, N, s[0], s[0], s[2], s[3], N, P, 2, 1, LR, B1, B2, EPS, 0)
    assert e.value.code == z.ZERO_EOVERLAP
    with pytest.raises(z.ZeroError) as e:      # params inside the gradients
        z.zero_adam_step(g, N, s[0], s[1], s[2], g.view(-1)[10:], N, P, 2, 1, LR, B1, B2, EPS, 0)
    assert e.value.code == z.ZERO_EOVERLAP
    with pytest.raises(z.ZeroError) as e:      # fp32 buffer at an odd byte address
        z.zero_adam_step(g, N, s[0].data_ptr() + 1, s[1], s[2], s[3], N - 1, P, 2, 1, LR, B1,
                         B2, EPS, 0)
    assert e.value.code == z.ZERO_EALIGN
    torch.cuda.synchronize()
    for x, y in zip(host_state(s), before):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


# ---------------------------------------------------------------------------
# the bulk-copy pipeline: large enough that every SM gets tiles of 2048
# ---------------------------------------------------------------------------

def _tma_size(extra):
    """Enough 2048-element tiles for the bulk-copy pipeline: it is chosen
    from 4 tiles per SM on."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return sms * 2048 * 4 + extra


def _assert_path(z, kernel, g, stride, s, N, P, mode=0):
    plan = z.zero_step_plan(g, stride, *s, N, P, 2, mode)
    assert plan["kernel"] == kernel, plan


@pytest.mark.parametrize("P", [1, 2, 3, 4, 5, 6, 7, 8, 9, 13, 16, 17, 24, 33, 64, 72, 100, 128, 144, 256])
def test_tma_path_matches_oracle(z, P):
    """P that fills whole 8-rank chunks and P that leaves a partial last chunk;
    every kind of instance (P = 1, 2, 4, 8, 16, 64, 72, 128, 144, 256 of their
    own, 72 and 144 with a mean that is a true division; 3 on the generic
    one of 1024 consumers, 6, 13 and 33 on the one of 512);
    a ragged tail of 5 elements; three steps of every mode."""
    N = _tma_size(4101)            # 4 x SMs full tiles, 2 more, a partial tile, a tail of 5
    stride = synth.round_up(N, 8) + 8
    worst = (0, 0)
    for mode in (0, 1, 2):
        w0, m0, v0, p0 = synth.np_state(N, 70 + P)
        ref = [w0.copy(), m0.copy(), v0.copy()]
        s = dev_state(w0, m0, v0, p0)
        for t in range(1, 4):
            codes = synth.np_grads(P, N, stride, 1e-3, 300 * t + P, heavy_tail_frac=0.01,
                                   zero_frac=0.05)
            gpu_step(z, dev_u16(codes), stride, s, N, P, t, mode)
            p_ref = oracle.adam_elems(codes, stride, P, *ref, t, LR, B1, B2, EPS, mode, threads=8)
            u = max_ulps(host_state(s), ref + [p_ref])
            worst = (max(worst[0], u[0]), max(worst[1], u[1]))
        _assert_path(z, "bulk", dev_u16(codes), stride, s, N, P, mode)
    assert worst == (0, 0), f"P={P}: max ulp {worst}"
    assert z.zero_device_timeouts() == 0


@pytest.mark.parametrize("head", [1, 3, 7])
def test_tma_path_with_head(z, head):
    """Every buffer starts `head` elements past a 16-byte boundary: the first
    8 - head elements are done one by one, the rest by the bulk pipeline."""
    P, N = 8, _tma_size(777)
    stride = synth.round_up(N + head, 8)
    codes = synth.np_grads(P, N, stride, 1e-3, 91 + head)
    g_buf = torch.zeros(P * stride + 8, dtype=torch.int16, device="cuda")
    g_buf[head: head + P * stride] = torch.from_numpy(codes.view(np.int16)).cuda()
    g = g_buf.view(torch.float16)[head:]
    w0, m0, v0, _ = synth.np_state(N, 5)
    bufs = []
    for arr in (w0, m0, v0):
        b = torch.zeros(N + 8, dtype=torch.float32, device="cuda")
        b[head: head + N] = torch.from_numpy(arr).cuda()
        bufs.append(b[head: head + N])
    p_buf = torch.zeros(N + 8, dtype=torch.int16, device="cuda")
    params = p_buf.view(torch.float16)[head: head + N]
    _assert_path(z, "bulk", g, stride, bufs + [params], N, P)
    z.zero_adam_step(g, stride, *bufs, params, N, P, 2, 1, LR, B1, B2, EPS, 0)
    ref = [w0.copy(), m0.copy(), v0.copy()]
    p_ref = oracle.adam_elems(codes, stride, P, *ref, 1, LR, B1, B2, EPS, 0, threads=8)
    assert max_ulps(host_state(bufs + [params]), ref + [p_ref]) == (0, 0)


def test_tma_and_vector_paths_agree(z):
    """The same problem through the bulk pipeline (aligned buffers) and the
    vector path (fp16 output one element off the gradients' phase) gives the
    same bytes."""
    P, N = 16, _tma_size(123)
    stride = synth.round_up(N, 8)
    codes = synth.np_grads(P, N, stride, 1e-3, 4)
    g = dev_u16(codes)
    w0, m0, v0, p0 = synth.np_state(N, 4)
    a = dev_state(w0, m0, v0, p0)
    _assert_path(z, "bulk", g, stride, a, N, P)
    gpu_step(z, g, stride, a, N, P, 2, 0)
    b = dev_state(w0, m0, v0, p0)
    p_buf = torch.zeros(N + 1, dtype=torch.int16, device="cuda")
    b[3] = p_buf.view(torch.float16)[1:]
    _assert_path(z, "vector", g, stride, b, N, P)
    gpu_step(z, g, stride, b, N, P, 2, 0)
    for x, y in zip(host_state(a), host_state(b)):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


# ---------------------------------------------------------------------------
# the other optimizers the pages name: plain SGD and SGD with momentum
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("mode", [3, 4])
@pytest.mark.parametrize("big", [False, True])
def test_sgd_and_momentum_match_oracle(z, mode, big):
    """Both kernels (vector path for the small problem, bulk pipeline for the
    large one); the unused state is passed as NULL in odd steps and as a
    sentinel-filled buffer, which must stay untouched, in even steps."""
    P = 8
    N = (torch.cuda.get_device_properties(0).multi_processor_count * 2048 * 4 + 13) if big else 50_001
    stride = synth.round_up(N, 8)
    w0, m0, v0, p0 = synth.np_state(N, 30 + mode)
    m0 = (np.random.default_rng(1).standard_normal(N) * 1e-3).astype(np.float32)
    ref = [w0.copy(), m0.copy(), v0.copy()]
    s = dev_state(w0, m0, v0, p0)
    _assert_path(z, "bulk" if big else "vector", dev_u16(synth.np_grads(P, N, stride, 1e-3, 1)),
                 stride, s, N, P, mode)
    sentinel = torch.full((N,), 1234.5, device="cuda")
    for t in range(1, 5):
        codes = synth.np_grads(P, N, stride, 1e-3, 500 + t, heavy_tail_frac=0.01)
        pass_null = t % 2 == 1
        m_arg = s[1] if mode == 4 else (None if pass_null else sentinel)
        v_arg = None if pass_null else sentinel
        z.zero_adam_step(dev_u16(codes), stride, s[0], m_arg, v_arg, s[3], N, P, 2, t, LR, B1, B2,
                         EPS, mode)
        p_ref = oracle.adam_elems(codes, stride, P, *ref, t, LR, B1, B2, EPS, mode, threads=8)
        got = host_state(s)
        assert max_ulps([got[0], got[1] if mode == 4 else ref[1], ref[2], got[3]],
                        ref + [p_ref]) == (0, 0), (mode, big, t)
    assert bool((sentinel == 1234.5).all())
    if mode == 3:
        assert np.array_equal(host_state(s)[1], m0)        # m untouched by plain SGD


# ---------------------------------------------------------------------------
# the SM cap (zero_set_step_max_sms): fewer CTAs, the same bytes
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("cap", [1, 5, 76, 1000])
def test_step_max_sms_leaves_results_unchanged(z, cap):
    """A capped step deals the same tiles to fewer CTAs: both kernels (a
    bulk-pipeline problem with a partial tile and a ragged tail, and a small
    vector-path one) must still agree with the oracle bit for bit."""
    prev = z.zero_set_step_max_sms(cap)
    try:
        for P, N in ((8, _tma_size(4101)), (5, 70_001)):
            stride = synth.round_up(N, 8)
            w0, m0, v0, p0 = synth.np_state(N, 60 + cap)
            ref = [w0.copy(), m0.copy(), v0.copy()]
            s = dev_state(w0, m0, v0, p0)
            for t in (1, 2):
                codes = synth.np_grads(P, N, stride, 1e-3, 900 + t + cap, heavy_tail_frac=0.01)
                gpu_step(z, dev_u16(codes), stride, s, N, P, t, 0)
                p_ref = oracle.adam_elems(codes, stride, P, *ref, t, LR, B1, B2, EPS, 0, threads=8)
                assert max_ulps(host_state(s), ref + [p_ref]) == (0, 0), f"cap={cap} P={P} t={t}"
    finally:
        assert z.zero_set_step_max_sms(prev) == cap
    assert z.zero_device_timeouts() == 0


def test_concurrent_callers_on_two_streams(z):
    """Two host threads enqueue steps of two different problems on two
    streams at once (one takes the bulk pipeline, one the vector path); the
    library's per-kernel set-up is shared between them, and each result must
    still equal the oracle bit for bit."""
    import threading

    problems = [(8, _tma_size(4101)), (5, 70_001)]
    cases = []
    for k, (P, N) in enumerate(problems):
        stride = synth.round_up(N, 8)
        w0, m0, v0, p0 = synth.np_state(N, 80 + k)
        codes = [synth.np_grads(P, N, stride, 1e-3, 81 + 10 * k + t) for t in (1, 2, 3)]
        cases.append(dict(P=P, N=N, stride=stride, init=(w0, m0, v0, p0), codes=codes,
                          state=dev_state(w0, m0, v0, p0), grads=[dev_u16(c) for c in codes],
                          stream=torch.cuda.Stream()))
    torch.cuda.synchronize()
    errors = []

    def run(c):
        try:
            for t in (1, 2, 3):
                z.zero_adam_step(c["grads"][t - 1], c["stride"], *c["state"], c["N"], c["P"], 2, t,
                                 LR, B1, B2, EPS, 0, c["stream"])
        except Exception as e:   # pragma: no cover - reported below
            errors.append(e)

    ths = [threading.Thread(target=run, args=(c,)) for c in cases]
    for th in ths:
        th.start()
    for th in ths:
        th.join()
    torch.cuda.synchronize()
    assert not errors
    for c in cases:
        w0, m0, v0, _ = c["init"]
        ref = [w0.copy(), m0.copy(), v0.copy()]
        for t in (1, 2, 3):
            p_ref = oracle.adam_elems(c["codes"][t - 1], c["stride"], c["P"], *ref, t, LR, B1, B2,
                                      EPS, 0, threads=8)
        assert max_ulps(host_state(c["state"]), ref + [p_ref]) == (0, 0), c["P"]


def test_step_plan_names_the_kernel(z):
    """The diagnostic agrees with the dispatch rule: the bulk pipeline for
    aligned problems of at least 4 tiles per SM (one CTA per SM, or the SM
    cap), the vector kernel below that or off the 16-byte phase."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    P = 8

    def bufs(N, p_off=0):
        g = torch.zeros((P, synth.round_up(N, 8)), dtype=torch.float16, device="cuda")
        st = [torch.zeros(N, device="cuda") for _ in range(3)]
        p = torch.zeros(N + 8, dtype=torch.float16, device="cuda")[p_off:p_off + N]
        return g, st, p

    big = sms * 2048 * 4
    g, st, p = bufs(big)
    plan = z.zero_step_plan(g, g.shape[1], *st, p, big, P, 1, 0)
    assert plan == {"kernel": "bulk", "vector_width": 8, "ctas": sms}
    small = big - 2048
    g, st, p = bufs(small)
    plan = z.zero_step_plan(g, g.shape[1], *st, p, small, P, 1, 0)
    assert plan["kernel"] == "vector" and plan["vector_width"] == 8
    g, st, p = bufs(big, p_off=1)          # parameters one half off the others' phase
    plan = z.zero_step_plan(g, g.shape[1], *st, p, big, P, 1, 0)
    assert plan["kernel"] == "vector" and plan["vector_width"] == 1
    prev = z.zero_set_step_max_sms(10)
    try:
        g, st, p = bufs(big)
        plan = z.zero_step_plan(g, g.shape[1], *st, p, big, P, 1, 0)
        assert plan == {"kernel": "bulk", "vector_width": 8, "ctas": 10}
    finally:
        z.zero_set_step_max_sms(prev)


def test_untouched_embedding_rows(z):
    """Rows of 768 parameters that no rank's batch touched: gradient exactly
    zero on every rank (one row -0 on every rank) and moments still zero, so
    whole warps take the branch that answers zero operands directly.  Four
    steps on the bulk pipeline, whole arrays bit for bit."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    P, rows = 8, sms * 2048 * 4 // 768 + 3
    N = rows * 768
    stride = N
    codes = synth.np_grads(P, N, stride, 1e-3, 71).reshape(P, rows, 768)
    rng = np.random.default_rng(72)
    untouched = rng.random(rows) < 0.3
    codes[:, untouched, :] = 0
    codes[:, np.flatnonzero(untouched)[0], :] = 0x8000          # -0 on every rank
    codes = codes.reshape(-1)
    w0, m0, v0, p0 = synth.np_state(N, 73)
    ref = [w0.copy(), m0.copy(), v0.copy()]
    s = dev_state(w0, m0, v0, p0)
    g = dev_u16(codes)
    _assert_path(z, "bulk", g, stride, s, N, P)
    for t in range(1, 5):
        gpu_step(z, g, stride, s, N, P, t, 0)
        p_ref = oracle.adam_elems(codes, stride, P, *ref, t, LR, B1, B2, EPS, 0, threads=8)
    assert max_ulps(host_state(s), ref + [p_ref]) == (0, 0)
    # the untouched rows kept zero moments and their weights
    m_now = host_state(s)[1].reshape(rows, 768)
    assert not m_now[untouched].any()


def test_fast_mean_is_the_ieee_mean_for_every_rank_count(z):
    """The divide-free mean (Markstein's correction step) equals the correctly
    rounded sum / P for every fp32 significand and every P the library takes
    (2^23 x 1024 cases, checked on the device against its correctly rounded
    divide); by power-of-two scaling this covers every nonzero sum of fp16
    gradients."""
    n, p, s = z.zero_selftest_mean_division(1, z.ZERO_MAX_RANKS)
    assert n == 0, f"{n} mismatches, the first at P = {p}, sum = {s!r}"
