"""The layer-pipelined ZeRO-3 step of the 4-layer scalar MLP (深度学习专题：模型
训练的数据并行（三） §（四）ZeRO-3 层间流水线优化) against the oracle's training
loop: real analytic gradients feed the ZeRO step, each layer owned by one rank,
each layer's update started as soon as its backward is done.  Every step's
losses, fp16 gradients, fp32 master / m / v and the owners' fp16 shards must
match bit for bit, in the pipelined and in the serial schedule."""
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


def _init(seed):
    rng = np.random.default_rng(seed)
    master = np.array([rng.uniform(0.6, 1.2) if i % 2 == 0 else rng.uniform(0.0, 0.2)
                       for i in range(8)], np.float32)
    return master, rng


def _u16(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("P,mode", [(4, 0), (4, 2), (2, 0), (8, 1), (3, 0)])
def test_training_matches_oracle(z, P, mode):
    n, T = 32, 60
    master0, rng = _init(P + mode)
    xs = [rng.uniform(0.1, 1.0, (P, n)).astype(np.float32) for _ in range(T)]

    # oracle: local gradients, then the ZeRO step of the 8 parameters
    om, omm, ov = master0.copy(), np.zeros(8, np.float32), np.zeros(8, np.float32)
    op16 = master0.astype(np.float16).view(np.uint16).copy()
    ref = []
    for t in range(1, T + 1):
        codes, loss = mlp4.local_grads(op16, xs[t - 1])
        oracle.zero_step(codes.reshape(-1), 8, P, 8, om, omm, ov, op16, t, LR, B1, B2, EPS, mode)
        ref.append((loss.copy(), codes.copy(), om.copy(), omm.copy(), ov.copy(), op16.copy()))
    # it learns (the literal folded reading's moments degenerate, so it only
    # has to make progress)
    assert ref[-1][0].mean() < (0.5 if mode != 1 else 1.0) * ref[0][0].mean()

    for pipelined in (True, False):
        dev = "cuda"
        master = torch.from_numpy(master0.copy()).to(dev)
        m = torch.zeros(8, device=dev)
        v = torch.zeros(8, device=dev)
        shard16 = torch.from_numpy(master0.astype(np.float16)).to(dev)
        gathered16 = torch.zeros(8, dtype=torch.float16, device=dev)
        grads16 = torch.zeros((P, 8), dtype=torch.float16, device=dev)
        loss = torch.zeros(P, device=dev)
        x = torch.zeros((P, n), device=dev)
        main, side = torch.cuda.current_stream(), torch.cuda.Stream()
        for t in range(1, T + 1):
            x.copy_(torch.from_numpy(xs[t - 1]))
            z.zero_mlp4_zero3_step(x, P, n, gathered16, master, m, v, shard16, grads16, 8, loss, t,
                                   LR, B1, B2, EPS, mode, pipelined=pipelined, main_stream=main,
                                   step_stream=side)
            torch.cuda.synchronize()
            r_loss, r_codes, r_m, r_mm, r_v, r_p16 = ref[t - 1]
            what = f"P={P} mode={mode} pipelined={pipelined} t={t}"
            assert np.array_equal(loss.cpu().numpy().view(np.uint32), r_loss.view(np.uint32)), what
            assert np.array_equal(_u16(grads16), r_codes), what
            assert np.array_equal(master.cpu().numpy().view(np.uint32), r_m.view(np.uint32)), what
            assert np.array_equal(m.cpu().numpy().view(np.uint32), r_mm.view(np.uint32)), what
            assert np.array_equal(v.cpu().numpy().view(np.uint32), r_v.view(np.uint32)), what
            assert np.array_equal(_u16(shard16), r_p16), what
    assert z.zero_device_timeouts() == 0


def test_layer_kernels_against_oracle(z):
    P, n = 4, 17
    master0, rng = _init(9)
    p16 = master0.astype(np.float16)
    x = rng.uniform(0.1, 1.0, (P, n)).astype(np.float32)
    codes, loss_ref = mlp4.local_grads(p16.view(np.uint16), x)
    dp = torch.from_numpy(p16).cuda()
    dx = torch.from_numpy(x).cuda()
    grads = torch.full((P, 12), float("nan"), dtype=torch.float16, device="cuda")
    for layer in (4, 3, 2, 1):
        z.zero_mlp4_layer_grads(layer, dp, dx, P, n, grads, 12)
    loss = torch.zeros(P, device="cuda")
    z.zero_mlp4_loss(dp, dx, P, n, loss)
    torch.cuda.synchronize()
    got = _u16(grads)
    assert np.array_equal(got[:, :8], codes)
    assert np.all(np.isnan(grads[:, 8:].float().cpu().numpy()))       # nothing past the 8
    assert np.array_equal(loss.cpu().numpy().view(np.uint32), loss_ref.view(np.uint32))
    with pytest.raises(z.ZeroError):
        z.zero_mlp4_layer_grads(5, dp, dx, P, n, grads, 12)
    with pytest.raises(z.ZeroError):
        z.zero_mlp4_layer_grads(1, dp, dx, 9, n, grads, 12)


def test_rejected_step_writes_nothing(z):
    """Arguments are checked before anything is enqueued: a misaligned master
    or whole buffers that overlap leave the loss, the gathered copy, the
    gradients and the shards as they were."""
    P, n = 4, 8
    x = torch.rand((P, n), device="cuda")
    master, m, v = torch.ones(8, device="cuda"), torch.zeros(8, device="cuda"), torch.zeros(8, device="cuda")
    shard16 = torch.ones(8, dtype=torch.float16, device="cuda")
    gathered16 = torch.full((8,), 7.0, dtype=torch.float16, device="cuda")
    grads16 = torch.full((P, 8), 5.0, dtype=torch.float16, device="cuda")
    loss = torch.full((P,), 123.0, device="cuda")
    raw = torch.zeros(24, device="cuda")
    keep = [t.clone() for t in (master, m, v, shard16, gathered16, grads16, loss)]
    cases = [
        (dict(master=raw.data_ptr() + 2), z.ZERO_EALIGN),
        (dict(m=raw.data_ptr(), v=raw.data_ptr() + 16), z.ZERO_EOVERLAP),   # m [0, 32) and v [16, 48) bytes
    ]
    for kw, code in cases:
        a = dict(master=master, m=m, v=v)
        a.update(kw)
        with pytest.raises(z.ZeroError) as e:
            z.zero_mlp4_zero3_step(x, P, n, gathered16, a["master"], a["m"], a["v"], shard16, grads16, 8,
                                   loss, 1, LR, B1, B2, EPS, 0, pipelined=True)
        assert e.value.code == code, kw
    torch.cuda.synchronize()
    for t, u in zip((master, m, v, shard16, gathered16, grads16, loss), keep):
        assert torch.equal(t, u)
