"""Pins of the 4-layer scalar MLP oracle (深度学习专题：模型训练的数据并行（三）
§（四）ZeRO-3 层间流水线优化): the printed backward formulas against finite
differences of the loss, the fp32 path against the float64 path, a worked
example derived by hand, and a dead ReLU."""
import numpy as np

from oracle import mlp4

F16 = np.float16


def _codes(vals):
    return np.asarray(vals, F16).view(np.uint16)


def test_backward_formulas_match_finite_differences():
    rng = np.random.default_rng(0)
    for _ in range(20):
        theta = np.concatenate([[rng.uniform(0.5, 1.5), rng.uniform(0.0, 0.3)] for _ in range(4)])
        x = rng.uniform(0.1, 1.0, 64)
        g = mlp4.grads_f64(theta, x)
        for i in range(8):
            e = np.zeros(8)
            e[i] = 1e-6
            fd = (mlp4.loss_f64(theta + e, x) - mlp4.loss_f64(theta - e, x)) / 2e-6
            assert abs(fd - g[i]) <= 1e-6 * max(1.0, abs(g[i])), (i, fd, g[i])


def test_fp32_path_tracks_the_double_formulas():
    rng = np.random.default_rng(1)
    P, n = 4, 16
    for _ in range(10):
        p16 = _codes(np.concatenate([[rng.uniform(0.5, 1.5), rng.uniform(0.0, 0.3)]
                                     for _ in range(4)]))
        x = rng.uniform(0.1, 1.0, (P, n)).astype(np.float32)
        codes, loss = mlp4.local_grads(p16, x)
        theta = p16.view(F16).astype(np.float64)
        per_rank = np.stack([mlp4.grads_f64(theta, x[r]) for r in range(P)])
        got = codes.view(F16).astype(np.float64)
        assert np.all(np.abs(got - per_rank) <= 2e-3 * np.abs(per_rank) + 1e-6)
        assert np.allclose(loss, [mlp4.loss_f64(theta, x[r]) for r in range(P)], rtol=1e-5)


def test_worked_example():
    # w = (1, 1, 1, 2), b = 0, x = 0.5: h1 = h2 = h3 = 0.5, y = 1, dL/dy = 0.5
    # dw4 = 0.5 * 0.5, db4 = 0.5, dL/dh3 = 0.5 * 2 = 1
    # dw3 = 1 * 0.5, db3 = 1, dL/dh2 = 1;  likewise layers 2 and 1
    p16 = _codes([1, 0, 1, 0, 1, 0, 2, 0])
    x = np.full((2, 3), 0.5, np.float32)
    codes, loss = mlp4.local_grads(p16, x)
    expect = np.array([0.5, 1, 0.5, 1, 0.5, 1, 0.25, 0.5], F16)
    assert np.array_equal(codes, np.tile(expect.view(np.uint16), (2, 1)))
    assert np.array_equal(loss, np.full(2, 0.125, np.float32))


def test_dead_relu_stops_the_gradient_below():
    # b1 = -2 keeps z1 = w1 x + b1 < 0 for x < 1: layer 1 gets no gradient, and
    # h1 = 0 makes w2's gradient 0 too; b2 still gets one (z2 = b2 > 0)
    p16 = _codes([1, -2, 1, 0.25, 1, 0, 1, 0])
    x = np.array([[0.25, 0.5, 0.75]], np.float32)
    codes, _ = mlp4.local_grads(p16, x)
    g = codes.view(F16)[0].astype(np.float64)
    assert g[0] == 0 and g[1] == 0 and g[2] == 0
    assert g[3] != 0 and g[6] != 0 and g[7] != 0
