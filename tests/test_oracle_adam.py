"""Pins of the oracle's step against what the pages and the mathematics fix,
independently of the oracle's own code:

* the gradient mean on rank data whose mean is exactly representable
  (all-reduce mean, 高效AI 第19讲 通信原语);
* the first Adam step from m = v = 0 in closed form, -lr*g/(|g|+eps), for
  every reading (深度学习专题：模型训练的数据并行（三） §（一）: m0 = v0 = 0,
  eps outside the square root);
* the two-step closed forms of each reading, derived by hand, with two
  different gradients (so a swapped beta, a wrong power in the bias
  correction or a dropped term changes the result);
* the constant-gradient steady state of the standard form (m_hat = g);
* the literal folded reading's constant-gradient factors 1/(1-b1^2),
  1/(1-b2^2) and its overflow of v without NaN;
* the cast of the new weights against numpy's float16;
* the shard-by-shard all-gather form against the unsharded loop, for every
  N <= 64 and P <= 64;
* a double-precision evaluation bounding the fp32 rounding.
"""
import numpy as np
import pytest

B1, B2 = np.float32(0.9), np.float32(0.999)
LR = np.float32(1e-3)


def f64(x):
    return float(np.float64(np.float32(x)))


def run(oracle, ranks, w, m, v, t, mode, lr=LR, b1=B1, b2=B2, eps=1e-8):
    """One oracle step; ranks is a P x n float array rounded to fp16."""
    codes = np.ascontiguousarray(np.asarray(ranks, np.float16)).view(np.uint16)
    P, n = codes.shape
    p = oracle.adam_elems(codes.reshape(-1), n, P, w, m, v, t, lr, b1, b2, eps, mode)
    return p


def test_mean_of_distinct_ranks_is_exact(oracle_mod):
    # rank r holds (r + 1 + j) * 2^-12 at element j: the mean (j + (P+1)/2) * 2^-12
    # is exact, so the first-step moments are single rounded products.
    for P in (1, 2, 3, 4, 5, 7, 8, 16, 33, 64):
        n = 37
        j = np.arange(n)
        ranks = np.array([(r + 1 + j) * 2.0 ** -12 for r in range(P)])
        g = ((j + (P + 1) / 2) * 2.0 ** -12).astype(np.float32)
        w = np.zeros(n, np.float32)
        m = np.zeros(n, np.float32)
        v = np.zeros(n, np.float32)
        run(oracle_mod, ranks, w, m, v, 1, 0)
        omb1 = np.float32(1) - B1
        omb2 = np.float32(1) - B2
        assert np.array_equal(m, omb1 * g), P
        assert np.array_equal(v, omb2 * (g * g)), P


def test_cancelling_ranks_leave_weights_untouched(oracle_mod):
    n = 16
    x = np.linspace(-0.5, 0.5, n)
    ranks = np.stack([x, -x, x, -x])
    w0 = np.linspace(-1, 1, n).astype(np.float32)
    for mode in (0, 1, 2):
        w, m, v = w0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
        run(oracle_mod, ranks, w, m, v, 1, mode)
        assert np.array_equal(w, w0) and not m.any() and not v.any()


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("eps", [1e-8, 1e-3])
def test_first_step_closed_form(oracle_mod, mode, eps):
    # P = 1 so that g is the fp16 gradient itself
    g = np.array([1e-3, -1e-3, 0.5, -2.0, 3e-2, -6e-8, 1e-5, 1.0, -1e-4, 65504.0],
                 np.float16).astype(np.float64)
    n = g.size
    w0 = np.float32(0.0123) * np.ones(n, np.float32)
    w, m, v = w0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    run(oracle_mod, g[None, :], w, m, v, 1, mode, eps=eps)
    step = f64(LR) * g / (np.abs(g) + f64(eps))
    expect = w0.astype(np.float64) - step
    tol = np.spacing(np.abs(w).astype(np.float32)) + np.abs(step) * 2e-6
    assert np.all(np.abs(w - expect) <= tol)
    # the update has the opposite sign of the gradient, about lr in size
    assert np.all(np.sign(w0 - w) == np.sign(g))


def _two_step(oracle, mode, g1, g2, eps=1e-8):
    n = g1.size
    w0 = np.full(n, 0.25, np.float32)
    w, m, v = w0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    run(oracle, g1[None, :], w, m, v, 1, mode, eps=eps)
    w1 = w.copy()
    run(oracle, g2[None, :], w, m, v, 2, mode, eps=eps)
    return w0, w1, w, m, v


G1 = np.array([2e-3, -1e-3, 0.25, 1e-4, -0.5], np.float16).astype(np.float64)
G2 = np.array([-1e-3, -3e-3, 0.125, 4e-4, 0.5], np.float16).astype(np.float64)


@pytest.mark.parametrize("mode", [0, 2])
def test_two_steps_standard_and_folded_storage(oracle_mod, mode):
    b1, b2, lr, eps = f64(B1), f64(B2), f64(LR), 1e-8
    w0, w1, w2, m, v = _two_step(oracle_mod, mode, G1, G2, eps)
    # hand derivation: m2 = (1-b1)(b1 g1 + g2), 1 - b1^2 = (1-b1)(1+b1)
    mh2 = (b1 * G1 + G2) / (1 + b1)
    vh2 = (b2 * G1 ** 2 + G2 ** 2) / (1 + b2)
    u1 = lr * G1 / (np.abs(G1) + eps)
    u2 = lr * mh2 / (np.sqrt(vh2) + eps)
    if mode == 0:
        m_exp, v_exp = (1 - b1) * (b1 * G1 + G2), (1 - b2) * (b2 * G1 ** 2 + G2 ** 2)
    else:
        m_exp, v_exp = mh2, vh2
    assert np.allclose(m, m_exp, rtol=1e-5, atol=0)
    assert np.allclose(v, v_exp, rtol=1e-5, atol=0)
    tol = 2 * np.spacing(np.float32(0.25)) + (np.abs(u1) + np.abs(u2)) * 1e-5
    assert np.all(np.abs(w2 - (w0.astype(np.float64) - u1 - u2)) <= tol)


def test_two_steps_folded_literal(oracle_mod):
    b1, b2, lr, eps = f64(B1), f64(B2), f64(LR), 1e-8
    w0, w1, w2, m, v = _two_step(oracle_mod, 1, G1, G2, eps)
    # hand derivation: m1 = g1, v1 = g1^2; m2 = (b1 m1 + (1-b1) g2) / (1-b1^2)
    m_exp = (b1 * G1 + (1 - b1) * G2) / (1 - b1 ** 2)
    v_exp = (b2 * G1 ** 2 + (1 - b2) * G2 ** 2) / (1 - b2 ** 2)
    assert np.allclose(m, m_exp, rtol=1e-5, atol=0)
    assert np.allclose(v, v_exp, rtol=1e-4, atol=0)
    u1 = lr * G1 / (np.abs(G1) + eps)
    u2 = lr * m_exp / (np.sqrt(v_exp) + eps)
    tol = 2 * np.spacing(np.float32(0.25)) + (np.abs(u1) + np.abs(u2)) * 1e-4
    assert np.all(np.abs(w2 - (w0.astype(np.float64) - u1 - u2)) <= tol)


def test_folded_literal_constant_gradient_factors(oracle_mod):
    # constant g: m_2 = g / (1 - b1^2) = g / 0.19 and v_2 = g^2 / (1 - b2^2)
    g = np.array([1e-3, -0.25], np.float16).astype(np.float64)
    _, _, _, m, v = _two_step(oracle_mod, 1, g, g)
    b1, b2 = f64(B1), f64(B2)
    assert np.allclose(m / g, 1 / (1 - b1 * b1), rtol=1e-5)
    assert np.allclose(v / g ** 2, 1 / (1 - b2 * b2), rtol=1e-4)
    assert abs(1 / (1 - 0.9 ** 2) - 5.263157894736842) < 1e-12


def test_folded_literal_overflows_without_nan(oracle_mod):
    # the literal recursion divides an already-divided v again each step: for
    # a constant gradient of 1e-3 it passes the largest fp32 within ~25 steps;
    # sqrt(inf) makes the update 0, never NaN
    n = 8
    g = np.full((1, n), 1e-3)
    w, m, v = np.full(n, 0.5, np.float32), np.zeros(n, np.float32), np.zeros(n, np.float32)
    first_inf = None
    for t in range(1, 41):
        run(oracle_mod, g, w, m, v, t, 1)
        assert not np.isnan(w).any() and not np.isnan(m).any() and not np.isnan(v).any()
        if first_inf is None and np.isinf(v).any():
            first_inf = t
    assert first_inf is not None and 15 <= first_inf <= 30
    w_before = w.copy()
    run(oracle_mod, g, w, m, v, 41, 1)
    assert np.array_equal(w, w_before)


@pytest.mark.parametrize("mode", [0, 2])
def test_constant_gradient_steady_state(oracle_mod, mode):
    # standard Adam: with g constant, m_hat = g and v_hat = g^2 for every t,
    # so each update is lr * g / (|g| + eps)
    g = np.array([1e-3, -2e-3, 0.1, -0.5, 3e-5], np.float16).astype(np.float64)
    n, T = g.size, 30
    w0 = np.full(n, 0.75, np.float32)
    w, m, v = w0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    for t in range(1, T + 1):
        run(oracle_mod, g[None, :], w, m, v, t, mode)
    u = f64(LR) * g / (np.abs(g) + 1e-8)
    expect = w0.astype(np.float64) - T * u
    tol = T * np.spacing(np.float32(0.75)) + T * np.abs(u) * 1e-5
    assert np.all(np.abs(w - expect) <= tol)


def test_cast_matches_numpy_float16(oracle_mod):
    from zero_sharded_mixed_shard_gb300 import synth
    P, n = 4, 5000
    codes = synth.np_grads(P, n, n, 1e-2, 11)
    w, m, v, _ = synth.np_state(n, 11, master_sigma=3.0)
    p = oracle_mod.adam_elems(codes, n, P, w, m, v, 1, 1e-3, 0.9, 0.999, 1e-8, 0)
    assert np.array_equal(p, w.astype(np.float16).view(np.uint16))


def test_sharded_all_gather_equals_unsharded_loop(oracle_mod):
    rng = np.random.default_rng(3)
    for N in range(1, 65):
        for P in sorted({1, 2, 3, 4, 5, 7, 8, 13, 16, 31, 32, 63, 64, N, N + 1}):
            if P > 64:
                continue
            stride = N + int(rng.integers(0, 3))
            codes = (rng.standard_normal(P * stride) * 1e-2).astype(np.float16).view(np.uint16)
            w0 = rng.standard_normal(N).astype(np.float32)
            m0 = (rng.standard_normal(N) * 1e-3).astype(np.float32)
            v0 = (rng.random(N) * 1e-6).astype(np.float32)
            a = [w0.copy(), m0.copy(), v0.copy()]
            params = np.full(N, 0x7E55, np.uint16)
            oracle_mod.zero_step(codes, stride, P, N, *a, params, 3, 1e-3, 0.9, 0.999, 1e-8, 0)
            b = [w0.copy(), m0.copy(), v0.copy()]
            p2 = oracle_mod.adam_elems(codes, stride, P, *b, 3, 1e-3, 0.9, 0.999, 1e-8, 0)
            assert np.array_equal(params, p2), (N, P)
            for x, y in zip(a, b):
                assert np.array_equal(x.view(np.uint32), y.view(np.uint32)), (N, P)


def test_thread_split_is_bitwise_neutral(oracle_mod):
    from zero_sharded_mixed_shard_gb300 import synth
    P, n = 8, 100_003
    codes = synth.np_grads(P, n, n + 5, 1e-3, 21)
    outs = []
    for threads in (1, 3, 8):
        w, m, v, _ = synth.np_state(n, 21)
        p = oracle_mod.adam_elems(codes, n + 5, P, w, m, v, 4, 1e-3, 0.9, 0.999, 1e-8, 2,
                                  threads=threads)
        outs.append((w, m, v, p))
    for o in outs[1:]:
        for x, y in zip(o, outs[0]):
            assert np.array_equal(x, y)


@pytest.mark.parametrize("mode", [0, 2])
def test_fp32_rounding_bounded_by_double_evaluation(oracle_mod, mode):
    from zero_sharded_mixed_shard_gb300 import synth
    P, n, T = 8, 4096, 20
    w, m, v, _ = synth.np_state(n, 3)
    w64, m64, v64 = w.astype(np.float64), m.astype(np.float64), v.astype(np.float64)
    for t in range(1, T + 1):
        codes = synth.np_grads(P, n, n, 1e-3, 100 + t)
        oracle_mod.adam_elems(codes, n, P, w, m, v, t, 1e-3, 0.9, 0.999, 1e-8, mode)
        oracle_mod.adam_elems_f64(codes, n, P, w64, m64, v64, t, 1e-3, f64(B1), f64(B2),
                                  f64(1e-8), mode)
        tol = 2 * t * np.spacing(np.abs(w)) + 2e-6 * t * 1e-3
        assert np.all(np.abs(w - w64) <= tol), t


def test_folded_storage_tracks_standard(oracle_mod):
    # mode 2 stores m/(1-b1^t), v/(1-b2^t) of the same averages as mode 0
    from zero_sharded_mixed_shard_gb300 import synth
    P, n, T = 4, 4096, 50
    s0 = list(synth.np_state(n, 9))[:3]
    s2 = [x.copy() for x in s0]
    for t in range(1, T + 1):
        codes = synth.np_grads(P, n, n, 1e-3, 500 + t)
        oracle_mod.adam_elems(codes, n, P, *s0, t, 1e-3, 0.9, 0.999, 1e-8, 0)
        oracle_mod.adam_elems(codes, n, P, *s2, t, 1e-3, 0.9, 0.999, 1e-8, 2)
    assert np.max(np.abs(s2[0].astype(np.float64) - s0[0])) <= T * 1e-3 * 1e-5
    bc1 = 1 - f64(B1) ** T
    assert np.allclose(s2[1], s0[1] / bc1, rtol=1e-3, atol=1e-12)


# ---------------------------------------------------------------------------
# ZeRO-Offload (ZeRO 技术原理：进阶与 Offload §2.2: the fp16 gradient crosses to
# the CPU, which runs the update and float2half)
# ---------------------------------------------------------------------------

def _rank_order_mean_fp16(codes, stride, P, n):
    """numpy: fp32 sum in rank order (one rounded add per rank), / P, to fp16."""
    x = codes.view(np.float16).reshape(P, stride)[:, :n].astype(np.float32)
    acc = np.zeros(n, np.float32)
    for r in range(P):
        acc = acc + x[r]
    return (acc / np.float32(P)).astype(np.float16)


@pytest.mark.parametrize("P", [1, 3, 4, 8, 16])
@pytest.mark.parametrize("mode", [0, 1, 2])
def test_offload_is_the_step_on_the_fp16_mean(oracle_mod, P, mode):
    from zero_sharded_mixed_shard_gb300 import synth
    n, stride = 5000, 5003
    codes = synth.np_grads(P, n, stride, 1e-3, 60 + P, heavy_tail_frac=0.05)
    w0, m0, v0, _ = synth.np_state(n, 61)
    a = [w0.copy(), m0.copy(), v0.copy()]
    p_off, g16 = oracle_mod.offload_elems(codes, stride, P, *a, 2, 1e-3, 0.9, 0.999, 1e-8, mode)
    # the gradient that crossed is numpy's fp16 of the rank-order mean
    mean16 = _rank_order_mean_fp16(codes, stride, P, n)
    assert np.array_equal(g16, mean16.view(np.uint16))
    # and the rest is exactly the one-rank step on that gradient
    b = [w0.copy(), m0.copy(), v0.copy()]
    p_one = oracle_mod.adam_elems(mean16.view(np.uint16), n, 1, *b, 2, 1e-3, 0.9, 0.999, 1e-8,
                                  mode)
    assert np.array_equal(p_off, p_one)
    for x, y in zip(a, b):
        assert np.array_equal(x.view(np.uint32), y.view(np.uint32))


def test_offload_differs_from_fused_only_through_the_gradient_rounding(oracle_mod):
    # with gradients whose mean is exactly an fp16 value the two agree bit for bit
    n, P = 64, 4
    j = np.arange(n)
    ranks = np.array([(r + 1 + j) * 2.0 ** -12 for r in range(P)], np.float16)
    codes = ranks.view(np.uint16).reshape(-1)
    w0 = np.linspace(-1, 1, n).astype(np.float32)
    a = [w0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)]
    b = [w0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)]
    p1, _ = oracle_mod.offload_elems(codes, n, P, *a, 1, 1e-3, 0.9, 0.999, 1e-8, 0)
    p2 = oracle_mod.adam_elems(codes, n, P, *b, 1, 1e-3, 0.9, 0.999, 1e-8, 0)
    assert np.array_equal(p1, p2)


# ---------------------------------------------------------------------------
# the other optimizers the pages name: plain SGD (深度学习专题：模型训练的数据并行
# （三） §（一）) and SGD with momentum (ZeRO 技术原理：进阶与 Offload §1.1.1)
# ---------------------------------------------------------------------------

def test_sgd_steps_and_independence_of_t(oracle_mod):
    g = np.array([1e-3, -2e-3, 0.5, -0.25, 3e-5], np.float16).astype(np.float64)
    n, T = g.size, 40
    w0 = np.full(n, 0.75, np.float32)
    w, m, v = w0.copy(), np.full(n, 7.0, np.float32), np.full(n, 9.0, np.float32)
    for t in range(1, T + 1):
        run(oracle_mod, g[None, :], w, m, v, t, 3)
    expect = w0.astype(np.float64) - T * f64(LR) * g
    assert np.all(np.abs(w - expect) <= T * np.spacing(np.float32(0.75)) + T * np.abs(g) * 1e-6)
    assert np.all(m == 7.0) and np.all(v == 9.0)              # no moments in plain SGD
    # the step does not depend on t (no bias correction)
    a, b = w0.copy(), w0.copy()
    run(oracle_mod, g[None, :], a, m, v, 1, 3)
    run(oracle_mod, g[None, :], b, m, v, 1000, 3)
    assert np.array_equal(a, b)


def test_momentum_geometric_series(oracle_mod):
    # constant g from m = 0: m_t = g (1 - mu^t) / (1 - mu); w_T = w0 - lr sum_t m_t
    g = np.array([1e-3, -2e-3, 0.5, -0.25], np.float16).astype(np.float64)
    n, T, mu = g.size, 25, f64(B1)
    w0 = np.full(n, 0.5, np.float32)
    w, m, v = w0.copy(), np.zeros(n, np.float32), np.full(n, 3.0, np.float32)
    for t in range(1, T + 1):
        run(oracle_mod, g[None, :], w, m, v, t, 4)
    m_exp = g * (1 - mu ** T) / (1 - mu)
    assert np.allclose(m, m_exp, rtol=1e-5, atol=0)
    s = sum((1 - mu ** t) / (1 - mu) for t in range(1, T + 1))
    expect = w0.astype(np.float64) - f64(LR) * g * s
    assert np.all(np.abs(w - expect) <= T * np.spacing(np.float32(0.5)) + np.abs(g) * s * 1e-4)
    assert np.all(v == 3.0)


def test_momentum_two_steps_by_hand(oracle_mod):
    # m1 = g1 exactly; m2 = mu g1 + g2; w2 = w0 - lr g1 - lr (mu g1 + g2)
    w0 = np.full(G1.size, 0.25, np.float32)
    w, m, v = w0.copy(), np.zeros(G1.size, np.float32), np.zeros(G1.size, np.float32)
    run(oracle_mod, G1[None, :], w, m, v, 1, 4)
    assert np.array_equal(m, G1.astype(np.float32))
    run(oracle_mod, G2[None, :], w, m, v, 2, 4)
    mu, lr = f64(B1), f64(LR)
    assert np.allclose(m, mu * G1 + G2, rtol=1e-6, atol=1e-12)
    expect = w0.astype(np.float64) - lr * G1 - lr * (mu * G1 + G2)
    assert np.all(np.abs(w - expect) <= 3 * np.spacing(np.float32(0.25)))
