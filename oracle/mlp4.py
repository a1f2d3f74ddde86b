"""The 4-layer scalar MLP of the layer-pipelined ZeRO-3 example -- oracle side.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Plain numpy, every
operation one IEEE binary32 operation (numpy's float32 add and multiply are
correctly rounded and never fused), in the order written here.

Source: 深度学习专题：模型训练的数据并行（三） §（四）ZeRO-3 层间流水线优化, 1.
前向传播和反向传播的计算资料: scalar input x and output y; layers 1-3 are
h_k = ReLU(w_k h_{k-1} + b_k) (h_0 = x), layer 4 is y = w_4 h_3 + b_4; the loss
is L = (y - x)^2 / 2; the backward pass is written out layer by layer:
dL/dy = y - x; dL/dw_4 = (y - x) h_3; dL/db_4 = y - x; dL/dh_3 = (y - x) w_4;
for k = 3, 2, 1: dL/dw_k = dL/dh_k h_{k-1} I(h_k > 0), dL/db_k = dL/dh_k
I(h_k > 0), dL/dh_{k-1} = dL/dh_k w_k I(h_k > 0).  2. 层间流水线: 4 GPUs, each
storing one layer's 2 parameters, each training on 1/4 of the mini-batch.

Readings (the page leaves them open):
* parameters in flat order (w1, b1, w2, b2, w3, b3, w4, b4): the ceil
  partition M = ceil(8/4) = 2 then gives layer k to GPU k, as the page says;
* the forward pass uses the gathered fp16 parameters, widened to fp32
  (mixed precision as in ZeRO 技术原理：进阶与 Offload §1.4);
* each rank's local gradient is the mean over its own samples (sum in sample
  order from +0, one division by the local sample count), rounded to fp16 --
  the P ranks' fp16 gradients are then what the ZeRO step reduces;
* ReLU(z) = z for z > 0 and +0 otherwise; I(h_k > 0) = (z_k > 0), and the
  masked gradient is a select (dL/dh_k where z_k > 0, +0 elsewhere);
* the reported loss of a rank is the mean of (y - x)^2 / 2 over its samples.
"""
from __future__ import annotations

import numpy as np

F = np.float32


def _relu(z):
    return np.where(z > F(0), z, F(0)).astype(F)


def _mean_rows(a):
    """Sequential fp32 sum over axis 1 (sample order) from +0, then / count."""
    acc = np.zeros(a.shape[0], F)
    for s in range(a.shape[1]):
        acc = (acc + a[:, s]).astype(F)
    return (acc / F(a.shape[1])).astype(F)


def forward(params16: np.ndarray, x: np.ndarray):
    """params16: 8 fp16 codes (w1,b1,...,w4,b4); x: float32 [P, n].
    Returns (activations dict of float32 [P, n] arrays, per-rank mean loss)."""
    p = params16.view(np.float16).astype(F)
    w = p[0::2]
    b = p[1::2]
    x = np.asarray(x, F)
    z1 = (w[0] * x + b[0]).astype(F)
    h1 = _relu(z1)
    z2 = (w[1] * h1 + b[1]).astype(F)
    h2 = _relu(z2)
    z3 = (w[2] * h2 + b[2]).astype(F)
    h3 = _relu(z3)
    y = (w[3] * h3 + b[3]).astype(F)
    d = (y - x).astype(F)
    loss = _mean_rows((F(0.5) * (d * d)).astype(F))
    return dict(x=x, z1=z1, h1=h1, z2=z2, h2=h2, z3=z3, h3=h3, y=y), loss


def local_grads(params16: np.ndarray, x: np.ndarray):
    """Each rank's mean gradient over its samples, as fp16 codes [P, 8] in
    flat parameter order, plus the per-rank loss."""
    p = params16.view(np.float16).astype(F)
    w = p[0::2]
    a, loss = forward(params16, x)
    x = a["x"]
    zero = F(0)
    dy = (a["y"] - x).astype(F)                       # dL/dy
    g = {}
    g["w4"] = (dy * a["h3"]).astype(F)
    g["b4"] = dy
    dh = (dy * w[3]).astype(F)                        # dL/dh3
    for k, (z, hin) in ((3, (a["z3"], a["h2"])), (2, (a["z2"], a["h1"])), (1, (a["z1"], x))):
        gz = np.where(z > zero, dh, zero).astype(F)   # dL/dh_k I(h_k > 0)
        g[f"w{k}"] = (gz * hin).astype(F)
        g[f"b{k}"] = gz
        dh = (gz * w[k - 1]).astype(F)                # dL/dh_{k-1}
    order = ["w1", "b1", "w2", "b2", "w3", "b3", "w4", "b4"]
    out = np.stack([_mean_rows(g[name]) for name in order], axis=1)
    return out.astype(np.float16).view(np.uint16), loss


def grads_f64(theta: np.ndarray, x: np.ndarray) -> np.ndarray:
    """The same backward formulas in float64 on float64 parameters (mean over
    all samples of x, any shape): for the finite-difference pin."""
    w, b = theta[0::2], theta[1::2]
    x = np.asarray(x, np.float64).ravel()
    z1 = w[0] * x + b[0]; h1 = np.where(z1 > 0, z1, 0.0)
    z2 = w[1] * h1 + b[1]; h2 = np.where(z2 > 0, z2, 0.0)
    z3 = w[2] * h2 + b[2]; h3 = np.where(z3 > 0, z3, 0.0)
    y = w[3] * h3 + b[3]
    dy = y - x
    g = np.zeros(8)
    g[6], g[7] = np.mean(dy * h3), np.mean(dy)
    dh = dy * w[3]
    for k, (z, hin) in ((3, (z3, h2)), (2, (z2, h1)), (1, (z1, x))):
        gz = np.where(z > 0, dh, 0.0)
        g[2 * (k - 1)], g[2 * (k - 1) + 1] = np.mean(gz * hin), np.mean(gz)
        dh = gz * w[k - 1]
    return g


def loss_f64(theta: np.ndarray, x: np.ndarray) -> float:
    w, b = theta[0::2], theta[1::2]
    x = np.asarray(x, np.float64).ravel()
    h = x
    for k in range(3):
        h = np.maximum(w[k] * h + b[k], 0.0)
    y = w[3] * h + b[3]
    return float(np.mean(0.5 * (y - x) ** 2))
