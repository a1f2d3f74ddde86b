"""Seeded synthetic workloads for the fused ZeRO step.

This module draws inputs only.  It holds none of the step's arithmetic (no
averaging, no Adam, no fp16 rounding of results) and it imports neither the
CUDA library nor the oracle, so both sides can be fed the same bytes from it.

The five workloads mirror the shapes the ZeRO pages reason about (a flat
parameter vector of N elements, P data-parallel ranks each holding an fp16
local gradient of the whole vector, fp32 master / momentum / variance):

* ``tiny``     N = 1,000,003 (P does not divide N), P = 4, ZeRO-2
* ``gpt2s``    N = 124,439,808 (GPT-2 small's tensors, flattened), P = 8, ZeRO-1,
               1 % of gradient entries scaled x100 (heavy tail)
* ``tf1p3b``   N = 1.3e9 as 24 transformer layers at d = 2048 plus one
               embedding tensor, P = 16, ZeRO-2 (shard cuts cross tensors)
* ``shard7p5b`` one rank's shard of a 7.5e9-parameter model at P = 64
               (M = 117,187,500), ZeRO-3, gradients in a packed per-rank
               receive buffer
* ``folded``   N = 2.7e8, P = 32, folded-bias-correction Adam, 10 % exact
               zero gradients, 50 steps

Values: master ~ N(0, 0.02); local gradients ~ N(0, sigma) rounded to fp16 by
the framework's dtype conversion; m = v = 0 at t = 1.  The initial fp16
parameter buffer is filled with a sentinel (the step overwrites every
element).  ``seed = 1000 + index`` unless a test chooses its own.
"""
from __future__ import annotations

import dataclasses

import numpy as np

SENTINEL_HALF = 0x7E55  # a quiet-NaN fp16 code: any element the step skips shows up


def transformer_layer_numels(d: int = 2048) -> list[int]:
    """Tensors of one transformer block in flat order: LayerNorm 1 (weight,
    bias), fused QKV weight and bias, output projection weight and bias,
    LayerNorm 2, MLP up-projection (4d x d) weight and bias, MLP
    down-projection (d x 4d) weight and bias."""
    return [d, d, 3 * d * d, 3 * d, d * d, d, d, d, 4 * d * d, 4 * d, d * 4 * d, d]


def transformer_numels(layers: int = 24, d: int = 2048, total: int = 1_300_000_000) -> list[int]:
    """``layers`` blocks followed by one embedding tensor that brings the
    flat vector to ``total`` elements."""
    body = transformer_layer_numels(d) * layers
    rest = total - sum(body)
    if rest < 0:
        raise ValueError("the blocks alone exceed the requested total")
    return body + ([rest] if rest else [])


def gpt2_small_numels(d: int = 768, layers: int = 12, vocab: int = 50257, ctx: int = 1024) -> list[int]:
    """GPT-2 small's tensors in flat order: token and position embeddings,
    12 blocks (LayerNorm 1, fused QKV weight and bias, attention projection,
    LayerNorm 2, MLP up and down projections) and the final LayerNorm:
    124,439,808 parameters, every size a multiple of 768."""
    block = [d, d, d * 3 * d, 3 * d, d * d, d, d, d, d * 4 * d, 4 * d, 4 * d * d, d]
    return [vocab * d, ctx * d] + block * layers + [d, d]


def bytes_per_elem(P: int, mode: int) -> int:
    """Bytes one step moves per element: P fp16 gradient reads, the fp32
    state the optimizer reads and writes (master, m, v for Adam; master and
    m with momentum; master for plain SGD), one fp16 parameter write."""
    state = {3: 1, 4: 2}.get(mode, 3)
    return 2 * P + 8 * state + 2


def round_up(x: int, q: int) -> int:
    return -(-x // q) * q


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    N: int                 # parameters in the flat vector
    P: int                 # simulated data-parallel ranks
    stage: int             # ZeRO stage (0 = plain data parallel)
    modes: tuple           # Adam readings run on this workload
    steps: int             # steps the workload is run for
    grad_sigma: float
    heavy_tail_frac: float = 0.0   # fraction of gradient entries scaled x100
    zero_frac: float = 0.0         # fraction of gradient entries set to exactly 0
    master_sigma: float = 0.02
    shard: int | None = None       # one rank's shard only (per-shard entry point)
    tensors: tuple | None = None   # tensor sizes of the flat vector, if structured
    seed: int = 1000
    lr: float = 1e-3
    b1: float = 0.9
    b2: float = 0.999
    eps: float = 1e-8

    @property
    def M(self) -> int:
        return -(-self.N // self.P)

    @property
    def elems(self) -> int:
        """Elements one step updates."""
        if self.shard is None:
            return self.N
        b = min(self.shard * self.M, self.N)
        return min(b + self.M, self.N) - b

    @property
    def bytes_per_elem(self) -> int:
        """P fp16 gradient reads, fp32 master/m/v read and written, one fp16
        parameter written."""
        return 2 * self.P + 24 + 2

    def rank_stride(self, padded: bool = True) -> int:
        """Distance in elements between two ranks' gradient slices.  The full
        layout holds each rank's whole local gradient (N elements); the
        per-shard workload holds a packed receive buffer of the shard only.
        ``padded`` rounds up to a multiple of 8 elements (16 bytes) so every
        rank's slice starts on the same 16-byte phase."""
        base = self.elems if self.shard is not None else self.N
        return round_up(base, 8) if padded else base


WORKLOADS = {
    "tiny": Workload("tiny", N=1_000_003, P=4, stage=2, modes=(0,), steps=10,
                     grad_sigma=1e-3, seed=1000),
    "gpt2s": Workload("gpt2s", N=124_439_808, P=8, stage=1, modes=(0,), steps=20,
                      grad_sigma=1e-3, heavy_tail_frac=0.01, seed=1001,
                      tensors=tuple(gpt2_small_numels())),
    "tf1p3b": Workload("tf1p3b", N=1_300_000_000, P=16, stage=2, modes=(0,), steps=5,
                       grad_sigma=1e-4, tensors=tuple(transformer_numels()), seed=1002),
    "shard7p5b": Workload("shard7p5b", N=7_500_000_000, P=64, stage=3, modes=(0,), steps=5,
                          grad_sigma=1e-4, shard=0, seed=1003),
    "folded": Workload("folded", N=270_000_000, P=32, stage=2, modes=(1, 2), steps=50,
                       grad_sigma=1e-3, zero_frac=0.1, seed=1004),
}


# --------------------------------------------------------------------------
# numpy (host) generation: small problems and host-buffer runs
# --------------------------------------------------------------------------

def np_grads(P: int, n: int, stride: int, sigma: float, seed: int,
             heavy_tail_frac: float = 0.0, zero_frac: float = 0.0) -> np.ndarray:
    """fp16 gradients as a flat uint16 array of P * stride codes; rank r's n
    values start at r * stride (padding entries are 0)."""
    rng = np.random.default_rng(seed)
    out = np.zeros((P, stride), np.float16)
    for r in range(P):
        x = rng.standard_normal(n, dtype=np.float32) * np.float32(sigma)
        if heavy_tail_frac:
            x = np.where(rng.random(n, dtype=np.float32) < heavy_tail_frac,
                         x * np.float32(100.0), x)
        if zero_frac:
            x = np.where(rng.random(n, dtype=np.float32) < zero_frac, np.float32(0.0), x)
        out[r, :n] = x.astype(np.float16)
    return out.reshape(-1).view(np.uint16)


def np_state(n: int, seed: int, master_sigma: float = 0.02):
    """(master, m, v, params) with master ~ N(0, master_sigma), m = v = 0 and
    the parameter buffer filled with the sentinel code."""
    rng = np.random.default_rng(seed + 7919)
    master = (rng.standard_normal(n, dtype=np.float32) * np.float32(master_sigma))
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    params = np.full(n, SENTINEL_HALF, np.uint16)
    return master, m, v, params


# --------------------------------------------------------------------------
# torch (device) generation: full-size workloads
# --------------------------------------------------------------------------

def torch_grads(P: int, n: int, stride: int, sigma: float, seed: int, device,
                heavy_tail_frac: float = 0.0, zero_frac: float = 0.0,
                step: int = 0, out=None):
    """fp16 gradients [P, stride] on ``device`` (padding entries 0), drawn
    rank by rank from a seeded device generator.  ``step`` selects a fresh
    draw for a later step of the same workload; ``out`` reuses a buffer."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed * 1_000_003 + step)
    if out is None:
        out = torch.zeros((P, stride), dtype=torch.float16, device=device)
    else:
        assert out.shape == (P, stride) and out.dtype == torch.float16
        out[:, n:].zero_()
    for r in range(P):
        x = torch.randn(n, generator=gen, device=device, dtype=torch.float32)
        x.mul_(sigma)
        if heavy_tail_frac:
            sel = torch.rand(n, generator=gen, device=device) < heavy_tail_frac
            x[sel] *= 100.0
            del sel
        if zero_frac:
            sel = torch.rand(n, generator=gen, device=device) < zero_frac
            x[sel] = 0.0
            del sel
        out[r, :n].copy_(x)
        del x
    return out


def torch_state(n: int, seed: int, device, master_sigma: float = 0.02):
    """(master, m, v, params) on ``device``; see :func:`np_state`."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed + 7919)
    master = torch.randn(n, generator=gen, device=device, dtype=torch.float32)
    master.mul_(master_sigma)
    m = torch.zeros(n, dtype=torch.float32, device=device)
    v = torch.zeros(n, dtype=torch.float32, device=device)
    params = torch.full((n,), SENTINEL_HALF, dtype=torch.int16, device=device)
    return master, m, v, params.view(torch.float16)
