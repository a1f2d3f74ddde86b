"""Partition, shard/tensor segment table and per-rank accounting -- oracle side.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Plain Python, written
from the pages' definitions with no attempt at speed.

Sources (page title, section):

* 深度学习专题：模型训练的数据并行（三）, §（三）ZeRO-1 优化原理 准备步骤:
  each of P GPUs manages M = ceil(N/P) parameters; GPU k (1-based) owns
  parameters s_k = 1 + (k-1) M through e_k = k M.  The same partition is
  restated in §（四） and §（五）.  Float counts per GPU: plain data parallel
  with Adam 4N (§（二）.2), ZeRO-1 2M + 2N (§（三）.2), ZeRO-2 3M + N
  (§（四）.2), ZeRO-3 4M (§（五）.2).
* ZeRO 技术原理：进阶与 Offload, §1.4 显存分析: mixed-precision model states
  2Φ + 2Φ + 12Φ = 16Φ bytes; P_os 4Φ + 12Φ/N; P_os+g 2Φ + (2Φ + 12Φ)/N;
  P_os+g+p 16Φ/N (K = 12).  §1.5 通信数据量分析: plain data parallel, P_os
  and P_os+g move about 2Φ per card per step; P_os+g+p adds one broadcast,
  50 % more (3Φ).
* 高效AI 第19讲：分布式训练（第一部分）, ZeRO 和 FSDP: 16, 2 + 2 + 12/N,
  2 + (2 + 12)/N and 16/N bytes per parameter.

Readings: indices here are 0-based, shard k = [k M, min((k+1) M, N)); the
page's e_k = k M runs past N for the last GPU when P does not divide N, so
it is clamped, and a GPU whose s_k is already past N owns nothing.
"""
from __future__ import annotations


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def shard_size(N: int, P: int) -> int:
    """M = ceil(N / P)."""
    if N < 1 or P < 1:
        raise ValueError("N and P must be positive")
    return ceil_div(N, P)


def partition(N: int, P: int) -> list[tuple[int, int]]:
    """0-based half-open bounds [begin, end) of each of the P shards.

    Written from the 1-based statement: GPU k owns s_k = 1 + (k-1) M through
    e_k = k M (inclusive), clamped to N; converted to 0-based half-open
    ranges [s_k - 1, e_k)."""
    M = shard_size(N, P)
    out = []
    for k1 in range(1, P + 1):
        s_k = 1 + (k1 - 1) * M
        e_k = min(k1 * M, N)
        if s_k > e_k:                # owns nothing
            out.append((min(s_k - 1, N), min(s_k - 1, N)))
        else:
            out.append((s_k - 1, e_k))
    return out


def owner(i: int, N: int, P: int) -> int:
    """The shard (0-based) that owns 0-based element i."""
    if not 0 <= i < N:
        raise IndexError(i)
    return i // shard_size(N, P)


def segments(tensor_numel: list[int], P: int) -> list[list[tuple[int, int, int, int]]]:
    """For each shard, the pieces of the flattened tensors it holds, as
    (tensor_id, offset_in_tensor, offset_in_shard, length), in flat order.

    Plain interval intersection of every shard with every tensor."""
    starts = []
    pos = 0
    for n in tensor_numel:
        if n < 0:
            raise ValueError("negative tensor size")
        starts.append(pos)
        pos += n
    N = pos
    out = []
    for (b, e) in partition(N, P):
        segs = []
        for tid, (ts, n) in enumerate(zip(starts, tensor_numel)):
            lo, hi = max(b, ts), min(e, ts + n)
            if lo < hi:
                segs.append((tid, lo - ts, lo - b, hi - lo))
        out.append(segs)
    return out


def floats_per_rank(N: int, P: int, stage: int) -> int:
    """Untyped float count per GPU for Adam: stage 0 (plain data parallel)
    4N, ZeRO-1 2M + 2N, ZeRO-2 3M + N, ZeRO-3 4M."""
    M = shard_size(N, P)
    return {0: 4 * N, 1: 2 * M + 2 * N, 2: 3 * M + N, 3: 4 * M}[stage]


def bytes_per_rank_mixed(N: int, P: int, stage: int, K: int = 12) -> float:
    """Mixed-precision model-state bytes per GPU: fp16 parameters (2),
    fp16 gradients (2) and K bytes of fp32 optimizer state per parameter,
    with the stage's parts divided over the P data-parallel ranks."""
    phi = float(N)
    if stage == 0:
        return (2 + 2 + K) * phi
    if stage == 1:
        return (2 + 2) * phi + K * phi / P
    if stage == 2:
        return 2 * phi + (2 + K) * phi / P
    if stage == 3:
        return (2 + 2 + K) * phi / P
    raise ValueError("stage must be 0..3")


def comm_elems_per_rank(N: int, stage: int) -> float:
    """Elements each rank sends plus receives per step: about 2N for plain
    data parallel (reduce-scatter + all-gather), ZeRO-1 and ZeRO-2; 3N for
    ZeRO-3 (one more parameter broadcast)."""
    if stage in (0, 1, 2):
        return 2.0 * N
    if stage == 3:
        return 3.0 * N
    raise ValueError("stage must be 0..3")


def buckets(tensor_numel: list[int], bucket_elems: int, backward: bool = True
            ) -> list[tuple[int, int, int, int]]:
    """Group whole tensors into buckets of at least ``bucket_elems`` elements,
    as (begin, end, first_tensor, last_tensor) of the flat vector.

    Reading of 'bucket' (ZeRO 技术原理：进阶与 Offload §1.4 and §1.5: small
    pieces are gathered into a bucket before they are sent; gradients are sent
    bucket by bucket while the backward pass goes on): walk the tensors in the
    order their gradients appear -- last to first for a backward pass -- and
    close a bucket as soon as it holds bucket_elems elements; what is left at
    the end is one more bucket, and trailing empty tensors join the previous
    bucket."""
    if bucket_elems < 1 or not tensor_numel or any(n < 0 for n in tensor_numel):
        raise ValueError("bad bucket request")
    starts = [0]
    for n in tensor_numel:
        starts.append(starts[-1] + n)
    if starts[-1] < 1:
        raise ValueError("empty vector")
    order = list(range(len(tensor_numel)))
    if backward:
        order.reverse()
    out, group, size = [], [], 0
    for i in order:
        group.append(i)
        size += tensor_numel[i]
        if size >= bucket_elems:
            lo, hi = min(group), max(group)
            out.append((starts[lo], starts[hi + 1], lo, hi))
            group, size = [], 0
    if group:
        lo, hi = min(group), max(group)
        if size > 0:
            out.append((starts[lo], starts[hi + 1], lo, hi))
        else:
            b, e, plo, phi = out[-1]
            out[-1] = (b, e, min(plo, lo), max(phi, hi))
    return out
