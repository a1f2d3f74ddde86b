"""Partition, layout table and accounting.

The oracle side (``oracle.layout``) is pinned against the numbers the pages
print (``tests/golden``) and against the partition's defining invariants by
brute force; the library's host C++ (through the C ABI, no GPU needed) is
then compared with the oracle."""
import os

import numpy as np
import pytest

from oracle import layout as L

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows, kv = [], {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            parts = line.split()
            if parts[0].isdigit() and len(parts[0]) == 1:
                rows.append(parts)
            else:
                kv[parts[0]] = parts[1]
    return kv, rows


# ---------------------------------------------------------------------------
# oracle pins
# ---------------------------------------------------------------------------

def test_model_states_7p5b_on_64_gpus():
    kv, rows = _golden("zero_model_states_7p5b_64gpu.txt")
    N, P = int(kv["N"]), int(kv["P"])
    for stage, printed, dec in rows:
        gb = L.bytes_per_rank_mixed(N, P, int(stage)) / 1e9
        assert round(gb, int(dec)) == float(printed), (stage, gb)
    # the unrounded figures
    assert [L.bytes_per_rank_mixed(N, P, s) / 1e9 for s in range(4)] == \
        [120.0, 31.40625, 16.640625, 1.875]


def test_bytes_per_param_and_capacity():
    kv, rows = _golden("bytes_per_param_64gpu.txt")
    P, gpu = int(kv["N_GPUS"]), float(kv["GPU_BYTES"])
    for stage, printed, dec, cap in rows:
        bpp = L.bytes_per_rank_mixed(10 ** 9, P, int(stage)) / 1e9
        assert round(bpp, int(dec)) == float(printed)
        capacity = gpu / bpp / 1e9
        if cap == "-":
            assert 100 <= capacity < 1000       # "hundreds of billions"
        else:
            assert round(capacity, len(cap.split(".")[1]) if "." in cap else 0) == float(cap)


def test_gpt2_model_states():
    kv, _ = _golden("gpt2_1p5b.txt")
    N = int(kv["N"])
    assert 2 * N / 1e9 == float(kv["fp16_weights_GB"])
    assert L.bytes_per_rank_mixed(N, 1, 0) / 1e9 == float(kv["model_states_GB"])
    # one rank holds everything: every stage gives the replicated figure
    assert {L.bytes_per_rank_mixed(N, 1, s) for s in range(4)} == {16.0 * N}


def test_float_count_limits_stated_on_the_page():
    # 深度学习专题：模型训练的数据并行（三）: as M << N the per-GPU float count of
    # ZeRO-1 tends to 2N, of ZeRO-2 to N and of ZeRO-3 to 0; plain data
    # parallel keeps 4N
    N = 10 ** 12
    P = 10 ** 6
    assert L.floats_per_rank(N, P, 0) == 4 * N
    assert abs(L.floats_per_rank(N, P, 1) / N - 2) < 1e-5
    assert abs(L.floats_per_rank(N, P, 2) / N - 1) < 1e-5
    assert L.floats_per_rank(N, P, 3) / N < 1e-5
    # sharding everything removes all redundancy: P shards of 4M cover 4N
    for N, P in [(100, 4), (101, 4), (7, 7), (5, 8)]:
        M = L.shard_size(N, P)
        assert 4 * N <= P * L.floats_per_rank(N, P, 3) < 4 * N + 4 * P
        assert M * P >= N > M * (P - 1) or M == 1


def test_comm_volume_ratio():
    # ZeRO 原理 and ZeRO 技术原理 §1.5: stages 1 and 2 move what plain data
    # parallel moves; stage 3 moves 1.5x
    for N in (1, 10 ** 6, 7_500_000_000):
        base = L.comm_elems_per_rank(N, 0)
        assert base == 2 * N
        assert L.comm_elems_per_rank(N, 1) == base == L.comm_elems_per_rank(N, 2)
        assert L.comm_elems_per_rank(N, 3) == 1.5 * base


def test_partition_worked_example():
    # N = 10, P = 4: M = 3; GPU 1..4 own 1-3, 4-6, 7-9, 10 (clamped e_4 = 12 -> 10)
    assert L.partition(10, 4) == [(0, 3), (3, 6), (6, 9), (9, 10)]
    # N = 5, P = 4: M = 2; GPU 4 would start at 7 > 5: it owns nothing
    assert L.partition(5, 4) == [(0, 2), (2, 4), (4, 5), (5, 5)]


def test_partition_brute_force():
    for N in range(1, 65):
        for P in range(1, 65):
            parts = L.partition(N, P)
            M = L.shard_size(N, P)
            assert M * P >= N and (M - 1) * P < N
            covered = []
            for b, e in parts:
                assert 0 <= b <= e <= N and e - b <= M
                covered.extend(range(b, e))
            assert covered == list(range(N))       # disjoint, ordered, complete
            sizes = [e - b for b, e in parts]
            full = [s == M for s in sizes]
            # only trailing shards are short: sizes never increase again
            assert all(sizes[k] >= sizes[k + 1] for k in range(P - 1))
            assert sum(full) >= 1
            for i in range(N):
                b, e = parts[L.owner(i, N, P)]
                assert b <= i < e


def test_segments_brute_force():
    rng = np.random.default_rng(0)
    for _ in range(300):
        numel = [int(x) for x in rng.integers(0, 9, size=int(rng.integers(1, 9)))]
        if sum(numel) == 0:
            numel[0] = 1
        P = int(rng.integers(1, 12))
        segs = L.segments(numel, P)
        # rebuild each flat element's (tensor, offset) from the pieces
        flat = [(t, o) for t, n in enumerate(numel) for o in range(n)]
        for (b, e), pieces in zip(L.partition(sum(numel), P), segs):
            got = []
            for tid, toff, soff, n in pieces:
                assert n > 0 and soff == len(got)
                got.extend((tid, toff + q) for q in range(n))
            assert got == flat[b:e]


# ---------------------------------------------------------------------------
# the library's host code against the oracle (C ABI, no GPU)
# ---------------------------------------------------------------------------

def test_lib_shard_range_matches_oracle(zlib):
    for N in range(1, 65):
        for P in range(1, 65):
            ref = L.partition(N, P)
            for k in range(P):
                assert zlib.zero_shard_range(N, P, k) == ref[k]
    for N, P in [(1_000_003, 4), (124_439_808, 8), (1_300_000_000, 16),
                 (7_500_000_000, 64), (270_000_000, 32), (2 ** 40 + 3, 1024)]:
        ref = L.partition(N, P)
        assert [zlib.zero_shard_range(N, P, k) for k in range(P)] == ref


def test_lib_memory_matches_oracle(zlib):
    for N in (1, 5, 1000, 1_000_003, 7_500_000_000):
        for P in (1, 2, 3, 64, 1024):
            for stage in range(4):
                b, f, c = zlib.zero_memory_bytes(N, P, stage)
                assert b == pytest.approx(L.bytes_per_rank_mixed(N, P, stage), rel=1e-15)
                assert f == L.floats_per_rank(N, P, stage)
                assert c == L.comm_elems_per_rank(N, stage)


def test_lib_layout_table_matches_oracle(zlib):
    rng = np.random.default_rng(1)
    cases = [([10], 4), ([5], 4), ([0, 3, 0, 2, 0], 4), ([1] * 17, 5), ([64], 64), ([3, 3], 64)]
    for _ in range(200):
        numel = [int(x) for x in rng.integers(0, 40, size=int(rng.integers(1, 12)))]
        if sum(numel) == 0:
            numel[-1] = 1
        cases.append((numel, int(rng.integers(1, 20))))
    for numel, P in cases:
        for stage in (0, 3):
            t = zlib.zero_init_layout(numel, P, stage)
            N = sum(numel)
            assert t["N"] == N and t["M"] == L.shard_size(N, P) and t["P"] == P
            assert t["shards"] == L.partition(N, P)
            assert t["segments"] == L.segments(numel, P)
            assert t["bytes_per_rank_mixed"] == pytest.approx(L.bytes_per_rank_mixed(N, P, stage))
            assert t["floats_per_rank_p1"] == L.floats_per_rank(N, P, stage)


def test_lib_layout_transformer_1p3b(zlib):
    from zero_sharded_mixed_shard_gb300 import synth
    numel = synth.transformer_numels()
    assert sum(numel) == 1_300_000_000 and len(numel) == 24 * 12 + 1
    assert sum(synth.transformer_layer_numels()) == 50_358_272
    t = zlib.zero_init_layout(numel, 16, 2)
    assert t["M"] == 81_250_000
    assert t["segments"] == L.segments(numel, 16)
    # shard cuts fall inside tensors: some tensor is split across two shards
    assert any(p[0][1] != 0 for p in t["segments"][1:])


def test_lib_layout_rejects_bad_input(zlib):
    for numel, P, stage in [([], 4, 0), ([0, 0], 4, 0), ([-1, 5], 4, 0), ([5], 0, 0),
                            ([5], 1025, 0), ([5], 4, 4), ([5], 4, -1)]:
        with pytest.raises(zlib.ZeroError) as e:
            zlib.zero_init_layout(numel, P, stage)
        assert e.value.code == zlib.ZERO_EINVAL
    with pytest.raises(zlib.ZeroError):
        zlib.zero_shard_range(10, 4, 4)
    with pytest.raises(zlib.ZeroError):
        zlib.zero_memory_bytes(0, 4, 1)


# ---------------------------------------------------------------------------
# buckets
# ---------------------------------------------------------------------------

def test_bucket_invariants_brute_force():
    rng = np.random.default_rng(4)
    for _ in range(500):
        numel = [int(x) for x in rng.integers(0, 12, size=int(rng.integers(1, 10)))]
        if sum(numel) == 0:
            numel[0] = 1
        be = int(rng.integers(1, 30))
        for backward in (True, False):
            bs = L.buckets(numel, be, backward)
            starts = np.concatenate([[0], np.cumsum(numel)])
            # disjoint, non-empty, cover [0, N), in walk order
            flat = sorted(bs)
            assert flat[0][0] == 0 and flat[-1][1] == sum(numel)
            for (b0, e0, *_), (b1, e1, *_) in zip(flat, flat[1:]):
                assert e0 == b1
            for k, (b, e, lo, hi) in enumerate(bs):
                assert b < e
                # whole tensors only
                assert starts[lo] == b and starts[hi + 1] == e
                # at least bucket_elems, except the last bucket in walk order
                if k < len(bs) - 1:
                    assert e - b >= be
                    # minimal: dropping the last tensor added leaves it short
                    last = lo if backward else hi
                    assert (e - b) - numel[last] < be or numel[last] == 0
            order = [b for b, *_ in bs]
            assert order == sorted(order, reverse=backward)


def test_lib_buckets_match_oracle(zlib):
    from zero_sharded_mixed_shard_gb300 import synth
    rng = np.random.default_rng(5)
    cases = [([10, 5, 0, 3, 20, 1], 12), ([0, 0, 7, 0, 0], 3), ([1] * 50, 7), ([100], 1),
             (synth.transformer_numels(), 1 << 25)]
    for _ in range(300):
        numel = [int(x) for x in rng.integers(0, 40, size=int(rng.integers(1, 15)))]
        if sum(numel) == 0:
            numel[-1] = 1
        cases.append((numel, int(rng.integers(1, 100))))
    for numel, be in cases:
        for backward in (True, False):
            assert zlib.zero_plan_buckets(numel, be, backward) == L.buckets(numel, be, backward)


def test_lib_buckets_reject(zlib):
    for numel, be in [([], 4), ([0, 0], 4), ([-1, 3], 4), ([5], 0)]:
        with pytest.raises(zlib.ZeroError):
            zlib.zero_plan_buckets(numel, be)
    import ctypes
    arr = (ctypes.c_int64 * 3)(5, 5, 5)
    out = (zlib.zero_bucket_t * 1)()
    n = ctypes.c_int32()
    assert zlib.lib().zero_plan_buckets(arr, 3, 5, 1, out, 1, ctypes.byref(n)) == zlib.ZERO_EINVAL
