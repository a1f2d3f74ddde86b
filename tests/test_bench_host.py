"""Host logic of bench.py without a GPU: argument defaults, the clock-log
parser, the profile lookup, and the multi-process path (barrier and the
max over ranks) as two gloo ranks on CPU."""
import os
import socket
import subprocess
import sys
import time

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_defaults():
    a = bench.parse_args([])
    # the headline is the largest workload that fits one GPU: 1.3e9 parameters at P = 16
    assert a.gpus == 1 and a.workload == "tf1p3b" and a.warmup >= 3 and a.steps >= 100
    assert not a.no_per_config
    with pytest.raises(SystemExit):
        bench.parse_args(["--warmup", "2"])
    a = bench.parse_args(["--unpadded-stride", "--no-per-config", "--workload", "shard7p5b"])
    assert a.unpadded_stride and a.no_per_config and a.workload == "shard7p5b"
    # the unpadded stride of the 7.5B shard is its natural packed length, 4 mod 8
    from zero_sharded_mixed_shard_gb300 import synth
    assert synth.WORKLOADS["shard7p5b"].rank_stride(False) % 8 == 4


def test_clock_parser_keeps_samples_of_the_timed_region():
    t0 = time.mktime(time.strptime("2026/12/02 08:00:01", "%Y/%m/%d %H:%M:%S"))
    lines = [
        "2026/12/02 08:00:00.500, 0, 900, 2070, 200.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/12/02 08:00:01.100, 0, 1900, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/12/02 08:00:01.300, 0, 1950, 2070, 950.5, 0x4, Not Active, Not Active, Not Active, Active",
        "2026/12/02 08:00:01.500, 0, 2000, 2070, 990.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
        "2026/12/02 08:00:03.000, 0, 800, 2070, 150.0, 0x0, Active, Not Active, Not Active, Not Active",
    ]
    c = bench.parse_clock_csv("\n".join(lines), t0, t0 + 0.6)
    assert c["samples"] == 3 and c["sm_mhz"] == 1950 and c["sm_max_mhz"] == 2070
    assert c["reasons"] == ["sw_power_cap"]


def test_profile_traffic_requires_matching_source_and_kernel(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "PROFILE_DIR", str(tmp_path))
    f = tmp_path / "zero_fused_step_gpt2s.txt"
    head = "kernel: zero_fused_step_tma_kernel<0,8,256,2>\n"
    f.write_text(head + f"source_sha256: {bench.kernel_source_hash()}\ntraffic_bytes_per_launch: 123\n")
    assert bench.profiled_traffic("gpt2s") == 123.0
    # a summary of the other kernel does not describe this launch
    assert bench.profiled_traffic("gpt2s", "zero_fused_step_kernel (vector width 8)") is None
    f.write_text(head + "source_sha256: 0000\ntraffic_bytes_per_launch: 123\n")
    assert bench.profiled_traffic("gpt2s") is None
    assert bench.profiled_traffic("shard7p5b") is None
    # a summary with one figure per Adam reading answers each mode with its own
    g = tmp_path / "zero_fused_step_folded.txt"
    g.write_text("kernel: zero_fused_step_tma_kernel<1,32,512,2,0>\n"
                 f"source_sha256: {bench.kernel_source_hash()}\ntraffic_bytes_per_launch: 10\n"
                 "traffic_bytes_per_launch_mode1: 10\ntraffic_bytes_per_launch_mode2: 20\n")
    assert bench.profiled_traffic("folded", mode=1) == 10.0
    assert bench.profiled_traffic("folded", mode=2) == 20.0
    assert bench.profiled_traffic("folded", mode=0) == 10.0   # no figure of its own: the summary's


def test_committed_profiles_match_the_current_kernel_source():
    """Every committed step summary was taken on the kernel source as it is
    now (else the bench's traffic would read null)."""
    for name in ("tiny", "gpt2s", "tf1p3b", "shard7p5b", "folded", "shard7p5b-unpadded"):
        kernel = "zero_fused_step_kernel" if name in ("tiny", "shard7p5b-unpadded") else "zero_fused_step_tma_kernel"
        assert bench.profiled_traffic(name, kernel) is not None, name


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    d = bench.Dist()
    d.init("gloo")
    d.barrier()
    got = d.max(10.0 + rank)
    d.barrier()
    both = d.all_true(True)
    one = d.all_true(rank == 0)     # false on one rank: false on both
    out.put((rank, d.world, got, both, one))
    d.close()


def test_two_gloo_ranks_take_the_slowest_time():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 2, 11.0, True, False), (1, 2, 11.0, True, False)]


def test_reference_arm_other_ranks_do_no_work(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--gpus", "2", "--steps", "3", "--warmup", "3"]) == 0


def test_ranks_override_is_checked_before_any_gpu_work():
    import bench
    with pytest.raises(SystemExit):
        bench.main(["--workload", "shard7p5b", "--ranks", "4"])
    with pytest.raises(SystemExit):
        bench.main(["--ranks", "0"])
    with pytest.raises(SystemExit):
        bench.main(["--workload", "shard7p5b", "--elements", "1000"])
    with pytest.raises(SystemExit):
        bench.main(["--elements", "0"])
    with pytest.raises(SystemExit):        # two GPUs asked for, one process running
        bench.main(["--gpus", "2", "--impl", "reference"])


def test_reference_arm_prints_one_contract_line():
    """bench.py --impl reference (the CPU oracle on the host cores) prints one
    JSON line with every key the benchmark contract asks for."""
    import json
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "tiny", "--steps", "2", "--warmup", "3"], capture_output=True, text=True, timeout=600,
                       cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 3
    assert d["value"] > 0 and d["higher_is_better"] is True and "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert cb["hardware_concurrency"] >= cb["affinity_cores"] >= cb["threads_used"] == cb["cores"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    # the same config object our arm prints for this workload; the sample is stated beside it
    from zero_sharded_mixed_shard_gb300 import synth
    wl = synth.WORKLOADS["tiny"]
    assert d["config"] == bench.workload_config(wl, 0, bench.l2_flush_for(wl, 0))
    assert "elements [0," in d["sample"]


def test_cpu_baseline_leg_reports_threads_and_every_config():
    """The oracle timing: all allowed cores and one thread on the headline
    workload, and a labelled per-element rate for each other workload."""
    from zero_sharded_mixed_shard_gb300 import synth
    W = synth.WORKLOADS
    cb = bench.cpu_baseline_leg(W["tiny"], 0, 1.0, [(W["gpt2s"], 0), (W["folded"], 2)])
    hw, allowed = bench.host_cores()
    assert cb["hardware_concurrency"] == hw and cb["affinity_cores"] == allowed
    assert cb["threads_used"] == allowed == cb["cores"] and cb["value"] > 0
    assert cb["single_thread"]["threads_used"] == 1 and cb["single_thread"]["value"] > 0
    per = cb["per_config"]
    assert per["gpt2s/mode0"]["kind"] == "whole step"
    assert "extrapolated" in per["folded/mode2"]["kind"]
    for e in per.values():
        assert e["value"] > 0 and e["step_s"] > 0 and e["sample"]


def test_oracle_inputs_repeat_a_draw_to_fill_a_sample():
    import numpy as np
    from zero_sharded_mixed_shard_gb300 import synth
    wl = synth.WORKLOADS["gpt2s"]
    codes, w, m, v = bench.oracle_inputs(wl, 10_000, draw=4096)
    c = codes.reshape(wl.P, 10_000)
    assert np.array_equal(c[:, 4096:8192], c[:, :4096]) and np.array_equal(w[4096:8192], w[:4096])
    assert not m.any() and not v.any() and codes.size == wl.P * 10_000


def test_kernel_source_hash_ignores_comments_only(tmp_path, monkeypatch):
    """A profile summary is keyed to the kernel's code: comment and spacing
    edits keep the key, a code edit changes it."""
    f = tmp_path / "k.cu"
    monkeypatch.setattr(bench, "KERNEL_SRC", str(f))
    f.write_text("int f(int x) { return x + 1; } // one\n")
    h0 = bench.kernel_source_hash()
    f.write_text("/* a new\n block */ int f(int x)  {\n  return x + 1; // two\n}\n")
    assert bench.kernel_source_hash() == h0
    f.write_text("int f(int x) { return x + 2; }\n")
    assert bench.kernel_source_hash() != h0
