"""The benchmark's own line on the GPU: python bench.py (a short run of the
default workload -- 1.3e9 parameters at P = 16 --, with the end-to-end leg,
every other workload in the per_config block and the CPU baseline) prints
one JSON line with every key the benchmark contract asks for, each roofline
object filled from the committed profile of the current kernel source."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_default_bench_line_has_the_contract_keys():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "20", "--warmup", "3",
                        "--cpu-seconds", "2"], capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e",
                "clocks", "gpu_launches"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 20 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["value"] > 0 and d["gpu_launches"] == 20 and "workload" in d["config"] and "l2" in d["config"]
    assert d["config"]["workload"].startswith("tf1p3b") and d["config"]["N"] == 1_300_000_000
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["achieved"] > 0 and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    assert rf["traffic"] is not None and rf["traffic"] > 0, "profile summary missing or stale"
    assert rf["kernel"] == "zero_fused_step_tma_kernel"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0 and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert cb["single_thread"]["value"] > 0 and cb["affinity_cores"] >= 1
    assert set(cb["per_config"]) == {"tiny/mode0", "gpt2s/mode0", "shard7p5b/mode0", "folded/mode1",
                                     "folded/mode2"}
    ck = d["clocks"]
    assert "sm_mhz" in ck and "sm_max_mhz" in ck and isinstance(ck["reasons"], list)
    pc = d["per_config"]
    assert set(pc) == {"tiny/mode0", "gpt2s/mode0", "shard7p5b/mode0", "shard7p5b/mode0/unpadded",
                       "folded/mode1", "folded/mode2", "clocks"}
    for name, e in pc.items():
        if name == "clocks":
            continue
        r = e["roofline"]
        assert e["value"] > 0 and e["steps"] >= 20 and abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9, name
        assert r["traffic"] is not None, f"{name}: profile summary missing or stale"
    assert pc["tiny/mode0"]["roofline"]["kernel"].startswith("zero_fused_step_kernel")
    tiny = pc["tiny/mode0"]
    assert 0 < tiny["one_element_step_ms"] < tiny["roofline"]["mean_launch_ms"]
    assert tiny["back_to_back"]["ms_per_step"] > 0 and tiny["back_to_back"]["copies"] >= 2
    for name in ("gpt2s/mode0", "shard7p5b/mode0", "folded/mode1", "folded/mode2"):
        assert pc[name]["roofline"]["kernel"] == "zero_fused_step_tma_kernel", name
    assert pc["shard7p5b/mode0/unpadded"]["roofline"]["kernel"] == "zero_fused_step_kernel (vector width 4)"
    assert pc["clocks"]["samples"] >= 1
