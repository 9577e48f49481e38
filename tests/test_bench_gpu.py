"""bench.py prints one JSON line with the keys its consumers read: the profiling
case of the headline workload, and the prefill-attention, serving-step,
long-context decode and single-tile cases, each run briefly."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def test_bench_small_case_line():
    d = _run("--case", "small", "--steps", "2", "--warmup", "3", "--no-cpu-baseline")
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 3
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["gpu_launches"] > 0
    assert d["roofline"]["bound"] in ("alu", "hbm", "tensor") and 0 < d["roofline"]["frac"] < 2
    assert d["e2e"]["value"] > 0 and d["e2e"]["h2d_bytes_per_step"] > 0
    w = d["e2e"]["windows_gbs"]
    assert len(w) == d["e2e"]["windows"] and min(w) <= d["e2e"]["value"] <= max(w)   # the median window


def test_bench_prefill_attention_line():
    d = _run("--case", "prefill_attn", "--steps", "2", "--warmup", "3")
    assert d["metric"] == "chunked_prefill_attention_tflops" and d["unit"] == "TFLOP/s"
    assert d["value"] > 0 and d["ms_per_call"] > 0 and d["prefill_tokens_per_s"] > 0


def test_bench_serve_line():
    d = _run("--case", "serve", "--steps", "2", "--warmup", "3")
    assert d["metric"] == "serving_step_sequences_per_s" and d["value"] > 0 and d["ms_per_step"] > 0
    for key in ("append_us", "decode_us", "two_calls_eager_us", "graph_us", "serve_step_one_launch_us"):
        assert d[key] > 0, key
    assert 0 < d["decode_frac_hbm"] < 2


def test_bench_decode_long_line():
    d = _run("--case", "decode_long", "--steps", "2", "--warmup", "3")
    assert d["metric"] == "decode_attention_gbs" and d["unit"] == "GB/s"
    assert d["value"] > 0 and d["ms_per_call"] > 0 and 0 < d["frac_hbm"] < 2


def test_bench_tile_line():
    d = _run("--case", "tile", "--steps", "3", "--warmup", "3")
    assert d["metric"] == "single_tile_latency_us" and d["higher_is_better"] is False
    assert d["quantize_us"] > 0 and d["decode_us"] > 0
