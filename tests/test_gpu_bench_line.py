"""The native arm of bench.py prints one JSON line with every key of its contract:
the metric, the whole-job value and its unit, the step counts, the roofline of
the dominant kernel, the CPU baseline, the end-to-end figure with its host<->device
bytes, the number of the library's launches, and the SM clocks seen during the
timed region. Run on the tiny workload, for the dispatch+combine step and the
step with the expert stage."""
from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest

from gpu_common import require_gpu

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _line(*extra):
    res = subprocess.run([sys.executable, "bench.py", "--workload", "tiny", "--steps", "3", "--warmup", "3",
                          "--cpu-seconds", "1", *extra], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, res.stdout[-2000:]
    return json.loads(lines[0])


def _check_common(j):
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks", "cpu_baseline"):
        assert key in j, key
    assert j["n_gpus"] == 1 and j["steps"] == 3 and j["warmup"] == 3 and j["value"] > 0 and j["ms_per_step"] > 0
    assert j["higher_is_better"] is True and j["scaling"] == "weak" and j["config"]["workload"].startswith("tiny")
    r = j["roofline"]
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in r, key
    assert r["bound"] in ("hbm", "tensor") and r["achieved"] > 0 and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3 * max(1.0, r["frac"])
    e = j["e2e"]
    for key in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"):
        assert key in e, key
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert j["gpu_launches"] > 0
    for key in ("sm_mhz", "sm_max_mhz", "reasons"):
        assert key in j["clocks"], key
    c = j["cpu_baseline"]
    for key in ("value", "unit", "cores", "kind", "sample"):
        assert key in c, key
    assert c["kind"] == "oracle" and c["cores"] >= 1


def test_dispatch_combine_line():
    require_gpu()
    j = _line("--no-per-config")
    _check_common(j)
    assert j["unit"] == "tokens/s" and j["roofline"]["bound"] == "hbm" and j["roofline"]["unit"] == "GB/s"
    assert j["gpu_launches"] == 2 * 3  # the fused layout+dispatch kernel and combine, per timed step
    assert j["per_config"] == {}
    assert j["clocks"]["samples"] >= 1 and j["clocks"]["interval_ms"] == 20


def test_dispatch_combine_line_with_the_other_configs():
    """The same line with ds_prefill, mixtral and skewed timed beside the headline
    workload: each entry has its step time, throughput, HBM fractions, per-kernel
    times and the roofline of its dominant kernel (or says why it could not run)."""
    require_gpu()
    j = _line("--no-e2e")
    assert set(j["per_config"]) == {"ds_prefill", "mixtral", "skewed"}
    launches = 2 * 3
    for name, c in j["per_config"].items():
        if "unavailable" in c:
            continue
        for key in ("us_per_step", "tokens_per_s", "step_GBps", "frac_of_measured", "frac_of_8TBps", "kernels",
                    "roofline", "step_kernels"):
            assert key in c, (name, key)
        assert c["us_per_step"] > 0 and c["tokens_per_s"] > 0 and c["steps"] == 3
        r = c["roofline"]
        assert r["bound"] == "hbm" and r["achieved"] > 0 and abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
        assert set(c["kernels"]) == {"layout_dispatch", "combine"}
        launches += c["gpu_launches"]
    assert j["gpu_launches"] == launches


def test_expert_step_line():
    require_gpu()
    j = _line("--expert", "--no-per-config")
    _check_common(j)
    assert j["unit"] == "tokens/s"
