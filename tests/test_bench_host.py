"""Host-side arithmetic of bench.py (no GPU): the algorithmic byte counts that
the roofline numerator uses, against the byte budgets worked out independently
for each configuration in the hot-path scope (packed4096 1914 MB per step,
the adapter-count sweep, the skewed batch, the three decode projections), and
the shape of the reference arm's JSON line."""
import json
import subprocess
import sys
import os

import pytest

import bench
import workloads as wl

MB = 1e6


@pytest.mark.parametrize("spec,want_mb", [
    (lambda: wl.packed4096(), 1914),
    (lambda: wl.sweep(2), 589),
    (lambda: wl.sweep(32), 9429),
    (lambda: wl.skewed(), 2220),
])
def test_step_bytes_match_the_scope_budgets(spec, want_mb):
    s = spec()
    b = bench.step_bytes(s)
    assert abs((b["fwd"] + b["bwd"]) / MB - want_mb) <= 0.005 * want_mb


@pytest.mark.parametrize("i,want_mb", [(0, 8.91), (1, 17.56), (2, 13.89)])
def test_decode_bytes_match_the_scope_budgets(i, want_mb):
    assert abs(bench.decode_bytes(wl.decode(i)) / MB - want_mb) <= 0.01


def test_step_flops_packed4096():
    # 6 flops per (token, rank unit, hidden element) over d_in + d_out: 72.48 GFLOP per step
    assert abs(bench.step_flops(wl.packed4096()) / 1e9 - 72.48) < 0.01


def test_reference_arm_line_shape():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "3", "--ref-tokens-per-adapter", "2"], capture_output=True, text=True,
                         timeout=600, cwd=root)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads([l for l in out.stdout.splitlines() if l.startswith("{")][-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["unit"] == bench.UNIT
    assert line["config"]["workload"] == bench.workload_config(wl.packed4096(), 4096)["workload"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["higher_is_better"] is True
