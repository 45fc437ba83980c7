"""The bench's JSON line on a GPU: a short run of the headline workload
(`bench.py --steps 8 --warmup 3 --no-secondary --no-cpu`) prints one line
with the fields the measurement contract asks for, and they are consistent
with each other: the kernel time is the step time, the roofline fraction is
the achieved rate over the peak, the DRAM traffic (when the source it was
taken on is unchanged) sits beside the algorithmic bytes, the end-to-end
figure counts its host copies, and the clocks were sampled."""

import json
import os
import subprocess
import sys

import pytest

from conftest import ROOT

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "8", "--warmup", "3",
                        "--no-secondary", "--no-cpu"], capture_output=True, text=True, cwd=ROOT,
                       timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def test_contract_fields(line):
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "roofline",
              "e2e", "clocks", "gpu_launches"):
        assert k in line, k
    assert line["n_gpus"] == 1 and line["steps"] == 8 and line["warmup"] == 3
    assert line["higher_is_better"] is True and line["scaling"] == "weak"
    assert line["gpu_launches"] == 8
    assert "workload" in line["config"]


def test_value_and_roofline_agree(line):
    T = 8192
    ms = line["ms_per_step"]
    assert line["value"] == pytest.approx(T / (ms * 1e-3), rel=1e-3)
    rf = line["roofline"]
    assert rf["kernel_ms"] <= ms * 1.0001
    assert rf["frac"] == pytest.approx(rf["achieved"] / rf["peak"], rel=1e-3)
    assert 0.2 < rf["frac"] < 1.2
    if rf["traffic"] is not None:
        assert rf["traffic_over_algorithmic"] == pytest.approx(
            rf["traffic"] / rf["algorithmic_bytes"], rel=1e-3)


def test_end_to_end_counts_host_copies(line):
    e2e = line["e2e"]
    assert e2e["h2d_bytes_per_step"] >= 8192 * 8 * 4096 * 2
    assert e2e["d2h_bytes_per_step"] >= 8192 * 8 * 1024 * 2
    assert 0 < e2e["value"] < line["value"]


def test_clocks_sampled(line):
    c = line["clocks"]
    assert c["samples"] >= 1 and c["sm_max_mhz"] > 0 and isinstance(c["reasons"], list)
