"""Host-side pieces of bench.py, without a GPU: the clock record taken during
the timed region (parsed from nvidia-smi's CSV, throttle reasons kept) and
the reference arm's JSON line (the oracle timed on the host cores)."""

import io
import json
import os
import sys
from contextlib import redirect_stdout
from types import SimpleNamespace

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


class _FakeSmi:
    """Stands in for the nvidia-smi process: returns fixed CSV lines."""

    def __init__(self, text):
        self.text = text
        self.terminated = False

    def terminate(self):
        self.terminated = True

    def communicate(self, timeout=None):
        return self.text, ""

    def kill(self):
        pass


def _sampler(lines):
    s = bench.ClockSampler(0)
    s.proc = _FakeSmi("\n".join(lines) + "\n")
    return s


def test_clock_record_median_max_and_reasons():
    lines = [
        "0, 2070, 2070, 850.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 2055, 2070, 990.4, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 1010.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "garbage line",
        "0, [N/A], 2070, 1000.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    s = _sampler(lines)
    rec = s.stop()
    assert s.proc.terminated
    assert rec == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "samples": 3,
                   "reasons": ["sw_power_cap"]}


def test_clock_record_flags_slowdowns():
    lines = [
        "0, 1400, 2070, 1300.0, 0x8, Active, Not Active, Not Active, Not Active",
        "0, 1380, 2070, 1300.0, 0x48, Active, Active, Not Active, Not Active",
        "0, 1390, 2070, 1300.0, 0x20, Not Active, Not Active, Active, Not Active",
    ]
    rec = _sampler(lines).stop()
    assert rec["sm_mhz"] == 1390.0 and rec["samples"] == 3
    assert rec["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]


def test_clock_record_absent_without_samples():
    assert _sampler([]).stop() is None
    assert bench.ClockSampler(0).stop() is None  # nvidia-smi never started


def test_reference_line_carries_the_contract_keys(monkeypatch):
    calls = []

    def fake_baseline(kind="streaming"):
        calls.append(kind)
        return {"value": 0.5 + 0.1 * len(calls), "unit": "GB/s", "cores": 1, "kind": "oracle",
                "sample": "every 64th position", "seconds": 2.0, "steps_per_s": 50.0}

    monkeypatch.setattr(bench, "run_cpu_baseline", fake_baseline)
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    out = io.StringIO()
    with redirect_stdout(out):
        bench.run_reference(SimpleNamespace(steps=2, warmup=1))
    line = json.loads(out.getvalue().strip().splitlines()[-1])
    assert len(calls) == 3                       # warm-up step + 2 timed steps
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 1
    assert abs(line["value"] - (0.7 + 0.8) / 2) < 1e-9   # timed steps only
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["metric"] == bench.METRIC and line["higher_is_better"] is True


def test_reference_arm_other_ranks_print_nothing(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    out = io.StringIO()
    with redirect_stdout(out):
        bench.run_reference(SimpleNamespace(steps=2, warmup=1))
    assert out.getvalue() == ""
