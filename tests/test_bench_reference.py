"""bench.py's reference arm (the oracle timed on the host cores) on the CPU,
with a short time budget: it prints one JSON line that keeps the bench
contract (metric, value, unit, steps, the cpu_baseline and e2e objects)."""
import io
import json
import contextlib
import types

import bench


def test_reference_arm_prints_one_contract_line(monkeypatch):
    monkeypatch.setattr(bench, "REFERENCE_BUDGET_S", 1.0)
    args = types.SimpleNamespace(workload="e4m3_verify_512k_stress", steps=2, warmup=1, gpus=1)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(args, 0, 1)
    lines = [l for l in buf.getvalue().splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 1
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["value"] > 0 and d["higher_is_better"] is True
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_is_silent_on_other_ranks():
    args = types.SimpleNamespace(workload="e4m3_verify_512k_stress", steps=1, warmup=0, gpus=2)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(args, 1, 2)
    assert buf.getvalue() == ""
