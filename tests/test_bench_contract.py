"""The JSON line of bench.py's CPU reference arm (the oracle timed on the host
cores) and the argument rules of the bench, on CPU."""
import io
import json
import os
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _reference_line(workload="tiny", rows=2):
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.reference(bench.parse_args(["--impl", "reference", "--workload", workload,
                                          "--steps", "1", "--warmup", "3",
                                          "--ref-rows-per-head", str(rows)]))
    lines = [l for l in buf.getvalue().splitlines() if l.strip()]
    assert len(lines) == 1, lines
    return json.loads(lines[0])


def test_reference_line_carries_the_contract_fields():
    d = _reference_line()
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 3
    assert d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["vs_baseline"] is None
    assert d["dtype"] == "f64" and d["data"] == "synthetic"
    assert d["config"]["workload"] and d["config"]["d"] == 64
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert cb["unit"] == d["unit"] and "rows per head" in cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_sample_scales_with_rows():
    # the FLOPs of a step follow the sampled rows: more rows, more work
    small = _reference_line(rows=1)["cpu_baseline"]["sample"]
    large = _reference_line(rows=4)["cpu_baseline"]["sample"]
    flops = lambda s: float(s.split("rows, ")[1].split(" FLOPs")[0])
    assert flops(large) > flops(small) > 0


@pytest.mark.parametrize("argv", [["--warmup", "2"], ["--steps", "0"]])
def test_bench_rejects_short_runs(argv):
    with pytest.raises(SystemExit):
        bench.parse_args(argv)


def test_bench_defaults_are_one_gpu_and_a_short_run():
    a = bench.parse_args([])
    assert a.gpus == 1 and a.impl == "native" and a.workload == "ragged"
    assert a.warmup >= 3 and a.steps >= 1
