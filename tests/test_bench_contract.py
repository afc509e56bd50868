"""bench.py's reference arm (the CPU oracle) prints one JSON line with the
contract's keys; runs on CPU."""

import io
import json
from contextlib import redirect_stdout

import bench


def test_reference_arm_line():
    buf = io.StringIO()
    with redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--steps", "1", "--warmup", "1", "--workload", "ag_a_tp2_256"])
    assert rc == 0
    lines = [l for l in buf.getvalue().splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s"
    assert d["higher_is_better"] is True and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"] == "ag_a_tp2_256"


def test_default_workload_is_the_tp8_run():
    args = bench.parse_args([])
    assert args.workload == "ag_a_tp8_pr" and args.gpus == 1 and args.warmup >= 3
