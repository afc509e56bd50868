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


def test_record_traffic_parses_an_ncu_csv(tmp_path, monkeypatch):
    import bench

    csv = tmp_path / "dram.csv"
    csv.write_text(
        "==PROF== Connected to process 1\n"
        '"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size","Grid Size",'
        '"Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"\n'
        '"0","1","p","h","void other_kernel()","1","7","(1,1,1)","(1,1,1)","0","10.3","s","dram__bytes_read.sum","byte","5"\n'
        '"1","1","p","h","void dg_gemm_kernel<2, 1, 0>(KParams)","1","7","(192, 1, 1)","(152, 1, 1)","0","10.3","s",'
        '"dram__bytes_read.sum","Gbyte","56.70"\n'
        '"1","1","p","h","void dg_gemm_kernel<2, 1, 0>(KParams)","1","7","(192, 1, 1)","(152, 1, 1)","0","10.3","s",'
        '"dram__bytes_write.sum","byte","3,491,002,624"\n'
        '"1","1","p","h","void dg_gemm_kernel<2, 1, 0>(KParams)","1","7","(192, 1, 1)","(152, 1, 1)","0","10.3","s",'
        '"gpu__time_duration.sum","ms","30.5"\n')
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "reduce_scatter_gb300" / "csrc").mkdir(parents=True)
    for name in ("dg_kernel.cuh", "dg_geom.h", "dg.cu"):
        (tmp_path / "reduce_scatter_gb300" / "csrc" / name).write_text(name)
    ent = bench.record_traffic("ag_a_tp8_pr", str(csv), "ncu ...", "note")
    assert ent["dram_bytes_read"] == 56_700_000_000 and ent["dram_bytes_write"] == 3_491_002_624
    assert ent["gpu__time_duration_ns"] == 30_500_000
    assert bench.recorded_traffic("ag_a_tp8_pr") == ent["bytes_per_launch"]
    (tmp_path / "reduce_scatter_gb300" / "csrc" / "dg_geom.h").write_text("changed")
    assert bench.recorded_traffic("ag_a_tp8_pr") is None       # stale once the kernel changes
    bench.record_traffic("ag_a_tp8_pr", str(csv), "ncu ...", "note")
    (tmp_path / "reduce_scatter_gb300" / "csrc" / "dg.cu").write_text("changed")
    assert bench.recorded_traffic("ag_a_tp8_pr") is None       # or the host code that picks its variant


def test_parity_check_of_the_timed_sample():
    import numpy as np

    ent = np.arange(12.0).reshape(3, 4) - 5.0
    assert bench.parity_check(ent + 1e-3, ent, 3, 4)["ok"]
    bad = ent.copy()
    bad[1, 2] += 1.0                                  # one wrong entry
    assert not bench.parity_check(bad, ent, 3, 4)["ok"]
    nan = ent.copy()
    nan[0, 0] = np.nan                                # an unwritten (NaN) entry
    assert not bench.parity_check(nan, ent, 3, 4)["ok"]


def test_parity_sample_spans_every_rank():
    from reduce_scatter_gb300 import configs

    for name, w in configs.WORKLOADS.items():
        ridx, cidx = bench.sample_indices(w, 128, 1024)
        assert ridx.min() == 0 and ridx.max() == w.m - 1 and cidx.min() == 0 and cidx.max() == w.n - 1
        assert len(set((ridx * w.tp) // w.m)) == w.tp, name   # rows from every M-shard
        assert len(set((cidx * w.tp) // w.n)) == w.tp, name   # columns from every N-shard


def test_both_arms_report_the_same_config():
    from reduce_scatter_gb300 import configs

    for name, w in configs.WORKLOADS.items():
        c1 = bench.workload_config(w, 1)
        assert c1["workload"] == name and "parallelism" in c1 and "l2" in c1
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main(["--impl", "reference", "--steps", "1", "--warmup", "1", "--workload", "ag_a_tp2_256"])
    d = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert d["config"] == bench.workload_config(configs.WORKLOADS["ag_a_tp2_256"], 1)
