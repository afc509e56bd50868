"""The command-line runner: its flags on the CPU, and one small run on the GPU."""

import subprocess
import sys

import pytest

from reduce_scatter_gb300 import __main__ as cli


def test_flags_follow_the_example():
    a = cli.parse([])
    assert (a.m, a.n, a.k, a.l) == (16384, 106496, 16384, 1)
    assert (a.alpha, a.beta, a.iterations, a.warmup_iterations, a.eps) == (1.0, 0.0, 100, 10, 0.0)
    assert (a.tp, a.schedule) == (8, "AllGather1D_TilingCD_RotatingA")
    a = cli.parse(["--m=256", "--n=512", "--k=128", "--l=2", "--alpha=0.5", "--beta=1", "--iterations=3",
                   "--warmup-iterations=1", "--eps=0.01", "--tp=2", "--schedule=ReduceScatter1D_TilingB_RotatingC"])
    assert (a.m, a.n, a.k, a.l, a.alpha, a.beta, a.iterations, a.warmup_iterations, a.eps, a.tp) == \
        (256, 512, 128, 2, 0.5, 1.0, 3, 1, 0.01, 2)
    assert cli.parse(["--dist=normal:0:0.02"]).dist == ("normal", 0.0, 0.02)
    assert cli.parse([]).dist == ("uniform", -1.0, 1.0) and cli.parse([]).mode == "fused"
    for bad in (["--m=0"], ["--iterations=0"], ["--eps=-1"], ["--tp=3"], ["--schedule=Nope"], ["--mode=x"],
                ["--dist=uniform:1:0"], ["--dist=normal:0:0"], ["--dist=poisson:1:2"], ["--dist=1:2"]):
        with pytest.raises(SystemExit):
            cli.parse(bad)


@pytest.mark.gpu
@pytest.mark.parametrize("schedule,eps,mode", [("AllGather1D_TilingCD_RotatingA", "0", "fused"),
                                               ("AllGather1D_TilingCD_RotatingB", "0", "gemm_only"),
                                               ("ReduceScatter1D_TilingA_RotatingC", "0.02", "fused"),
                                               ("ReduceScatter1D_TilingB_RotatingC", "0.02", "serial")])
def test_small_run_passes(schedule, eps, mode):
    out = subprocess.run([sys.executable, "-m", "reduce_scatter_gb300", "--m=2048", "--n=2048", "--k=1024",
                          "--tp=4", f"--schedule={schedule}", "--iterations=3", "--warmup-iterations=1",
                          f"--eps={eps}", "--beta=1", f"--mode={mode}", "--dist=normal:0:1"],
                         capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stdout + out.stderr
    assert f"Disposition (eps: {float(eps):g}): Passed" in out.stdout
    assert "Avg runtime:" in out.stdout and "TFLOPS:" in out.stdout
