"""dg_run_static: the run that allocates no device memory.

Some callers cannot allocate device memory where they run the GEMM: their
host framework owns and budgets all of it, or they are a plug-in that may not
grow the process's device footprint after start-up.  dg_run_static serves
them by keeping the workspace in one fixed-size device array built into the
library.  These tests check, through the C ABI, that its output matches the
ordinary dg_run (with a caller workspace) on two calls in a row, for several
plans handed the shared array in turn, and that a plan too large for the
array is refused before any GPU work.
"""

import pytest
import torch

from reduce_scatter_gb300 import dg
from tests.gpu_common import TOL, Runner, host_inputs, to_dev

CASES = [
    # (schedule, tp, m, n, k, l, alpha, beta)
    (dg.AG_ROTATING_A, 2, 256, 256, 256, 1, 1.0, 0.0),
    (dg.RS_TILING_A_ROTATING_C, 4, 1024, 1024, 1024, 1, 0.5, 1.0),
    (dg.AG_ROTATING_B, 4, 512, 1024, 512, 2, 1.0, 0.0),
    (dg.RS_TILING_B_ROTATING_C, 2, 392, 776, 320, 2, 0.75, -0.5),
]


def _close(D, ref):
    got, want = D.float(), ref.float()
    assert not torch.isnan(got).any()
    return (got - want).abs().max().item() <= TOL * max(want.abs().max().item(), 1e-30)


@pytest.mark.gpu
def test_static_run_matches_dg_run():
    main = torch.cuda.current_stream()
    copy = torch.cuda.Stream()
    for rounds in range(2):  # hand the shared array from plan to plan, twice over
        for sched, tp, m, n, k, l, alpha, beta in CASES:
            a, b, c = host_inputs(m, n, k, l, seed=40 + sched)
            A, B, C = to_dev(a), to_dev(b), to_dev(c)
            Cin = C if beta else None
            ref, _ = Runner(m, n, k, l, tp, sched, alpha, beta).run(A, B, Cin)
            plan = dg.Plan(m, n, k, l, tp, sched, alpha, beta)
            assert plan.workspace_bytes() <= dg.STATIC_WORKSPACE_BYTES
            for call in range(2):
                D = torch.full((l, m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
                plan.run_static(A, B, Cin, D, main, copy)
                plan.check(None, main)
                assert _close(D, ref), (dg.SCHEDULE_NAMES[sched], tp, rounds, call)


def test_static_run_rejects_plans_larger_than_the_array():
    # 8192 x 8192 x 8192, tp=8: the receive slots alone need 7 x 16 MiB x 8 bytes
    plan = dg.Plan(8192, 8192, 8192, 1, 8, dg.AG_ROTATING_A)
    assert plan.workspace_bytes() > dg.STATIC_WORKSPACE_BYTES
    rc = plan.run_static(16, 16, None, 16, None, None, raise_on_error=False)
    assert rc == dg.ERR_SHAPE
    msg = dg.last_error()
    assert "dg_run_static" in msg and str(dg.STATIC_WORKSPACE_BYTES) in msg
