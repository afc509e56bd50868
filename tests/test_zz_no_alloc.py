"""dg_run_static: the run that allocates no device memory.

Some callers cannot allocate device memory where they run the GEMM: their
host framework owns and budgets all of it, or they are a plug-in that may not
grow the process's device footprint after start-up.  dg_run_static serves
them by keeping the workspace in one fixed-size device array built into the
library.  These tests check, through the C ABI:

* its D is bit-for-bit the D of the ordinary dg_run (with a caller
  workspace) on two calls in a row, for several plans handed the shared
  array in turn (same kernel, same K order), and within tolerance of the CPU
  oracle;
* a warmed-up call leaves the device's free memory unchanged;
* a ready-flag wait that runs out is reported by dg_check(plan, NULL, ...),
  and the next call is correct;
* a plan too large for the array is refused before any GPU work.

This file is named so that pytest collects it last.
"""

import pytest
import torch

from reduce_scatter_gb300 import dg
from tests.gpu_common import TOL, Runner, host_inputs, oracle_full, rel_err, to_dev

CASES = [
    # (schedule, tp, m, n, k, l, alpha, beta)
    (dg.AG_ROTATING_A, 2, 256, 256, 256, 1, 1.0, 0.0),
    (dg.RS_TILING_A_ROTATING_C, 4, 1024, 1024, 1024, 1, 0.5, 1.0),
    (dg.AG_ROTATING_B, 4, 512, 1024, 512, 2, 1.0, 0.0),
    (dg.RS_TILING_B_ROTATING_C, 2, 392, 776, 320, 2, 0.75, -0.5),
]


def _nan_d(shape):
    return torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")


@pytest.mark.gpu
def test_static_run_matches_dg_run_and_the_oracle():
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
                D = _nan_d((l, m, n))  # tiles never written stay NaN and fail
                plan.run_static(A, B, Cin, D, main, copy)
                assert plan.check(None, main) == dg.OK
                assert torch.equal(D.view(torch.int16), ref.view(torch.int16)), \
                    (dg.SCHEDULE_NAMES[sched], tp, rounds, call)
            if rounds == 0:
                assert rel_err(D, oracle_full(a, b, c, alpha, beta)) <= TOL, dg.SCHEDULE_NAMES[sched]


@pytest.mark.gpu
def test_static_run_allocates_no_device_memory():
    sched, tp, m, n, k, l, alpha, beta = CASES[1]
    a, b, c = host_inputs(m, n, k, l, seed=44)
    A, B, C = to_dev(a), to_dev(b), to_dev(c)
    D = _nan_d((l, m, n))
    main = torch.cuda.current_stream()
    copy = torch.cuda.Stream()
    plan = dg.Plan(m, n, k, l, tp, sched, alpha, beta)
    plan.run_static(A, B, C, D, main, copy)   # warm: address lookup, kernel attributes, streams
    plan.check(None, main)
    torch.cuda.synchronize()
    same = False
    for _ in range(3):  # a free-memory reading can move with unrelated activity: retry
        free0, _ = torch.cuda.mem_get_info()
        plan.run_static(A, B, C, D, main, copy)
        plan.check(None, main)
        torch.cuda.synchronize()
        free1, _ = torch.cuda.mem_get_info()
        if free1 == free0:
            same = True
            break
    assert same, (free0, free1)


@pytest.mark.gpu
def test_static_run_reports_a_timeout_then_recovers():
    m, n, k, l, tp = 512, 512, 256, 1, 2
    a, b, c = host_inputs(m, n, k, l, seed=45)
    A, B = to_dev(a), to_dev(b)
    main = torch.cuda.current_stream()
    copy = torch.cuda.Stream()
    plan = dg.Plan(m, n, k, l, tp, dg.AG_ROTATING_A)
    plan.set_option(dg.OPT_TIMEOUT_MS, 100)
    D = _nan_d((l, m, n))
    plan.run_static(A, B, None, D, main, copy)
    assert plan.check(None, main) == dg.OK
    plan.set_option(dg.OPT_FAULT_SKIP_FLAG, 0)  # the first ready flag is never written
    plan.run_static(A, B, None, D, main, copy)
    rc = plan.check(None, main, raise_on_error=False)
    assert rc == dg.ERR_TIMEOUT and "flag 0" in dg.last_error()
    plan.set_option(dg.OPT_FAULT_SKIP_FLAG, -1)
    D = _nan_d((l, m, n))
    plan.run_static(A, B, None, D, main, copy)
    assert plan.check(None, main) == dg.OK
    assert rel_err(D, oracle_full(a, b, c, 1.0, 0.0)) <= TOL


def test_static_run_rejects_plans_larger_than_the_array():
    # 8192 x 8192 x 8192, tp=8: the receive slots alone need 7 x 16 MiB x 8 bytes
    plan = dg.Plan(8192, 8192, 8192, 1, 8, dg.AG_ROTATING_A)
    assert plan.workspace_bytes() > dg.STATIC_WORKSPACE_BYTES
    rc = plan.run_static(16, 16, None, 16, None, None, raise_on_error=False)
    assert rc == dg.ERR_SHAPE
    msg = dg.last_error()
    assert "dg_run_static" in msg and str(dg.STATIC_WORKSPACE_BYTES) in msg
