"""The seeded random sweep draws only configurations the planner accepts: every
case of the GPU sweep (and of its wider seeds) builds a plan and sets its
options without a GPU, so a failure on the GPU is a wrong result, never a
rejected draw."""

import pytest

from reduce_scatter_gb300 import dg
from tests.test_gpu_random_sweep import TCODE, _case, _medium_case

OUT_KINDS = ["bf16", "f32", "e4m3", "e5m2"]


def _plan_with(sched, tp, m, n, k, l, ta, tb, alpha, beta, sa, sb, opts, **kw):
    plan = dg.Plan(m, n, k, l, tp, sched, alpha, beta, TCODE[ta], TCODE[tb], sa, sb, **kw)
    for o, v in opts.items():
        plan.set_option(o, v)
    assert plan.workspace_bytes() >= 0
    return plan


@pytest.mark.parametrize("block", range(8))
def test_small_cases_are_accepted(block):
    # the GPU sweep's seeds (0-47, 500-531, 900-923) and the wider ones
    for i in range(block * 300, (block + 1) * 300):
        sched, tp, m, n, k, l, ta, tb, alpha, beta, sa, sb, opts = _case(i)
        _plan_with(sched, tp, m, n, k, l, ta, tb, alpha, beta, sa, sb, opts)
        _plan_with(sched, tp, m, n, k, l, ta, tb, alpha, beta, sa, sb, opts, out_type=OUT_KINDS[i % 4],
                   reduce_op="avg" if sched >= 2 and i % 2 else "sum", result_scale=1.0)


def test_medium_cases_are_accepted():
    for i in range(300):
        _, sched, tp, m, n, k, l, alpha, beta, opts = _medium_case(i)
        _plan_with(sched, tp, m, n, k, l, "bf16", "bf16", alpha, beta, 1.0, 1.0, opts)
