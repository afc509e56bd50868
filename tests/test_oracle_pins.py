"""The CPU oracle against facts outside itself (brute force, closed forms,
the pages' printed numbers, schedule invariance)."""

import numpy as np

from oracle import gemm as og
from oracle import schedules as osch
from tests import pin_checks as pc


def test_brute_force_exact():
    pc.check_brute_force_exact(og.gemm)


def test_brute_force_random_within_bound():
    pc.check_brute_force_random(og.gemm)


def test_closed_forms():
    pc.check_closed_forms(og.gemm)


def test_printed_blog_mean():
    pc.check_printed_mean(og.gemm)


def test_every_schedule_and_tp_gives_unsharded_d():
    pc.check_schedule_invariance(osch.run_schedule, og.gemm, osch.SCHEDULES)


def test_rotation_tables():
    pc.check_rotation_tables(osch.slab_index, osch.step_blocks, osch.SCHEDULES)


def test_printed_local_problem_sizes():
    pc.check_printed_local_sizes(osch.local_problem, osch.AG_ROTATING_A)


def test_rs_accumulation_order_ends_on_owner():
    for sched in (osch.RS_TILING_A_ROTATING_C, osch.RS_TILING_B_ROTATING_C):
        for P in (2, 4, 8):
            for j in range(P):
                order = osch.rs_accumulation_order(sched, P, j)
                assert order == [(j - 1 - s) % P for s in range(P)]
                assert order[-1] == j


def test_sampled_entries_match_full():
    A = pc._rand(3, 1, (1, 40, 24))[0]
    B = pc._rand(3, 2, (1, 30, 24))[0]
    C = pc._rand(3, 3, (1, 40, 30))[0]
    full = og.gemm(A[None], B[None], C[None], 0.5, 1.0)[0]
    rows, cols = np.array([0, 7, 39]), np.array([1, 29, 5])
    blk = og.gemm_entries(A[rows], B[cols], C[np.ix_(rows, cols)], 0.5, 1.0)
    assert np.array_equal(blk, full[np.ix_(rows, cols)])


def test_flops_matches_printed_tflops():
    import json, os
    with open(os.path.join(pc.GOLDEN, "pr1907_distgemm_printout.json")) as f:
        g = json.load(f)
    for run in g["runs"]:
        m, n, k, l = run["problem"]
        per_gpu = og.flops(m, n, k, l) / (run["avg_runtime_ms"] * 1e-3) / run["tp"] / 1e12
        assert abs(per_gpu - run["tflops_per_gpu"]) < 0.01
