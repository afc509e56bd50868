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


def test_fp8_decode_matches_torch_for_every_code():
    import torch
    codes = np.arange(256, dtype=np.uint8)
    for fmt, tdt in (("e4m3", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2)):
        ours = og.fp8_bits_to_f64(codes, fmt)
        theirs = torch.from_numpy(codes).view(tdt).to(torch.float64).numpy()
        assert np.array_equal(np.isnan(ours), np.isnan(theirs))
        ok = ~np.isnan(ours)
        assert np.array_equal(ours[ok], theirs[ok])


def test_fp8_format_facts():
    # OCP 8-bit floating point formats: largest finite, one, smallest subnormal
    e4 = og.fp8_bits_to_f64(np.array([0x7E, 0x38, 0x01, 0x08, 0xFE, 0x7F]), "e4m3")
    assert e4[:5].tolist() == [448.0, 1.0, 2.0 ** -9, 2.0 ** -6, -448.0] and np.isnan(e4[5])
    e5 = og.fp8_bits_to_f64(np.array([0x7B, 0x3C, 0x01, 0x04, 0x7C]), "e5m2")
    assert e5.tolist() == [57344.0, 1.0, 2.0 ** -16, 2.0 ** -14, np.inf]


def test_scaled_gemm_pins():
    # brute force with integer inputs and power-of-two scales: exact
    L, M, N, K = 2, 3, 4, 5
    A = pc._int_valued(1, 1, (L, M, K))
    B = pc._int_valued(1, 2, (L, N, K))
    C = pc._int_valued(1, 3, (L, M, N))
    got = og.scaled_gemm(A, B, C, 0.5, 2.0, 4.0, 0.25)
    want = pc.brute_gemm(A, B, C, 0.5, 2.0)  # 0.5 * 4 * 0.25 = 0.5
    assert np.array_equal(got, want)
    # all ones: D = K * alpha * scale_a * scale_b
    ones_a, ones_b = np.ones((1, 3, 64)), np.ones((1, 2, 64))
    assert np.all(og.scaled_gemm(ones_a, ones_b, None, 1.0, 0.0, 3.0, 0.5) == 64 * 1.5)


def test_bias_and_reduce_op_brute_force():
    pc.check_bias_reduce_brute_force(og.fused_gemm)


def test_bias_and_reduce_op_closed_forms():
    pc.check_bias_reduce_closed_forms(og.fused_gemm)


def test_every_schedule_with_bias_and_reduce_op():
    pc.check_schedule_bias_reduce(osch.run_schedule, og.fused_gemm, osch.SCHEDULES)


def test_fused_sampled_entries_match_full():
    # the sampled form agrees with the pinned full form (integer inputs: exact)
    A = pc._int_valued(4, 1, (1, 40, 24))[0]
    B = pc._int_valued(4, 2, (1, 30, 24))[0]
    C = pc._int_valued(4, 3, (1, 40, 30))[0]
    bias = pc._int_valued(4, 4, (30,))
    rows, cols = np.array([0, 7, 39]), np.array([1, 29, 5])
    for op, P in ((None, 1), ("sum", 4), ("avg", 4)):
        full = og.fused_gemm(A[None], B[None], C[None], 0.5, 1.0, P=P, reduce_op=op, bias=bias)[0]
        blk = og.fused_gemm_entries(A[rows], B[cols], C[np.ix_(rows, cols)], 0.5, 1.0, P=P, reduce_op=op,
                                    bias_cols=bias[cols])
        assert np.array_equal(blk, full[np.ix_(rows, cols)]), op


def test_fp8_result_encoding():
    import torch
    for fmt, tdt, top in (("e4m3", getattr(torch, "float8_e4m3fn", None), 448.0),
                          ("e5m2", getattr(torch, "float8_e5m2", None), 57344.0)):
        codes = np.arange(256)
        vals = og.fp8_bits_to_f64(codes, fmt)
        fin = np.isfinite(vals)
        # every finite code round-trips (the sign of zero included)
        assert np.array_equal(og.f64_to_fp8_bits(vals[fin], fmt), codes[fin].astype(np.uint8))
        # midpoints between neighbouring positive codes go to the even code
        pos = np.sort(vals[(codes < 128) & fin])
        mids = (pos[:-1] + pos[1:]) / 2
        got = og.f64_to_fp8_bits(mids, fmt)
        lo_code = og.f64_to_fp8_bits(pos[:-1], fmt)
        want = np.where(lo_code % 2 == 0, lo_code, lo_code + 1)
        assert np.array_equal(got, want.astype(np.uint8))
        # just off the midpoints: the nearer code
        assert np.array_equal(og.f64_to_fp8_bits(mids * (1 - 1e-9), fmt), lo_code)
        assert np.array_equal(og.f64_to_fp8_bits(mids * (1 + 1e-9), fmt), (lo_code + 1).astype(np.uint8))
        # saturation at the largest finite magnitude, both signs
        assert og.fp8_bits_to_f64(og.f64_to_fp8_bits(np.array([1e30, -1e30, top * 1.01]), fmt), fmt).tolist() == \
            [top, -top, top]
        # against torch's own float32 -> fp8 conversion on values inside the range
        if tdt is not None:
            x = (np.random.default_rng(5).standard_normal(20000) * top / 8).astype(np.float32)
            x = x[np.abs(x) < top]
            t = torch.from_numpy(x).to(tdt).view(torch.uint8).numpy()
            assert np.array_equal(og.f64_to_fp8_bits(x.astype(np.float64), fmt), t)
    # the result scale multiplies before rounding
    assert og.quantize_result(np.array([1.0, 3.0]), "e4m3", 0.5).tolist() == \
        og.f64_to_fp8_bits(np.array([0.5, 1.5]), "e4m3").tolist()


def _torch_bf16_to_f64(codes):
    import torch

    t = torch.from_numpy(np.asarray(codes, dtype=np.uint16).view(np.int16).copy()).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def test_bf16_decode_matches_the_format_and_torch():
    # every oracle input passes through this widening
    pc.check_bf16_decode(og.bf16_bits_to_f64, _torch_bf16_to_f64)
