"""Plant plausible mistakes in copies of the oracle (on the CPU) and check
that the pins catch every one of them."""

import numpy as np
import pytest

from oracle import gemm as og
from oracle import schedules as osch
from tests import pin_checks as pc


def _fails(fn, *args):
    try:
        fn(*args)
    except AssertionError:
        return True
    return False


def gemm_drop_beta(A, B, C, alpha, beta):
    return og.gemm(A, B, C, alpha, 0.0)


def gemm_no_transpose(A, B, C, alpha, beta):
    # treats the stored (N, K) B as (K, N) when it can
    L, M, K = A.shape
    Bt = np.reshape(B, (B.shape[0], K, -1)) if B.size == L * K * B.shape[1] else B
    D = alpha * np.matmul(A, Bt)
    return D + (beta * C if beta != 0 else 0)


def gemm_beta_on_alpha(A, B, C, alpha, beta):
    D = np.matmul(A, np.swapaxes(B, 1, 2))
    return alpha * (D + (beta * C if beta != 0 else 0))


def gemm_half_k(A, B, C, alpha, beta):
    K = A.shape[2]
    h = max(1, K // 2)
    return og.gemm(A[:, :, :h], B[:, :, :h], C, alpha, beta)


def gemm_reads_c_when_beta0(A, B, C, alpha, beta):
    D = alpha * np.matmul(A, np.swapaxes(B, 1, 2))
    return D + (beta * C if C is not None else 0)


GEMM_MUTANTS = [gemm_drop_beta, gemm_no_transpose, gemm_beta_on_alpha, gemm_half_k,
                gemm_reads_c_when_beta0]


@pytest.mark.parametrize("mutant", GEMM_MUTANTS, ids=lambda f: f.__name__)
def test_gemm_mutants_caught(mutant):
    checks = [pc.check_brute_force_exact, pc.check_brute_force_random, pc.check_closed_forms,
              pc.check_printed_mean]
    assert any(_fails(c, mutant) for c in checks)


def _rs_beta_every_step(sched, A, B, C, alpha, beta, P):
    if sched not in (osch.RS_TILING_A_ROTATING_C, osch.RS_TILING_B_ROTATING_C):
        return osch.run_schedule(sched, A, B, C, alpha, beta, P)
    # re-adds beta*C at every hop of the rotating partial
    D = osch.run_schedule(sched, A, B, C, alpha, beta, P)
    return D + (P - 1) * beta * np.asarray(C, np.float64) if beta != 0 else D


def _ag_b_wrong_cols(sched, A, B, C, alpha, beta, P):
    if sched != osch.AG_ROTATING_B or P == 1:
        return osch.run_schedule(sched, A, B, C, alpha, beta, P)
    D = osch.run_schedule(sched, A, B, C, alpha, beta, P)
    n = D.shape[2] // P
    return np.concatenate([D[:, :, n:], D[:, :, :n]], axis=2)  # slabs written to the wrong place


def _rs_drops_last_rank(sched, A, B, C, alpha, beta, P):
    if sched not in (osch.RS_TILING_A_ROTATING_C,) or P == 1:
        return osch.run_schedule(sched, A, B, C, alpha, beta, P)
    k = A.shape[2] // P
    A2 = np.array(A, np.float64)
    A2[:, :, (P - 1) * k:] = 0.0
    return osch.run_schedule(sched, A2, B, C, alpha, beta, P)


@pytest.mark.parametrize("mutant", [_rs_beta_every_step, _ag_b_wrong_cols, _rs_drops_last_rank],
                         ids=lambda f: f.__name__)
def test_schedule_mutants_caught(mutant):
    assert _fails(pc.check_schedule_invariance, mutant, og.gemm, osch.SCHEDULES)


def _slab_ag_not_local_first(sched, P, r, s):
    if sched in (osch.AG_ROTATING_A, osch.AG_ROTATING_B):
        return (r + s + 1) % P
    return osch.slab_index(sched, P, r, s)


def _slab_rs_wrong_ring(sched, P, r, s):
    if sched in (osch.RS_TILING_A_ROTATING_C, osch.RS_TILING_B_ROTATING_C):
        return (r - s - 1) % P  # partial hops to r+1: owner still last, but not the ring the pages use
    return osch.slab_index(sched, P, r, s)


def _slab_rs_owner_first(sched, P, r, s):
    if sched in (osch.RS_TILING_A_ROTATING_C, osch.RS_TILING_B_ROTATING_C):
        return (r + s) % P
    return osch.slab_index(sched, P, r, s)


@pytest.mark.parametrize("mutant", [_slab_ag_not_local_first, _slab_rs_wrong_ring, _slab_rs_owner_first],
                         ids=lambda f: f.__name__)
def test_rotation_mutants_caught(mutant):
    def blocks(sched, m, n, k, P, r, s):
        return osch.step_blocks(sched, m, n, k, P, r, s)
    assert _fails(pc.check_rotation_tables, mutant, blocks, osch.SCHEDULES)


def test_local_size_mutant_caught():
    def wrong(sched, m, n, k, l, P):
        return (m // P, n, k // P, l)
    assert _fails(pc.check_printed_local_sizes, wrong, osch.AG_ROTATING_A)


def test_scaled_gemm_mutant_caught():
    def drops_scale_b(A, B, C, alpha, beta, sa, sb):
        return og.scaled_gemm(A, B, C, alpha, beta, sa, 1.0)
    ones_a, ones_b = np.ones((1, 3, 64)), np.ones((1, 2, 64))
    assert not np.all(drops_scale_b(ones_a, ones_b, None, 1.0, 0.0, 3.0, 0.5) == 64 * 1.5)


# ------------------------------------------------ bias and the reduce op

def _fused_bias_once(A, B, C, alpha, beta, *, P=1, reduce_op=None, bias=None):
    # the reduce-scatter bias added once instead of once per rank
    return og.fused_gemm(A, B, C, alpha, beta, P=P, reduce_op=reduce_op, bias=None) + \
        (0.0 if bias is None else (bias / P if reduce_op == "avg" else bias))


def _fused_drops_bias(A, B, C, alpha, beta, *, P=1, reduce_op=None, bias=None):
    return og.fused_gemm(A, B, C, alpha, beta, P=P, reduce_op=reduce_op, bias=None)


def _fused_avg_divides_c(A, B, C, alpha, beta, *, P=1, reduce_op=None, bias=None):
    D = og.fused_gemm(A, B, C, alpha, 0.0, P=P, reduce_op=reduce_op, bias=bias)
    if beta != 0.0:
        D = D + (beta * C / P if reduce_op == "avg" else beta * C)
    return D


def _fused_avg_ignored(A, B, C, alpha, beta, *, P=1, reduce_op=None, bias=None):
    return og.fused_gemm(A, B, C, alpha, beta, P=P, reduce_op="sum" if reduce_op == "avg" else reduce_op,
                         bias=bias)


@pytest.mark.parametrize("mutant", [_fused_bias_once, _fused_drops_bias, _fused_avg_divides_c, _fused_avg_ignored],
                         ids=lambda f: f.__name__)
def test_fused_gemm_mutants_caught(mutant):
    checks = [pc.check_bias_reduce_brute_force, pc.check_bias_reduce_closed_forms]
    assert any(_fails(c, mutant) for c in checks)


def _sched_bias_first_step_only(sched, A, B, C, alpha, beta, P, *, bias=None, reduce_op="sum"):
    # the rotating partial picks up the bias at step 0 only
    if sched in (osch.RS_TILING_A_ROTATING_C, osch.RS_TILING_B_ROTATING_C) and bias is not None:
        D = osch.run_schedule(sched, A, B, C, alpha, beta, P, reduce_op=reduce_op)
        return D + (bias / P if reduce_op == "avg" else bias)
    return osch.run_schedule(sched, A, B, C, alpha, beta, P, bias=bias, reduce_op=reduce_op)


def _sched_avg_weights_product_only(sched, A, B, C, alpha, beta, P, *, bias=None, reduce_op="sum"):
    # avg divides the products but not the bias copies
    if sched in (osch.RS_TILING_A_ROTATING_C, osch.RS_TILING_B_ROTATING_C) and reduce_op == "avg" and bias is not None:
        D = osch.run_schedule(sched, A, B, C, alpha, beta, P, reduce_op="avg")
        return D + P * bias
    return osch.run_schedule(sched, A, B, C, alpha, beta, P, bias=bias, reduce_op=reduce_op)


@pytest.mark.parametrize("mutant", [_sched_bias_first_step_only, _sched_avg_weights_product_only],
                         ids=lambda f: f.__name__)
def test_schedule_bias_mutants_caught(mutant):
    assert _fails(pc.check_schedule_bias_reduce, mutant, og.fused_gemm, osch.SCHEDULES)


def test_fp8_result_encoding_mutants_caught():
    def truncates(x, fmt):                      # rounds toward zero instead of to nearest
        codes = np.arange(128)
        vals = og.fp8_bits_to_f64(codes, fmt)
        ok = np.isfinite(vals)
        pv, pc = vals[ok], codes[ok]
        a = np.abs(np.asarray(x, np.float64))
        i = np.clip(np.searchsorted(pv, a, side="right") - 1, 0, len(pv) - 1)
        return (pc[i] | (np.signbit(x).astype(np.int64) << 7)).astype(np.uint8)

    orig = og.f64_to_fp8_bits

    def ties_away(x, fmt):                      # ties away from zero instead of to even
        out = orig(x, fmt).astype(np.int64)
        codes = np.arange(128)
        vals = og.fp8_bits_to_f64(codes, fmt)
        pv = np.sort(vals[np.isfinite(vals)])
        mids = (pv[:-1] + pv[1:]) / 2
        a = np.abs(np.asarray(x, np.float64))
        hit = np.isin(a, mids)
        up = orig(np.nextafter(a, np.inf), fmt).astype(np.int64) | (np.signbit(x).astype(np.int64) << 7)
        return np.where(hit, up, out).astype(np.uint8)

    for mutant in (truncates, ties_away):
        og.f64_to_fp8_bits = mutant
        try:
            assert _fails(_pins_fp8_result)
        finally:
            og.f64_to_fp8_bits = orig


def _pins_fp8_result():
    from tests import test_oracle_pins as tp
    tp.test_fp8_result_encoding()


# ------------------------------------------------------- bf16 input decoding

def _bf16_shift_15(bits):
    u = np.asarray(bits).astype(np.uint16).astype(np.uint32) << np.uint32(15)
    return u.view(np.float32).astype(np.float64)


def _bf16_as_fp16(bits):
    # reads the 16-bit patterns as IEEE half precision
    return np.asarray(bits).astype(np.uint16).view(np.float16).astype(np.float64)


def _bf16_sign_extended(bits):
    # widens int16 patterns through a signed 32-bit integer, then drops the sign
    v = np.asarray(bits).astype(np.int16).astype(np.int32)
    return (np.abs(v).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def _bf16_truncates_mantissa(bits):
    # keeps only 6 of the 7 stored mantissa bits
    u = (np.asarray(bits).astype(np.uint16).astype(np.uint32) & np.uint32(0xFFFE)) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


@pytest.mark.parametrize("mutant", [_bf16_shift_15, _bf16_as_fp16, _bf16_sign_extended, _bf16_truncates_mantissa],
                         ids=lambda f: f.__name__)
def test_bf16_decode_mutants_caught(mutant):
    from tests.test_oracle_pins import _torch_bf16_to_f64
    assert _fails(pc.check_bf16_decode, mutant, _torch_bf16_to_f64)
