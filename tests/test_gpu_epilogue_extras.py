"""The epilogue extras of the scaled fused ops (a per-column bias, fp32 D,
the "avg" reduce op) against the CPU oracle, through ``dg_run_ex``.

Tolerances: bf16 D as everywhere (2e-2 of max|D|).  fp32 D carries only the
fp32 accumulation error: |fl(sum) - sum| <= K * 2^-24 * sum|a b|, about
3e-5 * K/4 for K = 512 uniform [-1, 1) inputs against max|D| of several
sqrt(K/9); 5e-4 of max|D| bounds that with room and still fails a D that was
rounded to bf16 on the way (2^-9 relative)."""

import numpy as np
import pytest
import torch

from oracle import gemm as og
from reduce_scatter_gb300 import dg, synth
from tests.gpu_common import TOL, host_inputs, host_inputs_fp8, to_dev, to_dev_u8

pytestmark = pytest.mark.gpu

SCHEDS = [dg.AG_ROTATING_A, dg.AG_ROTATING_B, dg.RS_TILING_A_ROTATING_C, dg.RS_TILING_B_ROTATING_C]
TOL_F32 = 5e-4


def _bias_bits(n, seed):
    return synth.tensor_bits_np(seed, synth.STREAM_BIAS, (n,), ("uniform", -4.0, 4.0))


def _ok(sched, m, n, k, tp, kq=8):
    # kq: K elements per 16 bytes (8 bf16, 16 fp8), the granule of each rank's K-slab
    if sched in (0, 1, 2) and m % tp:
        return False
    if sched != 2 and n % tp:
        return False
    if sched >= 2 and (k % tp or (k // tp) % kq):
        return False
    return True


def _run(plan, A, B, C, bias, out_dtype, shape, mode=dg.MODE_FUSED):
    plan.set_mode(mode)
    ws = torch.zeros(max(plan.workspace_bytes(), 256), dtype=torch.uint8, device="cuda")
    D = torch.full(shape, float("nan"), dtype=out_dtype, device="cuda")
    main = torch.cuda.current_stream()
    copy = torch.cuda.Stream() if mode != dg.MODE_SERIAL else main
    plan.run_ex(A, B, C, bias, D, ws, main, copy)
    plan.check(ws, main)
    return D


def _err(D, want):
    got = D.float().cpu().numpy().astype(np.float64)
    assert not np.any(np.isnan(got)), "NaN in D"
    return float(np.abs(got - want).max() / max(np.abs(want).max(), 1e-30))


def _want(a, b, c, bias, alpha, beta, sched, tp, op):
    f = og.bf16_bits_to_f64
    return og.fused_gemm(f(a), f(b), f(c) if beta != 0 else None, alpha, beta, P=tp,
                         reduce_op=None if sched <= 1 else op, bias=None if bias is None else f(bias))


@pytest.mark.parametrize("epi", [0, 1, 2, 3, 4])
@pytest.mark.parametrize("sched", SCHEDS, ids=lambda s: dg.SCHEDULE_NAMES[s])
@pytest.mark.parametrize("shape", [(1024, 2048, 512, 2), (392, 776, 320, 2)], ids=lambda s: "x".join(map(str, s)))
def test_bias_f32_out_and_reduce_op_vs_oracle(sched, epi, shape):
    m, n, k, l = shape
    ops = ["sum"] if sched <= 1 else ["sum", "avg"]
    for tp in (1, 2, 8):
        if not _ok(sched, m, n, k, tp):
            continue
        a, b, c = host_inputs(m, n, k, l, seed=300 + tp + 10 * sched + epi)
        bias = _bias_bits(n, 300 + tp)
        A, B, C, Bias = to_dev(a), to_dev(b), to_dev(c), to_dev(bias)
        for op in ops:
            for alpha, beta in [(1.0, 0.0), (0.5, 1.0)]:
                want = _want(a, b, c, bias, alpha, beta, sched, tp, op)
                outs = {}
                for out_type, dt in ((dg.TYPE_BF16, torch.bfloat16), (dg.TYPE_F32, torch.float32)):
                    plan = dg.Plan(m, n, k, l, tp, sched, alpha, beta, out_type=out_type, reduce_op=op)
                    plan.set_option(dg.OPT_EPILOGUE, epi)
                    outs[out_type] = _run(plan, A, B, C if beta else None, Bias, dt, (l, m, n))
                assert _err(outs[dg.TYPE_BF16], want) <= TOL, (tp, op, alpha, beta)
                assert _err(outs[dg.TYPE_F32], want) <= TOL_F32, (tp, op, alpha, beta)
                # one fp32 result in the epilogue, rounded to bf16 (RNE) or stored as is
                assert torch.equal(outs[dg.TYPE_F32].to(torch.bfloat16).view(torch.int16),
                                   outs[dg.TYPE_BF16].view(torch.int16)), (tp, op)


@pytest.mark.parametrize("sched", [dg.RS_TILING_A_ROTATING_C, dg.RS_TILING_B_ROTATING_C],
                         ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_avg_is_sum_over_tp_bit_for_bit(sched):
    # with beta = 0 every term of the mean is the sum's term times 1/tp, a power
    # of two, so the fp32 results differ by exactly that factor
    m, n, k, l, tp = 1024, 1024, 1024, 1, 4
    a, b, _ = host_inputs(m, n, k, l, seed=320 + sched)
    bias = _bias_bits(n, 321)
    A, B, Bias = to_dev(a), to_dev(b), to_dev(bias)
    D = {}
    for op in ("sum", "avg"):
        plan = dg.Plan(m, n, k, l, tp, sched, 0.75, 0.0, out_type="f32", reduce_op=op)
        D[op] = _run(plan, A, B, None, Bias, torch.float32, (l, m, n))
    assert torch.equal(D["avg"] * tp, D["sum"])


@pytest.mark.parametrize("sched", [dg.AG_ROTATING_A, dg.AG_ROTATING_B], ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_allgather_f32_bias_bit_exact_vs_unsharded(sched):
    m, n, k, l = 1024, 1024, 328, 1
    a, b, c = host_inputs(m, n, k, l, seed=330 + sched)
    bias = _bias_bits(n, 331)
    A, B, C, Bias = to_dev(a), to_dev(b), to_dev(c), to_dev(bias)
    ref = _run(dg.Plan(m, n, k, l, 1, sched, 0.5, 1.0, out_type="f32"), A, B, C, Bias, torch.float32, (l, m, n))
    for tp in (2, 4, 8):
        D = _run(dg.Plan(m, n, k, l, tp, sched, 0.5, 1.0, out_type="f32"), A, B, C, Bias, torch.float32,
                 (l, m, n))
        assert torch.equal(D, ref), tp


@pytest.mark.parametrize("sched", [dg.RS_TILING_A_ROTATING_C, dg.RS_TILING_B_ROTATING_C],
                         ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_nonfused_baseline_and_ce_handoff_with_extras(sched):
    # the non-fused baseline and the copy-engine hand-off take the same extras
    m, n, k, l, tp = 1024, 1024, 1024, 2, 4
    a, b, c = host_inputs(m, n, k, l, seed=340 + sched)
    bias = _bias_bits(n, 341)
    A, B, C, Bias = to_dev(a), to_dev(b), to_dev(c), to_dev(bias)
    for op in ("sum", "avg"):
        want = _want(a, b, c, bias, 0.5, 1.0, sched, tp, op)
        plan = dg.Plan(m, n, k, l, tp, sched, 0.5, 1.0, out_type="f32", reduce_op=op)
        Dser = _run(plan, A, B, C, Bias, torch.float32, (l, m, n), mode=dg.MODE_SERIAL)
        assert _err(Dser, want) <= TOL_F32, op
        fused = _run(dg.Plan(m, n, k, l, tp, sched, 0.5, 1.0, out_type="f32", reduce_op=op), A, B, C, Bias,
                     torch.float32, (l, m, n))
        ce = dg.Plan(m, n, k, l, tp, sched, 0.5, 1.0, out_type="f32", reduce_op=op)
        ce.set_option(dg.OPT_RS_CE_PARTIALS, 1)
        Dce = _run(ce, A, B, C, Bias, torch.float32, (l, m, n))
        assert torch.equal(Dce, fused), op


@pytest.mark.parametrize("sched", SCHEDS, ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_fp8_with_bias_and_f32_out(sched):
    m, n, k, l, tp = 1024, 1024, 512, 1, 4
    a, b, c = host_inputs_fp8(m, n, k, l, seed=350 + sched, fmt_a="e4m3", fmt_b="e5m2")
    bias = _bias_bits(n, 351)
    A, B, Bias = to_dev_u8(a), to_dev_u8(b), to_dev(bias)
    sa, sb = 0.5, 0.125
    ops = ["sum"] if sched <= 1 else ["sum", "avg"]
    for op in ops:
        plan = dg.Plan(m, n, k, l, tp, sched, 1.0, 0.0, "e4m3", "e5m2", sa, sb, out_type="f32", reduce_op=op)
        D = _run(plan, A, B, None, Bias, torch.float32, (l, m, n))
        want = og.fused_gemm(og.fp8_bits_to_f64(a, "e4m3"), og.fp8_bits_to_f64(b, "e5m2"), None, sa * sb, 0.0,
                             P=tp, reduce_op=None if sched <= 1 else op, bias=og.bf16_bits_to_f64(bias))
        assert _err(D, want) <= TOL_F32, op


def _fp8_close(got_codes, want_codes, fmt):
    """fp8 results against the oracle's codes: equal, or neighbours (the device
    rounds an fp32 value, the oracle the fp64 one; a value within fp32 error of
    a rounding midpoint may land on either side)."""
    g = og.fp8_bits_to_f64(got_codes, fmt)
    w = og.fp8_bits_to_f64(want_codes, fmt)
    assert not np.any(np.isnan(g))
    vals = np.sort(np.unique(og.fp8_bits_to_f64(np.arange(256), fmt)[np.isfinite(og.fp8_bits_to_f64(np.arange(256), fmt))]))
    gi, wi = np.searchsorted(vals, g), np.searchsorted(vals, w)
    assert np.abs(gi - wi).max() <= 1
    return float(np.mean(got_codes == want_codes))


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("epi", [0, 1, 2, 3, 4])
@pytest.mark.parametrize("sched", SCHEDS, ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_fp8_out_with_result_scale_vs_oracle(sched, epi, fmt):
    m, n, k, l = 392, 776, 320, 2
    ops_ = ["sum"] if sched <= 1 else ["sum", "avg"]
    for tp in (2, 8):
        if not _ok(sched, m, n, k, tp, kq=16):
            continue
        a, b, c = host_inputs_fp8(m, n, k, l, seed=600 + tp + 10 * sched + epi, fmt_a="e4m3", fmt_b="e4m3")
        bias = _bias_bits(n, 601)
        A, B, Bias = to_dev_u8(a), to_dev_u8(b), to_dev(bias)
        for op in ops_:
            rs = 4.0 if fmt == "e4m3" else 0.5
            plan = dg.Plan(m, n, k, l, tp, sched, 1.0, 0.0, "e4m3", "e4m3", 0.5, 0.25, out_type=fmt,
                           reduce_op=op, result_scale=rs)
            plan.set_option(dg.OPT_EPILOGUE, epi)
            ws = torch.zeros(max(plan.workspace_bytes(), 256), dtype=torch.uint8, device="cuda")
            D = torch.full((l, m, n), 0x7F, dtype=torch.uint8, device="cuda")   # NaN codes until written
            main = torch.cuda.current_stream()
            plan.run_ex(A, B, None, Bias, D, ws, main, torch.cuda.Stream())
            plan.check(ws, main)
            want = og.quantize_result(
                og.fused_gemm(og.fp8_bits_to_f64(a, "e4m3"), og.fp8_bits_to_f64(b, "e4m3"), None, 0.125, 0.0,
                              P=tp, reduce_op=None if sched <= 1 else op, bias=og.bf16_bits_to_f64(bias)),
                fmt, rs)
            same = _fp8_close(D.cpu().numpy(), want, fmt)
            assert same >= 0.99, (tp, op, same)


@pytest.mark.parametrize("sched", [dg.RS_TILING_A_ROTATING_C, dg.RS_TILING_B_ROTATING_C],
                         ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_fp8_out_nonfused_baseline(sched):
    m, n, k, l, tp = 1024, 1024, 1024, 1, 4
    a, b, c = host_inputs(m, n, k, l, seed=620 + sched)
    A, B = to_dev(a), to_dev(b)
    plan = dg.Plan(m, n, k, l, tp, sched, 1.0, 0.0, out_type="e4m3", result_scale=2.0)
    plan.set_mode(dg.MODE_SERIAL)
    ws = torch.zeros(plan.workspace_bytes(), dtype=torch.uint8, device="cuda")
    D = torch.full((l, m, n), 0x7F, dtype=torch.uint8, device="cuda")
    main = torch.cuda.current_stream()
    plan.run_ex(A, B, None, None, D, ws, main, main)
    plan.check(ws, main)
    want = og.quantize_result(og.gemm(og.bf16_bits_to_f64(a), og.bf16_bits_to_f64(b), None, 1.0, 0.0), "e4m3", 2.0)
    assert _fp8_close(D.cpu().numpy(), want, "e4m3") >= 0.99
