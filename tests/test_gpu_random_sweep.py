"""A seeded random sweep over the configuration space against the CPU oracle:
schedule, TP, tile configuration, epilogue, middle-step reduction, B
multicast, input type, RS hand-off, batch, alpha / beta / scales and ragged
shapes (within the shape rules)."""

import numpy as np
import pytest

from reduce_scatter_gb300 import dg
from tests.gpu_common import (TOL, Runner, host_inputs, host_inputs_fp8, oracle_fp8, oracle_full, rel_err, to_dev,
                              to_dev_u8)

pytestmark = pytest.mark.gpu

TYPES = [("bf16", "bf16"), ("e4m3", "e4m3"), ("e5m2", "e5m2"), ("e4m3", "e5m2")]
TCODE = {"bf16": dg.TYPE_BF16, "e4m3": dg.TYPE_E4M3, "e5m2": dg.TYPE_E5M2}


def _case(i):
    rng = np.random.default_rng(1000 + i)
    sched = int(rng.integers(0, 4))
    tp = int(rng.choice([1, 2, 4, 8]))
    ta, tb = TYPES[int(rng.integers(0, len(TYPES)))]
    kq = 8 if ta == "bf16" else 16                     # K granule (16-byte rows)
    l = int(rng.integers(1, 4))
    m = int(rng.integers(1, 9)) * 8 * tp if sched in (0, 1, 2) else int(rng.integers(8, 700))
    n = int(rng.integers(1, 13)) * 8 * (tp if sched != 2 else 1)
    if sched >= 2:
        k = int(rng.integers(1, 7)) * kq * tp
    else:
        k = int(rng.integers(1, 50)) * kq
    if sched == 3 and (n // tp) % 8:
        n = 8 * tp * max(1, n // (8 * tp))
    cep = sched >= 2 and tp > 1 and (sched == 2 or (n // tp) % 8 == 0) and bool(rng.integers(0, 2))
    # the reduction may be forced on RS plans only (an AG plan rejects it)
    opts = {dg.OPT_CTA_GROUP: int(rng.integers(1, 3)), dg.OPT_EPILOGUE: int(rng.integers(0, 5)),
            dg.OPT_RS_REDUCE: int(rng.integers(-1, 2 if sched >= 2 else 1)), dg.OPT_MULTICAST: int(rng.integers(-1, 2))}
    if cep:
        opts[dg.OPT_RS_CE_PARTIALS] = 1
    alpha = float(rng.choice([1.0, 0.5, -1.25]))
    beta = float(rng.choice([0.0, 1.0, 0.75]))
    sa, sb = (1.0, 1.0) if ta == "bf16" else (float(rng.choice([1.0, 0.5])), float(rng.choice([1.0, 0.03125])))
    return sched, tp, m, n, k, l, ta, tb, alpha, beta, sa, sb, opts


@pytest.mark.parametrize("i", range(48))
def test_random_configuration(i):
    sched, tp, m, n, k, l, ta, tb, alpha, beta, sa, sb, opts = _case(i)
    if ta == "bf16":
        a, b, c = host_inputs(m, n, k, l, seed=2000 + i)
        A, B = to_dev(a), to_dev(b)
        want = oracle_full(a, b, c, alpha, beta)
    else:
        a, b, c = host_inputs_fp8(m, n, k, l, seed=2000 + i, fmt_a=ta, fmt_b=tb)
        A, B = to_dev_u8(a), to_dev_u8(b)
        want = oracle_fp8(a, b, c, ta, tb, alpha, beta, sa, sb)
    C = to_dev(c)
    r = Runner(m, n, k, l, tp, sched, alpha, beta, options=opts, a_type=TCODE[ta], b_type=TCODE[tb],
               scale_a=sa, scale_b=sb)
    D, _ = r.run(A, B, C if beta else None)
    err = rel_err(D, want)
    assert err <= TOL, (err, sched, tp, m, n, k, l, ta, tb, opts)


@pytest.mark.parametrize("i", range(32))
def test_random_configuration_with_epilogue_extras(i):
    # the same space with a bias, fp32 or bf16 D and, for RS, sum or avg, against the oracle's
    # fused_gemm (the definition of those extras); fp32 D is held to the fp32 tolerance
    import torch

    from oracle import gemm as og
    from reduce_scatter_gb300 import synth
    sched, tp, m, n, k, l, ta, tb, alpha, beta, sa, sb, opts = _case(500 + i)
    rng = np.random.default_rng(7000 + i)
    out_kind = ["bf16", "f32", "e4m3", "e5m2"][int(rng.integers(0, 4))]
    out_f32 = out_kind == "f32"
    op = "avg" if sched >= 2 and rng.integers(0, 2) else "sum"
    bias_bits = synth.tensor_bits_np(3000 + i, synth.STREAM_BIAS, (n,), ("uniform", -4.0, 4.0))
    if ta == "bf16":
        a, b, c = host_inputs(m, n, k, l, seed=3000 + i)
        A, B = to_dev(a), to_dev(b)
        a64, b64 = og.bf16_bits_to_f64(a), og.bf16_bits_to_f64(b)
    else:
        a, b, c = host_inputs_fp8(m, n, k, l, seed=3000 + i, fmt_a=ta, fmt_b=tb)
        A, B = to_dev_u8(a), to_dev_u8(b)
        a64, b64 = og.fp8_bits_to_f64(a, ta), og.fp8_bits_to_f64(b, tb)
    want = og.fused_gemm(a64, b64, og.bf16_bits_to_f64(c) if beta else None, alpha * sa * sb, beta, P=tp,
                         reduce_op=None if sched <= 1 else op, bias=og.bf16_bits_to_f64(bias_bits))
    fp8_out = out_kind in ("e4m3", "e5m2")
    rscale = 1.0 / max(float(np.abs(want).max()), 1e-30) * 64.0 if fp8_out else 1.0   # results well inside the format
    plan = dg.Plan(m, n, k, l, tp, sched, alpha, beta, TCODE[ta], TCODE[tb], sa, sb, out_type=out_kind,
                   reduce_op=op if sched >= 2 else "sum", result_scale=rscale)
    for o, v in opts.items():
        plan.set_option(o, v)
    ws = torch.zeros(max(plan.workspace_bytes(), 256), dtype=torch.uint8, device="cuda")
    if fp8_out:
        D = torch.full((l, m, n), 0x7F, dtype=torch.uint8, device="cuda")
    else:
        D = torch.full((l, m, n), float("nan"), dtype=torch.float32 if out_f32 else torch.bfloat16, device="cuda")
    main = torch.cuda.current_stream()
    plan.run_ex(A, B, to_dev(c) if beta else None, to_dev(bias_bits), D, ws, main, torch.cuda.Stream())
    plan.check(ws, main)
    if fp8_out:
        # codes equal to the oracle's, or neighbours (fp32 against fp64 rounding of a midpoint)
        got = D.cpu().numpy()
        wc = og.quantize_result(want, out_kind, rscale)
        table = og.fp8_bits_to_f64(np.arange(256), out_kind)
        vals = np.sort(np.unique(table[np.isfinite(table)]))
        gv, wv = og.fp8_bits_to_f64(got, out_kind), og.fp8_bits_to_f64(wc, out_kind)
        assert not np.any(np.isnan(gv))
        assert np.abs(np.searchsorted(vals, gv) - np.searchsorted(vals, wv)).max() <= 1, (sched, tp, out_kind)
        return
    err = rel_err(D, want)
    assert err <= (5e-4 if out_f32 else TOL), (err, sched, tp, m, n, k, l, ta, tb, opts, out_f32, op)


@pytest.mark.parametrize("i", range(24))
def test_random_configuration_from_host_buffers(i):
    # the same space through dg_run_host: pinned or pageable host buffers, transfers
    # overlapping the kernel or not, either block order (AG); bit-equal to the run on
    # device buffers
    import torch
    sched, tp, m, n, k, l, ta, tb, alpha, beta, sa, sb, opts = _case(900 + i)
    rng = np.random.default_rng(9000 + i)
    if ta == "bf16":
        a, b, c = host_inputs(m, n, k, l, seed=4000 + i)
        A, B = to_dev(a), to_dev(b)
        in_dt, view = torch.bfloat16, np.int16
    else:
        a, b, c = host_inputs_fp8(m, n, k, l, seed=4000 + i, fmt_a=ta, fmt_b=tb)
        A, B = to_dev_u8(a), to_dev_u8(b)
        in_dt, view = torch.uint8, np.uint8
    C = to_dev(c) if beta else None
    mk = lambda: Runner(m, n, k, l, tp, sched, alpha, beta, options=opts, a_type=TCODE[ta],  # noqa: E731
                        b_type=TCODE[tb], scale_a=sa, scale_b=sb)
    want, _ = mk().run(A, B, C)
    r = mk()
    r.plan.set_option(dg.OPT_HOST_OVERLAP, int(rng.integers(0, 2)))
    if sched <= 1:
        r.plan.set_option(dg.OPT_TILE_ORDER, int(rng.integers(-1, 2)))
    pinned = bool(rng.integers(0, 4))  # mostly pinned
    host = lambda x: (torch.from_numpy(np.ascontiguousarray(x).view(view)).pin_memory() if pinned  # noqa: E731
                      else torch.from_numpy(np.ascontiguousarray(x).view(view)).clone())
    A_h, B_h = host(a), host(b)
    C_h = (torch.from_numpy(c.view(np.int16)).pin_memory() if pinned else torch.from_numpy(c.view(np.int16)).clone()) \
        if beta else None
    D_h = torch.zeros((l, m, n), dtype=torch.int16)
    if pinned:
        D_h = D_h.pin_memory()
    poison = 0xFF if in_dt == torch.uint8 else float("nan")  # NaN in bf16, e4m3 and e5m2
    A2 = torch.full((l, m, k), poison, dtype=in_dt, device="cuda")
    B2 = torch.full((l, n, k), poison, dtype=in_dt, device="cuda")
    C2 = torch.full((l, m, n), float("nan"), dtype=torch.bfloat16, device="cuda") if beta else None
    D2 = torch.full((l, m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
    r.plan.run_host(A_h, B_h, C_h, None, D_h, A2, B2, C2, D2, r.ws, r.main, r.copy)
    r.plan.check(r.ws, r.main)
    assert torch.equal(D_h, want.view(torch.int16).cpu()), (sched, tp, m, n, k, l, ta, tb, opts, pinned)


def _medium_case(i):
    rng = np.random.default_rng(6000 + i)
    sched = int(rng.integers(0, 4))
    tp = int(rng.choice([2, 4, 8]))
    m = int(rng.integers(2048 // (8 * tp), 8192 // (8 * tp) + 1)) * 8 * tp
    n = int(rng.integers(2048 // (8 * tp), 8192 // (8 * tp) + 1)) * 8 * tp
    k = int(rng.integers(512 // (16 * tp), 4096 // (16 * tp) + 1)) * 16 * tp
    l = int(rng.integers(1, 3))
    alpha, beta = float(rng.choice([1.0, 0.5])), float(rng.choice([0.0, 1.0]))
    opts = {dg.OPT_CTA_GROUP: int(rng.integers(1, 3)), dg.OPT_WAVE_SYNC: int(rng.integers(-1, 2)),
            dg.OPT_MULTICAST: int(rng.integers(-1, 2)), dg.OPT_EPILOGUE: int(rng.integers(0, 5))}
    if sched >= 2:
        opts[dg.OPT_RS_REDUCE] = int(rng.integers(-1, 2))
        if rng.integers(0, 2):
            opts[dg.OPT_RS_CE_PARTIALS] = 1
    return rng, sched, tp, m, n, k, l, alpha, beta, opts


@pytest.mark.parametrize("i", range(24))
def test_random_medium_configuration(i):
    # shapes of 2048-8192 rows and columns: many waves of the persistent grid, the
    # wave gate in any setting, the copy-engine hand-off; sampled entries against the
    # oracle and, for AG, the same bits as tp = 1
    import torch

    from oracle import gemm as og
    from reduce_scatter_gb300 import synth
    rng, sched, tp, m, n, k, l, alpha, beta, opts = _medium_case(i)
    seed, dist = 100 + i, ("normal", 0.0, 1.0)
    A = synth.tensor_bits_torch(seed, synth.STREAM_A, (l, m, k), dist, device="cuda").view(torch.bfloat16)
    B = synth.tensor_bits_torch(seed, synth.STREAM_B, (l, n, k), dist, device="cuda").view(torch.bfloat16)
    C = synth.tensor_bits_torch(seed, synth.STREAM_C, (l, m, n), dist, device="cuda").view(torch.bfloat16) \
        if beta else None
    D, _ = Runner(m, n, k, l, tp, sched, alpha, beta, options=opts).run(A, B, C)
    assert not torch.isnan(D).any()
    rows = np.unique(rng.integers(0, l * m, 24))
    cols = np.unique(rng.integers(0, n, 24))
    Dh = D.view(l * m, n)[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()].float().cpu().numpy()
    for b in range(l):
        rs = rows[(rows >= b * m) & (rows < (b + 1) * m)]
        if len(rs) == 0:
            continue
        a = og.bf16_bits_to_f64(synth.rows_bits_np(seed, synth.STREAM_A, (l * m, k), rs, dist))
        bb = og.bf16_bits_to_f64(synth.rows_bits_np(seed, synth.STREAM_B, (l * n, k), cols + b * n, dist))
        c = og.bf16_bits_to_f64(synth.rows_bits_np(seed, synth.STREAM_C, (l * m, n), rs, dist)[:, cols]) \
            if beta else None
        want = og.gemm_entries(a, bb, c, alpha, beta)
        got = Dh[np.isin(rows, rs)].astype(np.float64)
        assert np.abs(got - want).max() / np.abs(want).max() <= TOL, (sched, tp, m, n, k, l, opts)
    if sched <= 1:
        ref, _ = Runner(m, n, k, l, 1, sched, alpha, beta, options={dg.OPT_CTA_GROUP: opts[dg.OPT_CTA_GROUP]}).run(
            A, B, C)
        assert torch.equal(D.view(torch.int16), ref.view(torch.int16))
