"""ReduceScatter with the rotating partial handed from rank to rank by
copy-engine transfers (DG_OPT_RS_CE_PARTIALS): against the oracle, bit-equal
to the in-place hand-off (same order of the K-slab sums), gated by its ready
flags (poisoned receive buffers, late copies), and bounded when a ready flag
never comes."""

import numpy as np
import pytest
import torch

from reduce_scatter_gb300 import dg
from tests.gpu_common import TOL, Runner, host_inputs, oracle_full, rel_err, to_dev

pytestmark = pytest.mark.gpu

RS = [dg.RS_TILING_A_ROTATING_C, dg.RS_TILING_B_ROTATING_C]


def _ok(sched, m, n, k, tp):
    if sched == dg.RS_TILING_A_ROTATING_C and m % tp:
        return False
    if sched == dg.RS_TILING_B_ROTATING_C and (n % tp or (n // tp) % 8):
        return False
    return k % tp == 0 and (k // tp) % 8 == 0


@pytest.mark.parametrize("cg", [1, 2])
@pytest.mark.parametrize("tp", [2, 4, 8])
@pytest.mark.parametrize("sched", RS, ids=lambda s: dg.SCHEDULE_NAMES[s])
@pytest.mark.parametrize("shape", [(1024, 2048, 1024, 2), (392, 800, 640, 1)], ids=lambda s: "x".join(map(str, s)))
def test_ce_handoff_vs_oracle_and_in_place(shape, sched, tp, cg):
    m, n, k, l = shape
    if not _ok(sched, m, n, k, tp):
        pytest.skip("shape not divisible")
    a, b, c = host_inputs(m, n, k, l, seed=100 + tp + sched)
    A, B, C = to_dev(a), to_dev(b), to_dev(c)
    ref, _ = Runner(m, n, k, l, tp, sched, 0.5, 1.0, options={dg.OPT_CTA_GROUP: cg}).run(A, B, C)
    for ns in (1, 3):
        r = Runner(m, n, k, l, tp, sched, 0.5, 1.0,
                   options={dg.OPT_CTA_GROUP: cg, dg.OPT_RS_CE_PARTIALS: 1, dg.OPT_COPY_STREAMS: ns})
        D, _ = r.run(A, B, C)
        assert rel_err(D, oracle_full(a, b, c, 0.5, 1.0)) <= TOL
        assert torch.equal(D.view(torch.int16), ref.view(torch.int16))
        D2, _ = r.run(A, B, C)  # second run: epochs and per-run counters
        assert torch.equal(D2.view(torch.int16), ref.view(torch.int16))


def test_ce_handoff_gated_by_its_flags():
    m, n, k, l, tp = 1024, 2048, 1024, 1, 4
    a, b, c = host_inputs(m, n, k, l, seed=110)
    A, B = to_dev(a), to_dev(b)
    r = Runner(m, n, k, l, tp, dg.RS_TILING_A_ROTATING_C,
               options={dg.OPT_RS_CE_PARTIALS: 1, dg.OPT_FAULT_DELAY_MS: 40, dg.OPT_TIMEOUT_MS: 5000})
    info = r.plan.info()
    # poison everything after the flag words (counters, send and receive buffers)
    r.ws[info["off_slots"]:].view(torch.int32).fill_(0x7FC00000)
    D, _ = r.run(A, B, None)
    assert rel_err(D, oracle_full(a, b, c, 1.0, 0.0)) <= TOL


def test_ce_handoff_missing_flag_times_out_and_recovers():
    m, n, k, l, tp = 512, 1024, 512, 1, 2
    a, b, c = host_inputs(m, n, k, l, seed=111)
    A, B = to_dev(a), to_dev(b)
    r = Runner(m, n, k, l, tp, dg.RS_TILING_A_ROTATING_C, options={dg.OPT_RS_CE_PARTIALS: 1, dg.OPT_TIMEOUT_MS: 100})
    r.run(A, B, None)
    r.plan.set_option(dg.OPT_FAULT_SKIP_FLAG, 0)
    _, rc = r.run(A, B, None, check=False)
    assert rc == dg.ERR_TIMEOUT, dg.last_error()
    r.plan.set_option(dg.OPT_FAULT_SKIP_FLAG, -1)
    D, rc = r.run(A, B, None)
    assert rc == dg.OK
    assert rel_err(D, oracle_full(a, b, c, 1.0, 0.0)) <= TOL


def test_ce_handoff_needs_a_separate_copy_stream():
    p = dg.Plan(512, 512, 512, 1, 2, dg.RS_TILING_A_ROTATING_C)
    p.set_option(dg.OPT_RS_CE_PARTIALS, 1)
    ws = torch.zeros(p.workspace_bytes(), dtype=torch.uint8, device="cuda")
    A = torch.zeros((512, 512), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream()
    assert p.run(A, A, None, torch.empty_like(A), ws, s, s, raise_on_error=False) == dg.ERR_ARG


@pytest.mark.parametrize("sched", RS, ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_serial_baseline_unaffected_by_ce_option(sched):
    m, n, k, l, tp = 1024, 1024, 1024, 1, 4
    a, b, c = host_inputs(m, n, k, l, seed=112)
    A, B, C = to_dev(a), to_dev(b), to_dev(c)
    plan = dg.Plan(m, n, k, l, tp, sched, 0.5, 1.0)
    plan.set_option(dg.OPT_RS_CE_PARTIALS, 1)
    plan.set_mode(dg.MODE_SERIAL)
    ws = torch.zeros(plan.workspace_bytes(), dtype=torch.uint8, device="cuda")
    D = torch.full((l, m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
    main = torch.cuda.current_stream()
    plan.run(A, B, C, D, ws, main, main)
    plan.check(ws, main)
    assert rel_err(D, oracle_full(a, b, c, 0.5, 1.0)) <= TOL


@pytest.mark.parametrize("sched", RS, ids=lambda s: dg.SCHEDULE_NAMES[s])
@pytest.mark.parametrize("epi", [0, 1, 2, 3, 4])
def test_ce_handoff_direct_paths_and_fp8_out(sched, epi):
    # tiles that leave the staged path (fp8 D at the last step; every tile with EPILOGUE=0 set
    # after the hand-off option) read the partial from the receive buffer and write the send buffer
    from oracle import gemm as og
    m, n, k, l, tp = 1024, 2048, 1024, 2, 4
    a, b, c = host_inputs(m, n, k, l, seed=140 + sched + epi)
    A, B, C = to_dev(a), to_dev(b), to_dev(c)
    ref, _ = Runner(m, n, k, l, tp, sched, 0.5, 1.0).run(A, B, C)
    r = Runner(m, n, k, l, tp, sched, 0.5, 1.0, options={dg.OPT_RS_CE_PARTIALS: 1, dg.OPT_EPILOGUE: epi})
    D, _ = r.run(A, B, C)
    assert torch.equal(D.view(torch.int16), ref.view(torch.int16))
    plan = dg.Plan(m, n, k, l, tp, sched, 0.5, 1.0, out_type="e4m3", result_scale=2.0)
    plan.set_option(dg.OPT_RS_CE_PARTIALS, 1)
    plan.set_option(dg.OPT_EPILOGUE, epi)
    ws = torch.zeros(plan.workspace_bytes(), dtype=torch.uint8, device="cuda")
    D8 = torch.full((l, m, n), 0x7F, dtype=torch.uint8, device="cuda")
    main = torch.cuda.current_stream()
    plan.run_ex(A, B, C, None, D8, ws, main, torch.cuda.Stream())
    plan.check(ws, main)
    want = og.quantize_result(og.gemm(og.bf16_bits_to_f64(a), og.bf16_bits_to_f64(b), og.bf16_bits_to_f64(c),
                                      0.5, 1.0), "e4m3", 2.0)
    assert np.mean(D8.cpu().numpy() == want) >= 0.98


@pytest.mark.parametrize("sched,n", [(dg.RS_TILING_A_ROTATING_C, 8200), (dg.RS_TILING_B_ROTATING_C, 16400)],
                         ids=["RS-TilingA", "RS-TilingB"])
def test_ce_handoff_with_tall_copies(sched, n):
    # 256-row bands of 8200 fp32 columns = 8,396,800 bytes: the tall copy
    # (DG_OPT_COPY_KIND=2) moves each as 65,600 rows of 128 bytes
    m, k, l, tp = 1024, 256, 1, 2
    a, b, c = host_inputs(m, n, k, l, seed=130 + sched)
    A, B, C = to_dev(a), to_dev(b), to_dev(c)
    ref, _ = Runner(m, n, k, l, tp, sched, 0.5, 1.0).run(A, B, C)
    r = Runner(m, n, k, l, tp, sched, 0.5, 1.0, options={dg.OPT_RS_CE_PARTIALS: 1, dg.OPT_COPY_KIND: 2})
    D, _ = r.run(A, B, C)
    assert rel_err(D, oracle_full(a, b, c, 0.5, 1.0)) <= TOL
    assert torch.equal(D.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("sched", RS, ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_ce_handoff_band_merging_and_copy_shapes(sched):
    # hand-off copies of 1, 3 (a shorter last group) or all bands at once, in the
    # operand's rows or reshaped tall: the same bits as the in-place hand-off
    # (4096 rows: RS-TilingA slabs of 4 bands, RS-TilingB of 16)
    m, n, k, l, tp = 4096, 2048, 1024, 2, 4
    a, b, c = host_inputs(m, n, k, l, seed=140 + sched)
    A, B, C = to_dev(a), to_dev(b), to_dev(c)
    ref, _ = Runner(m, n, k, l, tp, sched, 0.5, 1.0).run(A, B, C)
    for bands in (1, 3, 0, 64):
        for kind in (-1, 0, 2):
            r = Runner(m, n, k, l, tp, sched, 0.5, 1.0,
                       options={dg.OPT_RS_CE_PARTIALS: 1, dg.OPT_RS_CE_BANDS: bands, dg.OPT_COPY_KIND: kind})
            D, _ = r.run(A, B, C)
            assert torch.equal(D.view(torch.int16), ref.view(torch.int16)), (bands, kind)
