"""Device path against the CPU oracle, through the C ABI, on small problems
that span several tiles and ragged tails; bit-exactness of the AllGather
schedules against the unsharded run; run modes; closed forms; edge cases."""

import numpy as np
import pytest
import torch

from reduce_scatter_gb300 import dg
from tests.gpu_common import TOL, Runner, host_inputs, oracle_full, rel_err, to_dev

pytestmark = pytest.mark.gpu

SCHEDS = [dg.AG_ROTATING_A, dg.AG_ROTATING_B, dg.RS_TILING_A_ROTATING_C, dg.RS_TILING_B_ROTATING_C]
# (m, n, k, l): several tiles; ragged shards and a ragged K block
SHAPES = [(512, 1024, 512, 1), (392, 776, 320, 2), (1024, 528, 200, 1)]


def _shape_ok(sched, m, n, k, tp):
    if sched in (0, 1, 2) and m % tp:
        return False
    if sched != 2 and n % tp:
        return False
    if sched >= 2 and (k % tp or (k // tp) % 8):
        return False
    return True


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("tp", [1, 2, 4, 8])
@pytest.mark.parametrize("sched", SCHEDS, ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_parity_vs_oracle(sched, tp, shape):
    m, n, k, l = shape
    if not _shape_ok(sched, m, n, k, tp):
        pytest.skip("shape not divisible for this schedule/tp")
    a, b, c = host_inputs(m, n, k, l, seed=tp + 10 * sched)
    A, B, C = to_dev(a), to_dev(b), to_dev(c)
    for alpha, beta in [(1.0, 0.0), (0.5, 1.0)]:
        r = Runner(m, n, k, l, tp, sched, alpha, beta)
        D, _ = r.run(A, B, C if beta else None)
        err = rel_err(D, oracle_full(a, b, c, alpha, beta))
        assert err <= TOL, (err, alpha, beta)
        # a second run reuses the workspace: epochs, not memsets, guard the flags
        D2, _ = r.run(A, B, C if beta else None)
        assert torch.equal(D.view(torch.int16), D2.view(torch.int16))


@pytest.mark.parametrize("sched", [dg.AG_ROTATING_A, dg.AG_ROTATING_B], ids=lambda s: dg.SCHEDULE_NAMES[s])
@pytest.mark.parametrize("shape", [(1024, 1024, 328, 1), (392, 776, 320, 2)], ids=lambda s: "x".join(map(str, s)))
def test_allgather_bit_exact_vs_unsharded(sched, shape):
    m, n, k, l = shape
    a, b, c = host_inputs(m, n, k, l, seed=3)
    A, B, C = to_dev(a), to_dev(b), to_dev(c)
    ref, _ = Runner(m, n, k, l, 1, sched, 0.5, 1.0).run(A, B, C)
    for tp in (2, 4, 8):
        if not _shape_ok(sched, m, n, k, tp):
            continue
        D, _ = Runner(m, n, k, l, tp, sched, 0.5, 1.0).run(A, B, C)
        assert torch.equal(D.view(torch.int16), ref.view(torch.int16)), tp


def test_rs_tp1_is_the_plain_gemm_bit_for_bit():
    m, n, k, l = 512, 768, 512, 1
    a, b, c = host_inputs(m, n, k, l, seed=4)
    A, B, C = to_dev(a), to_dev(b), to_dev(c)
    ref, _ = Runner(m, n, k, l, 1, dg.AG_ROTATING_A, 0.75, -0.5).run(A, B, C)
    for sched in (dg.RS_TILING_A_ROTATING_C, dg.RS_TILING_B_ROTATING_C):
        D, _ = Runner(m, n, k, l, 1, sched, 0.75, -0.5).run(A, B, C)
        assert torch.equal(D.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("sched", [dg.AG_ROTATING_A, dg.AG_ROTATING_B], ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_modes_agree(sched):
    m, n, k, l, tp = 1024, 1024, 512, 1, 4
    a, b, c = host_inputs(m, n, k, l, seed=5)
    A, B = to_dev(a), to_dev(b)
    fused, _ = Runner(m, n, k, l, tp, sched).run(A, B, None)
    serial, _ = Runner(m, n, k, l, tp, sched, mode=dg.MODE_SERIAL).run(A, B, None)
    r = Runner(m, n, k, l, tp, sched)
    r.run(A, B, None)  # fills the receive slots
    r.plan.set_mode(dg.MODE_GEMM_ONLY)
    gemm_only, _ = r.run(A, B, None)
    for D in (serial, gemm_only):
        assert torch.equal(D.view(torch.int16), fused.view(torch.int16))
    # copy stream == main stream runs the transfers first
    r2 = Runner(m, n, k, l, tp, sched)
    D = torch.empty_like(fused)
    r2.plan.run(A, B, None, D, r2.ws, r2.main, r2.main)
    r2.plan.check(r2.ws, r2.main)
    assert torch.equal(D.view(torch.int16), fused.view(torch.int16))


@pytest.mark.parametrize("sched", SCHEDS, ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_closed_forms(sched):
    tp = 4
    # all ones: D = K * alpha + beta * C, exact
    for k in (256, 8192):
        m, n, l = 512, 512, 1
        A = torch.ones((l, m, k), dtype=torch.bfloat16, device="cuda")
        B = torch.ones((l, n, k), dtype=torch.bfloat16, device="cuda")
        C = torch.full((l, m, n), 3.0, dtype=torch.bfloat16, device="cuda")
        D, _ = Runner(m, n, k, l, tp, sched, 0.5, 2.0).run(A, B, C)
        # the fp32 value 0.5*K + 6 is exact; D holds it rounded to bf16
        want = torch.tensor(0.5 * k + 6.0).to(torch.bfloat16).float().item()
        assert torch.all(D.float() == want)
    # identity B (N = K): D = A; one-hot B: D[:, n] = A[:, perm[n]]
    m, k, l = 256, 512, 1
    a, _, _ = host_inputs(m, k, k, l, seed=6)
    A = to_dev(a)
    eye = torch.eye(k, dtype=torch.bfloat16, device="cuda")[None]
    D, _ = Runner(m, k, k, l, tp, sched).run(A, eye, None)
    assert torch.equal(D.float(), A.float())  # value equality (+0 == -0)
    n = 384
    perm = torch.randint(0, k, (n,), generator=torch.Generator().manual_seed(7))
    onehot = torch.zeros((1, n, k), dtype=torch.bfloat16)
    onehot[0, torch.arange(n), perm] = 1.0
    D, _ = Runner(m, n, k, l, tp, sched).run(A, onehot.cuda(), None)
    assert torch.equal(D.float(), A[:, :, perm.cuda()].float())


@pytest.mark.parametrize("sched", SCHEDS, ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_k_zero_gives_beta_c(sched):
    m, n, k, l, tp = 256, 512, 0, 1, 2
    c = host_inputs(m, n, 8, l, seed=8)[2]
    C = to_dev(c)
    A = torch.empty((16,), dtype=torch.bfloat16, device="cuda")
    B = torch.empty((16,), dtype=torch.bfloat16, device="cuda")
    D, _ = Runner(m, n, k, l, tp, sched, 1.0, 0.5).run(A, B, C)
    assert torch.equal(D.float(), (0.5 * C.float()).to(torch.bfloat16).float())


def test_beta_zero_ignores_nan_c():
    m, n, k, l = 256, 512, 128, 1
    a, b, c = host_inputs(m, n, k, l, seed=9)
    A, B = to_dev(a), to_dev(b)
    Cn = torch.full((l, m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
    for sched in SCHEDS:
        D, _ = Runner(m, n, k, l, 2, sched, 1.0, 0.0).run(A, B, Cn)
        assert rel_err(D, oracle_full(a, b, c, 1.0, 0.0)) <= TOL


def test_single_row_shards():
    # tp = 8 with M = 8: one row per shard, 127 of every 128 tile rows masked
    m, n, k, l, tp = 8, 64, 64, 3, 8
    a, b, c = host_inputs(m, n, k, l, seed=10)
    A, B, C = to_dev(a), to_dev(b), to_dev(c)
    for sched in SCHEDS:
        if not _shape_ok(sched, m, n, k, tp):
            continue
        D, _ = Runner(m, n, k, l, tp, sched, 1.0, 1.0).run(A, B, C)
        assert rel_err(D, oracle_full(a, b, c, 1.0, 1.0)) <= TOL


def test_does_not_write_outside_d():
    m, n, k, l, tp = 392, 776, 320, 1, 4
    a, b, c = host_inputs(m, n, k, l, seed=11)
    A, B = to_dev(a), to_dev(b)
    for sched in SCHEDS:
        big = torch.full((l * m * n + 4096,), 7.0, dtype=torch.bfloat16, device="cuda")
        D = big[2048: 2048 + l * m * n].view(l, m, n)
        Runner(m, n, k, l, tp, sched).run(A, B, None, D)
        assert torch.all(big[:2048] == 7.0) and torch.all(big[2048 + l * m * n:] == 7.0)


@pytest.mark.parametrize("tp", [1, 2, 4, 8])
@pytest.mark.parametrize("sched", SCHEDS, ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_single_sm_tiles_vs_oracle(sched, tp):
    # the 128 x 256 single-SM tile configuration (DG_OPT_CTA_GROUP = 1)
    m, n, k, l = 392, 776, 320, 2
    if not _shape_ok(sched, m, n, k, tp):
        pytest.skip("shape not divisible for this schedule/tp")
    a, b, c = host_inputs(m, n, k, l, seed=50 + tp + 10 * sched)
    A, B, C = to_dev(a), to_dev(b), to_dev(c)
    r = Runner(m, n, k, l, tp, sched, 0.5, 1.0, options={dg.OPT_CTA_GROUP: 1})
    D, _ = r.run(A, B, C)
    assert rel_err(D, oracle_full(a, b, c, 0.5, 1.0)) <= TOL
    if sched in (dg.AG_ROTATING_A, dg.AG_ROTATING_B) and tp > 1:
        ref, _ = Runner(m, n, k, l, 1, sched, 0.5, 1.0, options={dg.OPT_CTA_GROUP: 1}).run(A, B, C)
        assert torch.equal(D.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("epi", [0, 1, 2, 3, 4])
@pytest.mark.parametrize("sched", SCHEDS, ids=lambda s: dg.SCHEDULE_NAMES[s])
@pytest.mark.parametrize("shape", [(1024, 2048, 512, 2), (392, 776, 320, 2)], ids=lambda s: "x".join(map(str, s)))
def test_both_epilogues_vs_oracle(sched, epi, shape):
    # staged (TMA through shared memory) and direct epilogues, every schedule;
    # the ragged shape mixes staged tiles with tiles whose column offset is not
    # 16-byte aligned (those fall back to direct accesses)
    m, n, k, l = shape
    for tp in (2, 4):
        if not _shape_ok(sched, m, n, k, tp):
            continue
        a, b, c = host_inputs(m, n, k, l, seed=70 + tp + 10 * sched + epi)
        A, B, C = to_dev(a), to_dev(b), to_dev(c)
        for alpha, beta in [(1.0, 0.0), (0.5, 1.0)]:
            r = Runner(m, n, k, l, tp, sched, alpha, beta, options={dg.OPT_EPILOGUE: epi})
            D, _ = r.run(A, B, C if beta else None)
            assert rel_err(D, oracle_full(a, b, c, alpha, beta)) <= TOL, (tp, alpha, beta)
            D2, _ = r.run(A, B, C if beta else None)
            assert torch.equal(D.view(torch.int16), D2.view(torch.int16))


@pytest.mark.parametrize("sched", [dg.RS_TILING_A_ROTATING_C, dg.RS_TILING_B_ROTATING_C],
                         ids=lambda s: dg.SCHEDULE_NAMES[s])
@pytest.mark.parametrize("epi", [0, 1, 2, 3, 4])
def test_rs_nonfused_baseline_vs_oracle(sched, epi):
    # SERIAL on an RS plan: per-rank partial GEMMs, then the separate reduction
    m, n, k, l, tp = 1024, 1024, 1024, 2, 4
    a, b, c = host_inputs(m, n, k, l, seed=80 + sched)
    A, B, C = to_dev(a), to_dev(b), to_dev(c)
    for alpha, beta in [(1.0, 0.0), (0.5, 1.0)]:
        plan = dg.Plan(m, n, k, l, tp, sched, alpha, beta)
        plan.set_option(dg.OPT_EPILOGUE, epi)
        plan.set_mode(dg.MODE_SERIAL)
        ws = torch.zeros(plan.workspace_bytes(), dtype=torch.uint8, device="cuda")
        D = torch.full((l, m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
        main = torch.cuda.current_stream()
        plan.run(A, B, C if beta else None, D, ws, main, main)
        plan.check(ws, main)
        assert rel_err(D, oracle_full(a, b, c, alpha, beta)) <= TOL


def test_rs_serial_needs_the_serial_workspace():
    plan = dg.Plan(256, 256, 256, 1, 2, dg.RS_TILING_A_ROTATING_C)
    small = plan.workspace_bytes()          # FUSED sizing
    plan.set_mode(dg.MODE_SERIAL)
    ws = torch.zeros(small, dtype=torch.uint8, device="cuda")
    A = torch.zeros((256, 256), dtype=torch.bfloat16, device="cuda")
    rc = plan.run(A, A, None, torch.empty_like(A), ws, raise_on_error=False)
    assert rc == dg.ERR_STATE


@pytest.mark.parametrize("hint", [2, 6, 9, 16, 32, 18])
def test_l2_hints_do_not_change_results(hint):
    # operand policies (bits 0-3) and the epilogue's (bits 4-5, in every staged epilogue)
    m, n, k, l, tp = 1024, 2048, 512, 1, 4
    a, b, c = host_inputs(m, n, k, l, seed=90)
    A, B, C = to_dev(a), to_dev(b), to_dev(c)
    for sched in SCHEDS:
        for epi in ([None] if hint < 16 else [None, 1, 2, 3, 4]):
            extra = {} if epi is None else {dg.OPT_EPILOGUE: epi}
            ref, _ = Runner(m, n, k, l, tp, sched, 0.5, 1.0, options=extra).run(A, B, C)
            D, _ = Runner(m, n, k, l, tp, sched, 0.5, 1.0, options={dg.OPT_L2_HINT: hint, **extra}).run(A, B, C)
            assert torch.equal(D.view(torch.int16), ref.view(torch.int16)), (sched, epi)


@pytest.mark.parametrize("sched", SCHEDS, ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_wave_sync_does_not_change_results(sched):
    m, n, k, l, tp = 2048, 4096, 512, 1, 4
    a, b, c = host_inputs(m, n, k, l, seed=91)
    A, B, C = to_dev(a), to_dev(b), to_dev(c)
    ref, _ = Runner(m, n, k, l, tp, sched, 0.5, 1.0).run(A, B, C)
    r = Runner(m, n, k, l, tp, sched, 0.5, 1.0, options={dg.OPT_WAVE_SYNC: 1, dg.OPT_TIMEOUT_MS: 1000})
    for _ in range(2):
        D, rc = r.run(A, B, C)
        assert rc == dg.OK
        assert torch.equal(D.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("sched", SCHEDS, ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_run_host_matches_device_run(sched):
    # dg_run_host: pinned host inputs uploaded, the run, D downloaded; same bits as dg_run
    m, n, k, l, tp = 1024, 1024, 512, 2, 4
    a, b, c = host_inputs(m, n, k, l, seed=90 + sched)
    A_h = torch.from_numpy(a.view(np.int16)).pin_memory()
    B_h = torch.from_numpy(b.view(np.int16)).pin_memory()
    C_h = torch.from_numpy(c.view(np.int16)).pin_memory()
    D_h = torch.empty((l, m, n), dtype=torch.int16).pin_memory()
    r = Runner(m, n, k, l, tp, sched, 0.5, 1.0)
    A = torch.empty((l, m, k), dtype=torch.bfloat16, device="cuda")
    B = torch.empty((l, n, k), dtype=torch.bfloat16, device="cuda")
    C = torch.empty((l, m, n), dtype=torch.bfloat16, device="cuda")
    D = torch.empty((l, m, n), dtype=torch.bfloat16, device="cuda")
    r.plan.run_host(A_h, B_h, C_h, None, D_h, A, B, C, D, r.ws, r.main, r.copy)
    r.plan.check(r.ws, r.main)
    want, _ = Runner(m, n, k, l, tp, sched, 0.5, 1.0).run(to_dev(a), to_dev(b), to_dev(c))
    assert torch.equal(D_h, want.view(torch.int16).cpu())


@pytest.mark.parametrize("tp", [1, 2, 4])
@pytest.mark.parametrize("sched", SCHEDS, ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_tiny_shapes_against_brute_force(sched, tp):
    # the device path against the triple loop itself (not only the oracle) on
    # integer-valued inputs, where every summation order is exact
    from tests.pin_checks import brute_gemm
    for (m, n, k, l) in [(64, 64, 64, 1), (32, 48, 64, 2)]:
        if not _shape_ok(sched, m, n, k, tp):
            continue
        rng = np.random.default_rng(1000 + 10 * sched + tp + m)
        Ai = rng.integers(-4, 5, (l, m, k)).astype(np.float32)
        Bi = rng.integers(-4, 5, (l, n, k)).astype(np.float32)
        Ci = rng.integers(-4, 5, (l, m, n)).astype(np.float32)
        A = torch.from_numpy(Ai).cuda().to(torch.bfloat16)
        B = torch.from_numpy(Bi).cuda().to(torch.bfloat16)
        C = torch.from_numpy(Ci).cuda().to(torch.bfloat16)
        D, _ = Runner(m, n, k, l, tp, sched, 0.5, 2.0).run(A, B, C)
        want = brute_gemm(Ai.astype(np.float64), Bi.astype(np.float64), Ci.astype(np.float64), 0.5, 2.0)
        # every partial and the fp32 epilogue are exact here (|acc| <= 64 * 16), so D is the exact
        # result rounded once to bf16 (nearest even): equal bits
        want_bf16 = torch.from_numpy(want.astype(np.float32)).to(torch.bfloat16)
        assert torch.equal(D.cpu().view(torch.int16), want_bf16.view(torch.int16)), (m, n, k, l)


@pytest.mark.parametrize("tp", [1, 2, 4])
@pytest.mark.parametrize("sched", SCHEDS, ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_zero_k(sched, tp):
    # K = 0: no MMA, the accumulator is zero, D = beta * C exactly (beta = 1 gives C's
    # bits, beta = 0 gives +0), through every hand-off and transfer path
    m, n, k, l = 512, 768, 0, 2
    if not _shape_ok(sched, m, n, 8 * tp, tp):
        pytest.skip("shape not divisible")
    a, b, c = host_inputs(m, n, 8, l, seed=150 + sched)
    C = to_dev(c)
    A = torch.zeros(64, dtype=torch.bfloat16, device="cuda")  # never read (no K blocks), but not NULL
    B = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    for opts in ({}, {dg.OPT_CTA_GROUP: 1}, {dg.OPT_RS_CE_PARTIALS: 1} if sched >= 2 and tp > 1 else {}):
        D, _ = Runner(m, n, k, l, tp, sched, 0.75, 1.0, options=opts).run(A, B, C)
        assert torch.equal(D.view(torch.int16), C.view(torch.int16)), opts
        D0, _ = Runner(m, n, k, l, tp, sched, 0.75, 0.0, options=opts).run(A, B, None)
        assert torch.equal(D0.view(torch.int16), torch.zeros_like(D0.view(torch.int16))), opts


@pytest.mark.parametrize("cg", [1, 2])
@pytest.mark.parametrize("sched", SCHEDS, ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_one_row_and_eight_column_shards(sched, cg):
    # tp = 8 with one row per M-shard (M = 8) or eight columns per N-shard (N = 64):
    # tiles almost all outside the shard, transfers of one row, K of one block
    tp, l = 8, 2
    m, n, k = (8, 200, 64) if sched in (dg.AG_ROTATING_A, dg.RS_TILING_A_ROTATING_C) else (40, 64, 64)
    a, b, c = host_inputs(m, n, k, l, seed=160 + sched)
    A, B, C = to_dev(a), to_dev(b), to_dev(c)
    D, _ = Runner(m, n, k, l, tp, sched, 0.5, 1.0, options={dg.OPT_CTA_GROUP: cg}).run(A, B, C)
    assert rel_err(D, oracle_full(a, b, c, 0.5, 1.0)) <= TOL
    if sched in (dg.AG_ROTATING_A, dg.AG_ROTATING_B):
        ref, _ = Runner(m, n, k, l, 1, sched, 0.5, 1.0, options={dg.OPT_CTA_GROUP: cg}).run(A, B, C)
        assert torch.equal(D.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("cg", [1, 2])
@pytest.mark.parametrize("sched", SCHEDS, ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_per_warp_epilogue_same_bits_as_staged(sched, cg):
    # the per-warp and the stores-only epilogues compute every element the same way (one fmaf of
    # the accumulator and its source, or with alpha a power of two its exact equivalent by
    # reduction, the same hand-off order), so D matches the per-CTA staged epilogue bit for bit,
    # on full and ragged tiles, with and without C
    for m, n, k, l in [(1024, 2048, 512, 2), (392, 776, 320, 2), (1000, 1096, 256, 1)]:
        for tp in (1, 4):
            if not _shape_ok(sched, m, n, k, tp):
                continue
            a, b, c = host_inputs(m, n, k, l, seed=90 + tp + 10 * sched)
            A, B, C = to_dev(a), to_dev(b), to_dev(c)
            for alpha, beta in [(1.0, 0.0), (0.5, 1.0)]:
                out = {}
                for epi in (1, 2, 3, 4):
                    r = Runner(m, n, k, l, tp, sched, alpha, beta,
                               options={dg.OPT_EPILOGUE: epi, dg.OPT_CTA_GROUP: cg})
                    out[epi], _ = r.run(A, B, C if beta else None)
                for epi in (2, 3, 4):
                    assert torch.equal(out[1].view(torch.int16), out[epi].view(torch.int16)), (m, n, tp, alpha, epi)
                assert rel_err(out[2], oracle_full(a, b, c, alpha, beta)) <= TOL


@pytest.mark.parametrize("epi", [1, 2, 4])
@pytest.mark.parametrize("cg", [1, 2])
@pytest.mark.parametrize("sched", [dg.RS_TILING_A_ROTATING_C, dg.RS_TILING_B_ROTATING_C],
                         ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_rs_reduction_into_the_partial_vs_oracle(sched, cg, epi):
    # middle steps add their product into the rotating partial by TMA reductions; ragged boxes
    # load, add and store directly; repeated runs give the same bits (the hand-off order is fixed)
    for m, n, k, l in [(1024, 2048, 512, 2), (392, 776, 320, 2), (1000, 1096, 256, 1)]:
        for tp in (2, 4, 8):
            if not _shape_ok(sched, m, n, k, tp):
                continue
            a, b, c = host_inputs(m, n, k, l, seed=95 + tp + 10 * sched)
            A, B, C = to_dev(a), to_dev(b), to_dev(c)
            for alpha, beta in [(1.0, 0.0), (0.5, 1.0)]:
                r = Runner(m, n, k, l, tp, sched, alpha, beta,
                           options={dg.OPT_RS_REDUCE: 1, dg.OPT_CTA_GROUP: cg, dg.OPT_EPILOGUE: epi})
                D, _ = r.run(A, B, C if beta else None)
                assert rel_err(D, oracle_full(a, b, c, alpha, beta)) <= TOL, (m, n, tp, alpha, beta)
                D2, _ = r.run(A, B, C if beta else None)
                assert torch.equal(D.view(torch.int16), D2.view(torch.int16))


@pytest.mark.parametrize("epi", [1, 2])
@pytest.mark.parametrize("sched", [dg.RS_TILING_A_ROTATING_C, dg.RS_TILING_B_ROTATING_C],
                         ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_rs_reduction_same_bits_when_alpha_is_a_power_of_two(sched, epi):
    # alpha' * acc is exact for alpha' = 2^e, so the L2's round-to-nearest add of it to the
    # partial gives the bits of fmaf(alpha', acc, partial): for such alpha' the reduction, on by
    # default, changes no bit
    for m, n, k, l in [(1024, 2048, 1024, 2), (392, 776, 320, 2)]:
        for tp in (4, 8):
            if not _shape_ok(sched, m, n, k, tp):
                continue
            a, b, c = host_inputs(m, n, k, l, seed=97 + tp + 10 * sched)
            A, B, C = to_dev(a), to_dev(b), to_dev(c)
            for alpha, beta in [(1.0, 0.0), (0.5, 1.0), (-0.25, 0.75)]:
                out = {}
                for red in (0, 1, -1):
                    r = Runner(m, n, k, l, tp, sched, alpha, beta,
                               options={dg.OPT_RS_REDUCE: red, dg.OPT_EPILOGUE: epi})
                    out[red], _ = r.run(A, B, C if beta else None)
                for red in (1, -1):
                    assert torch.equal(out[0].view(torch.int16), out[red].view(torch.int16)), (m, tp, alpha, red)


@pytest.mark.parametrize("sched", [dg.RS_TILING_A_ROTATING_C, dg.RS_TILING_B_ROTATING_C],
                         ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_rs_reduction_by_default_with_alpha_not_a_power_of_two(sched):
    # without a bias the middle steps reduce by default whatever alpha' is: the product is
    # rounded, then added (two roundings); the staged epilogues agree bit for bit on whole
    # tiles, and every variant, the one-rounding path (RS_REDUCE=0) and the copy-engine
    # hand-off included, stays within tolerance of the oracle
    for m, n, k, l in [(1024, 2048, 1024, 2), (392, 776, 320, 2)]:
        whole = m == 1024
        for tp in (4, 8):
            if not _shape_ok(sched, m, n, k, tp):
                continue
            a, b, c = host_inputs(m, n, k, l, seed=98 + tp + 10 * sched)
            A, B, C = to_dev(a), to_dev(b), to_dev(c)
            for alpha, beta in [(0.75, 1.0), (-1.3, 0.0)]:
                want = oracle_full(a, b, c, alpha, beta)
                ref, _ = Runner(m, n, k, l, tp, sched, alpha, beta, options={dg.OPT_EPILOGUE: 1}).run(
                    A, B, C if beta else None)
                assert rel_err(ref, want) <= TOL
                variants = [{dg.OPT_EPILOGUE: e} for e in (0, 2, 3, 4)] + [{dg.OPT_CTA_GROUP: 1},
                                                                           {dg.OPT_RS_REDUCE: 0}]
                if sched == dg.RS_TILING_A_ROTATING_C or (n // tp) % 8 == 0:
                    variants += [{dg.OPT_RS_CE_PARTIALS: 1}]
                for opts in variants:
                    D, _ = Runner(m, n, k, l, tp, sched, alpha, beta, options=opts).run(A, B, C if beta else None)
                    assert rel_err(D, want) <= TOL, (m, tp, alpha, opts)
                    if whole and opts.get(dg.OPT_EPILOGUE) in (2, 4):
                        assert torch.equal(D.view(torch.int16), ref.view(torch.int16)), (m, tp, alpha, opts)


@pytest.mark.parametrize("sched", [dg.AG_ROTATING_A, dg.AG_ROTATING_B], ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_b_multicast_between_pairs_same_bits(sched):
    # clusters of two CTA pairs sharing their B rows compute every tile with the same MMAs:
    # the same bits as independent pairs, and within tolerance of the oracle
    for m, n, k, l in [(1024, 2048, 512, 2), (2048, 1024, 1024, 1), (512, 1536, 256, 1)]:
        for tp in (1, 2, 4):
            if not _shape_ok(sched, m, n, k, tp):
                continue
            a, b, c = host_inputs(m, n, k, l, seed=99 + tp + 10 * sched)
            A, B, C = to_dev(a), to_dev(b), to_dev(c)
            for alpha, beta in [(1.0, 0.0), (0.5, 1.0)]:
                out = {}
                for mc in (0, 1):
                    r = Runner(m, n, k, l, tp, sched, alpha, beta,
                               options={dg.OPT_MULTICAST: mc, dg.OPT_TIMEOUT_MS: 500})
                    out[mc], rc = r.run(A, B, C if beta else None, check=False)
                    assert rc == dg.OK, (m, n, tp, mc, dg.last_error())
                assert torch.equal(out[0].view(torch.int16), out[1].view(torch.int16)), (m, n, tp, alpha)
                assert rel_err(out[1], oracle_full(a, b, c, alpha, beta)) <= TOL
