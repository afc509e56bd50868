"""Flag gating and bounded waits on the GPU.

* Receive slots poisoned with NaN and the copy stream held back: the kernel
  must wait for every chunk's ready flag, so D is still correct.
* The same poisoned slots read without waiting (GEMM_ONLY) do give NaN, which
  shows the poison reaches D when a wait is missing.
* A ready flag that nothing writes: the wait runs out after the configured
  limit, the kernel finishes, dg_check reports DG_ERR_TIMEOUT, and the next
  run on the same context is correct.
Nothing here faults or hangs the GPU: every wait in the kernel is bounded.
"""

import numpy as np
import pytest
import torch

from reduce_scatter_gb300 import dg
from tests.gpu_common import TOL, Runner, host_inputs, oracle_full, rel_err, to_dev

pytestmark = pytest.mark.gpu


def _poison_slots(r: Runner):
    info = r.plan.info()
    lo = info["off_slots"]
    hi = lo + info["tp"] * (info["tp"] - 1) * info["l"] * info["slot_bytes"]
    r.ws[lo:hi].view(torch.int16).fill_(0x7FC0)  # bf16 quiet NaN


@pytest.mark.parametrize("sched", [dg.AG_ROTATING_A, dg.AG_ROTATING_B], ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_poisoned_slots_with_late_copies(sched):
    m, n, k, l, tp = 1024, 1024, 512, 2, 4
    a, b, c = host_inputs(m, n, k, l, seed=21)
    A, B = to_dev(a), to_dev(b)
    want = oracle_full(a, b, c, 1.0, 0.0)
    r = Runner(m, n, k, l, tp, sched, options={dg.OPT_FAULT_DELAY_MS: 50, dg.OPT_TIMEOUT_MS: 5000})
    _poison_slots(r)
    D, _ = r.run(A, B, None)
    assert rel_err(D, want) <= TOL
    # without the waits the poison shows
    _poison_slots(r)
    r.plan.set_mode(dg.MODE_GEMM_ONLY)
    D2 = torch.zeros_like(D)
    r.run(A, B, None, D2)
    assert torch.isnan(D2.float()).any()


def test_missing_flag_times_out_and_context_survives():
    m, n, k, l, tp = 512, 512, 256, 1, 2
    a, b, c = host_inputs(m, n, k, l, seed=22)
    A, B = to_dev(a), to_dev(b)
    r = Runner(m, n, k, l, tp, dg.AG_ROTATING_A, options={dg.OPT_TIMEOUT_MS: 100})
    r.run(A, B, None)          # warm: flags hold this run's epoch
    r.plan.set_option(dg.OPT_FAULT_SKIP_FLAG, 0)
    _, rc = r.run(A, B, None, check=False)
    assert rc == dg.ERR_TIMEOUT, dg.last_error()
    assert "flag 0" in dg.last_error()
    r.plan.set_option(dg.OPT_FAULT_SKIP_FLAG, -1)
    D, rc = r.run(A, B, None)
    assert rc == dg.OK
    assert rel_err(D, oracle_full(a, b, c, 1.0, 0.0)) <= TOL


def test_workspace_handed_between_plans():
    # a workspace reused by another plan has its flags cleared first, so the
    # other plan's larger epochs cannot satisfy this plan's waits
    m, n, k, l, tp = 512, 512, 256, 1, 4
    a, b, c = host_inputs(m, n, k, l, seed=23)
    A, B = to_dev(a), to_dev(b)
    r1 = Runner(m, n, k, l, tp, dg.AG_ROTATING_A)
    for _ in range(5):
        r1.run(A, B, None)
    r2 = Runner(m, n, k, l, tp, dg.AG_ROTATING_A, options={dg.OPT_FAULT_DELAY_MS: 30})
    r2.ws = r1.ws
    _poison_slots(r2)
    D, _ = r2.run(A, B, None)
    assert rel_err(D, oracle_full(a, b, c, 1.0, 0.0)) <= TOL


def test_plan_alternating_between_workspaces():
    # one plan, two workspaces used in turn, with another plan on the second
    # in between: stale flag words in either workspace must never satisfy a
    # wait of a later run (copies held back, slots poisoned)
    m, n, k, l, tp = 512, 512, 256, 1, 4
    a, b, c = host_inputs(m, n, k, l, seed=24)
    A, B = to_dev(a), to_dev(b)
    want = oracle_full(a, b, c, 1.0, 0.0)
    r1 = Runner(m, n, k, l, tp, dg.AG_ROTATING_A)
    ws_a = r1.ws
    ws_b = torch.zeros_like(ws_a)
    for _ in range(4):
        r1.run(A, B, None)                      # plan 1 on ws_a, epochs 1..4
    r1.ws = ws_b
    r1.run(A, B, None)                          # plan 1 on ws_b
    other = Runner(m, n, k, l, tp, dg.AG_ROTATING_A)
    other.ws = ws_b
    for _ in range(8):
        other.run(A, B, None)                   # another plan pushes ws_b's flags high
    r1.plan.set_option(dg.OPT_FAULT_DELAY_MS, 30)
    for ws in (ws_a, ws_b, ws_a):
        r1.ws = ws
        _poison_slots(r1)
        D, _ = r1.run(A, B, None)
        assert rel_err(D, want) <= TOL


@pytest.mark.parametrize("ns", [2, 3, 8])
def test_transfers_over_several_copy_streams(ns):
    m, n, k, l, tp = 1024, 2048, 512, 2, 4
    a, b, c = host_inputs(m, n, k, l, seed=25)
    A, B = to_dev(a), to_dev(b)
    want = oracle_full(a, b, c, 1.0, 0.0)
    for sched in (dg.AG_ROTATING_A, dg.AG_ROTATING_B):
        r = Runner(m, n, k, l, tp, sched, options={dg.OPT_COPY_STREAMS: ns, dg.OPT_FAULT_DELAY_MS: 20,
                                                   dg.OPT_CHUNK_TILES: 1})
        _poison_slots(r)
        D, _ = r.run(A, B, None)
        assert rel_err(D, want) <= TOL
        D2, _ = r.run(A, B, None)
        assert torch.equal(D.view(torch.int16), D2.view(torch.int16))


@pytest.mark.parametrize("epi", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("tp", [2, 4])
@pytest.mark.parametrize("sched", [dg.RS_TILING_A_ROTATING_C, dg.RS_TILING_B_ROTATING_C],
                         ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_rs_grid_equal_to_step_distance(sched, tp, epi):
    # epi 3, 4, 5: the staged and the two per-warp epilogues with the middle steps' TMA reductions
    # With as many CTA pairs as tiles between a tile and its next step, every
    # pair's next tile waits on the hand-off it made itself; the kernel must
    # release it first (a missed release shows up as a timeout, not a hang).
    m, n, k, l = 256 * tp, 2048, 128 * tp, 1
    plan_tiles = dg.Plan(m, n, k, l, tp, sched).info()
    per_block = plan_tiles["tiles_m"] * plan_tiles["tiles_n"] * l
    pairs = (tp - 1) * per_block
    a, b, c = host_inputs(m, n, k, l, seed=26)
    A, B, C = to_dev(a), to_dev(b), to_dev(c)
    r = Runner(m, n, k, l, tp, sched, 0.5, 1.0,
               options={dg.OPT_GRID: 2 * pairs, dg.OPT_TIMEOUT_MS: 500, dg.OPT_EPILOGUE: (0, 1, 2, 1, 2, 4)[epi],
                        dg.OPT_RS_REDUCE: int(epi >= 3)})
    D, rc = r.run(A, B, C, check=False)
    assert rc == dg.OK, dg.last_error()
    assert rel_err(D, oracle_full(a, b, c, 0.5, 1.0)) <= TOL


@pytest.mark.parametrize("sched", [dg.AG_ROTATING_A, dg.AG_ROTATING_B], ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_paced_transfers_same_bits(sched):
    # copies of step s >= 2 held until the kernel reaches step s - 1, or all at once
    m, n, k, l, tp = 2048, 2048, 512, 2, 8
    a, b, c = host_inputs(m, n, k, l, seed=400 + sched)
    A, B, C = to_dev(a), to_dev(b), to_dev(c)
    D = {}
    for pace in (0, 1):
        r = Runner(m, n, k, l, tp, sched, 0.5, 1.0, options={dg.OPT_COPY_PACE: pace, dg.OPT_CHUNK_TILES: 1})
        D[pace], _ = r.run(A, B, C)
        D2, _ = r.run(A, B, C)                        # the progress words are reset per run
        assert torch.equal(D[pace].view(torch.int16), D2.view(torch.int16))
    assert torch.equal(D[0].view(torch.int16), D[1].view(torch.int16))
    assert rel_err(D[1], oracle_full(a, b, c, 0.5, 1.0)) <= TOL


def test_paced_transfers_with_held_copies():
    # copies held back on the host and NaN-poisoned slots: pacing must still gate every load
    m, n, k, l, tp = 1024, 1024, 256, 1, 4
    a, b, c = host_inputs(m, n, k, l, seed=410)
    A, B = to_dev(a), to_dev(b)
    r = Runner(m, n, k, l, tp, dg.AG_ROTATING_A, options={dg.OPT_COPY_PACE: 1, dg.OPT_FAULT_DELAY_MS: 50})
    info = r.plan.info()
    r.ws[info["off_slots"]:info["off_slots"] + info["slot_bytes"] * tp * (tp - 1)].view(torch.int16).fill_(0x7FC0)
    D, _ = r.run(A, B, None)
    assert rel_err(D, oracle_full(a, b, c, 1.0, 0.0)) <= TOL


@pytest.mark.parametrize("sched", [dg.AG_ROTATING_A, dg.AG_ROTATING_B], ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_copy_kinds_same_bits(sched):
    # row-shaped 2D, one-dimensional and tall 2D transfers move the same bytes
    m, n, k, l, tp = 1024, 2048, 512, 2, 4
    a, b, c = host_inputs(m, n, k, l, seed=420 + sched)
    A, B, C = to_dev(a), to_dev(b), to_dev(c)
    D = {}
    for kind in (0, 1, 2):
        r = Runner(m, n, k, l, tp, sched, 0.5, 1.0, options={dg.OPT_COPY_KIND: kind})
        D[kind], _ = r.run(A, B, C)
    assert torch.equal(D[0].view(torch.int16), D[1].view(torch.int16))
    assert torch.equal(D[0].view(torch.int16), D[2].view(torch.int16))


@pytest.mark.parametrize("sched,m,n,tp", [(dg.AG_ROTATING_A, 8198, 512, 2), (dg.AG_ROTATING_B, 256, 32792, 8)],
                         ids=["AG-RotatingA", "AG-RotatingB"])
def test_tall_copies_with_a_remainder(sched, m, n, tp):
    # one chunk per shard of 4099 rows x 2064 bytes = 8,460,336 bytes: the tall
    # copy (kind 2) takes 66,096 rows of 128 bytes and a 48-byte remainder
    k, l = 1032, 1
    a, b, c = host_inputs(m, n, k, l, seed=431 + sched)
    A, B, C = to_dev(a), to_dev(b), to_dev(c)
    D = {}
    for kind in (0, 1, 2):
        r = Runner(m, n, k, l, tp, sched, 0.5, 1.0, options={dg.OPT_COPY_KIND: kind, dg.OPT_CHUNK_TILES: 64})
        assert r.plan.info()["chunks_per_shard"] == 1
        D[kind], _ = r.run(A, B, C)
    assert torch.equal(D[0].view(torch.int16), D[1].view(torch.int16))
    assert torch.equal(D[0].view(torch.int16), D[2].view(torch.int16))
    rows = np.r_[0:3, m // 2 - 1:m // 2 + 2, m - 3:m]
    ref = oracle_full(a[:, rows], b, c[:, rows], 0.5, 1.0)
    assert rel_err(D[0][:, torch.as_tensor(rows, device="cuda")], ref) <= TOL
