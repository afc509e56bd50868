"""A run captured into a CUDA graph: every replay clears the workspace's status
and flag words, so each replay waits for its own shard transfers (and, for
the RS schedules, its own hand-offs) and matches an eager run bit for bit."""

import numpy as np
import pytest
import torch

from reduce_scatter_gb300 import dg
from tests.gpu_common import Runner, host_inputs, to_dev

pytestmark = pytest.mark.gpu

SCHEDS = [dg.AG_ROTATING_A, dg.AG_ROTATING_B, dg.RS_TILING_A_ROTATING_C, dg.RS_TILING_B_ROTATING_C]


@pytest.mark.parametrize("sched", SCHEDS, ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_graph_replays_match_eager_runs(sched):
    m, n, k, l, tp = 1024, 1024, 512, 2, 4
    alpha, beta = 0.5, 1.0
    cap = Runner(m, n, k, l, tp, sched, alpha, beta, options={dg.OPT_FAULT_DELAY_MS: 0})
    ref = Runner(m, n, k, l, tp, sched, alpha, beta)
    a, b, c = host_inputs(m, n, k, l, seed=500 + sched)
    A, B, C = to_dev(a), to_dev(b), to_dev(c)
    D = torch.empty((l, m, n), dtype=torch.bfloat16, device="cuda")
    cap.run(A, B, C, D)                                  # eager first run: sets up the kernels
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cap.plan.run(A, B, C, D, cap.ws, torch.cuda.current_stream(), cap.copy)
    info = cap.plan.info()
    for i in range(3):
        a2, b2, c2 = host_inputs(m, n, k, l, seed=510 + 7 * i + sched)
        A.copy_(to_dev(a2)); B.copy_(to_dev(b2)); C.copy_(to_dev(c2))
        if sched <= 1:
            # stale shards from the previous replay must not be read: poison the slots
            n_slots = tp * (tp - 1) * l
            cap.ws[info["off_slots"]:info["off_slots"] + info["slot_bytes"] * n_slots].view(torch.int16).fill_(0x7FC0)
        D.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert cap.plan.check(cap.ws, torch.cuda.current_stream(), raise_on_error=False) == dg.OK
        want, _ = ref.run(A, B, C)
        assert not torch.isnan(D.float()).any()
        assert torch.equal(D.view(torch.int16), want.view(torch.int16)), i


@pytest.mark.parametrize("sched", SCHEDS, ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_graph_of_a_host_buffer_run(sched):
    # dg_run_host captured whole (uploads gating the tiles, the kernel, block-wise
    # downloads on the plan's own streams): replays with new host inputs in the same
    # pinned buffers give the eager results in the pinned D, over NaN-filled device buffers
    m, n, k, l, tp = 1024, 1024, 512, 2, 4
    alpha, beta = 0.5, 1.0
    cap = Runner(m, n, k, l, tp, sched, alpha, beta)
    ref = Runner(m, n, k, l, tp, sched, alpha, beta)
    a, b, c = host_inputs(m, n, k, l, seed=520 + sched)
    A_h = torch.from_numpy(a.view(np.int16)).pin_memory()
    B_h = torch.from_numpy(b.view(np.int16)).pin_memory()
    C_h = torch.from_numpy(c.view(np.int16)).pin_memory()
    D_h = torch.zeros((l, m, n), dtype=torch.int16).pin_memory()
    A = torch.empty((l, m, k), dtype=torch.bfloat16, device="cuda")
    B = torch.empty((l, n, k), dtype=torch.bfloat16, device="cuda")
    C = torch.empty((l, m, n), dtype=torch.bfloat16, device="cuda")
    D = torch.empty((l, m, n), dtype=torch.bfloat16, device="cuda")
    cap.plan.run_host(A_h, B_h, C_h, None, D_h, A, B, C, D, cap.ws, torch.cuda.current_stream(), cap.copy)
    cap.plan.check(cap.ws, torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cap.plan.run_host(A_h, B_h, C_h, None, D_h, A, B, C, D, cap.ws, torch.cuda.current_stream(), cap.copy)
    for i in range(3):
        a2, b2, c2 = host_inputs(m, n, k, l, seed=530 + 7 * i + sched)
        A_h.copy_(torch.from_numpy(a2.view(np.int16)))
        B_h.copy_(torch.from_numpy(b2.view(np.int16)))
        C_h.copy_(torch.from_numpy(c2.view(np.int16)))
        for t in (A, B, C, D):
            t.fill_(float("nan"))
        D_h.zero_()
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert cap.plan.check(cap.ws, torch.cuda.current_stream(), raise_on_error=False) == dg.OK
        want, _ = ref.run(to_dev(a2), to_dev(b2), to_dev(c2))
        assert torch.equal(D_h, want.view(torch.int16).cpu()), i


@pytest.mark.parametrize("sched", [dg.AG_ROTATING_A, dg.AG_ROTATING_B], ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_multicast_runs_in_graphs_and_with_host_buffers(sched):
    # clusters of two pairs sharing B rows: a captured run replayed with new inputs over poisoned
    # slots, and a dg_run_host call (upload-frontier block order), bit-equal to independent pairs
    m, n, k, l, tp = 2048, 2048, 512, 1, 4
    mc = Runner(m, n, k, l, tp, sched, options={dg.OPT_MULTICAST: 1})
    ref = Runner(m, n, k, l, tp, sched, options={dg.OPT_MULTICAST: 0})
    assert mc.plan.info()["multicast"] == 1
    a, b, c = host_inputs(m, n, k, l, seed=520 + sched)
    A, B = to_dev(a), to_dev(b)
    D = torch.empty((l, m, n), dtype=torch.bfloat16, device="cuda")
    mc.run(A, B, None, D)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        mc.plan.run(A, B, None, D, mc.ws, torch.cuda.current_stream(), mc.copy)
    info = mc.plan.info()
    for i in range(2):
        a2, b2, _ = host_inputs(m, n, k, l, seed=530 + 7 * i + sched)
        A.copy_(to_dev(a2)); B.copy_(to_dev(b2))
        n_slots = tp * (tp - 1) * l
        mc.ws[info["off_slots"]:info["off_slots"] + info["slot_bytes"] * n_slots].view(torch.int16).fill_(0x7FC0)
        D.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert mc.plan.check(mc.ws, torch.cuda.current_stream(), raise_on_error=False) == dg.OK
        want, _ = ref.run(A, B, None)
        assert torch.equal(D.view(torch.int16), want.view(torch.int16)), i
    del g
    A_h, B_h = A.cpu().pin_memory(), B.cpu().pin_memory()
    D_h = torch.empty((l, m, n), dtype=torch.bfloat16).pin_memory()
    A_d, B_d = torch.full_like(A, float("nan")), torch.full_like(B, float("nan"))
    D_d = torch.full_like(D, float("nan"))
    mc.plan.run_host(A_h, B_h, None, None, D_h, A_d, B_d, None, D_d, mc.ws, mc.main, mc.copy)
    assert mc.plan.check(mc.ws, mc.main, raise_on_error=False) == dg.OK
    want, _ = ref.run(A, B, None)
    assert torch.equal(D_h.view(torch.int16), want.cpu().view(torch.int16))
