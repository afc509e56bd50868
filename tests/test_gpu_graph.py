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
