"""FUSED runs under a layer that serializes launches.

Profilers and CUDA_LAUNCH_BLOCKING=1 run each piece of work to completion in
the order it was issued.  A FUSED run enqueues its shard transfers (and the
uploads of dg_run_host) before the kernel, so under such a layer they land
before the kernel starts and every ready flag is already set when it is
waited on.  Each case runs in a child process with CUDA_LAUNCH_BLOCKING=1 and
a 200 ms flag-wait limit: a transfer stuck behind the kernel would end the run
with DG_ERR_TIMEOUT within that limit, not hang it.
"""

import os
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent("""
    import sys
    import torch
    from reduce_scatter_gb300 import dg
    from tests.gpu_common import TOL, Runner, host_inputs, oracle_full, rel_err, to_dev

    cases = [  # (schedule, tp, m, n, k, l, alpha, beta)
        (dg.AG_ROTATING_A, 2, 256, 256, 256, 1, 1.0, 0.0),      # the smoke problem
        (dg.AG_ROTATING_A, 8, 2048, 2048, 512, 1, 1.0, 0.0),
        (dg.AG_ROTATING_B, 4, 1024, 2048, 512, 2, 0.5, 1.0),
    ]
    for sched, tp, m, n, k, l, alpha, beta in cases:
        a, b, c = host_inputs(m, n, k, l, seed=50 + tp)
        A, B, C = to_dev(a), to_dev(b), to_dev(c)
        r = Runner(m, n, k, l, tp, sched, alpha, beta, options={dg.OPT_TIMEOUT_MS: 200})
        D, rc = r.run(A, B, C if beta else None, check=False)
        assert rc == dg.OK, (dg.SCHEDULE_NAMES[sched], tp, dg.last_error())
        err = rel_err(D, oracle_full(a, b, c, alpha, beta))
        assert err <= TOL, (dg.SCHEDULE_NAMES[sched], tp, err)
        # the same through dg_run_host with pinned buffers (uploads gate tiles)
        if sched != dg.AG_ROTATING_A or tp != 2:
            continue
        A_h, B_h = A.cpu().pin_memory(), B.cpu().pin_memory()
        D_h = torch.empty(D.shape, dtype=D.dtype).pin_memory()
        Dd = torch.full_like(D, float("nan"))
        r.plan.run_host(A_h, B_h, None, None, D_h, A, B, None, Dd, r.ws, r.main, r.copy)
        assert r.plan.check(r.ws, r.main, raise_on_error=False) == dg.OK, dg.last_error()
        assert torch.equal(D_h.view(torch.int16), D.cpu().view(torch.int16))
    print("SERIALIZED_OK")
""")


@pytest.mark.gpu
def test_fused_runs_under_launch_blocking():
    env = dict(os.environ, CUDA_LAUNCH_BLOCKING="1")
    env["PYTHONPATH"] = ROOT + os.pathsep + env.get("PYTHONPATH", "")
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and "SERIALIZED_OK" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]
