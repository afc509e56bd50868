"""dg_run_host with its transfers overlapping the kernel (DG_OPT_HOST_OVERLAP):
uploads in P units gate the tiles that need them (AG also in the
upload-frontier block order), finished (step, rank) blocks of D are downloaded
while later steps run.  The result must be bit-equal to the
sequential form (upload all, run, download) and to a run on device buffers,
whatever the schedule, tp, tile config, beta or input type; uploads that
arrive late must still be waited for; a missing upload must end in a bounded
timeout and leave the plan usable."""

import numpy as np
import pytest
import torch

from reduce_scatter_gb300 import dg
from tests.gpu_common import TOL, Runner, host_inputs, host_inputs_fp8, oracle_full, rel_err, to_dev

pytestmark = pytest.mark.gpu

SCHEDS = [dg.AG_ROTATING_A, dg.AG_ROTATING_B, dg.RS_TILING_A_ROTATING_C, dg.RS_TILING_B_ROTATING_C]


def _host(x, pinned=True):
    t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16 if x.dtype != np.uint8 else np.uint8))
    return t.pin_memory() if pinned else t.clone()


def _run_host(r, a, b, c, out_elems_dtype=torch.int16, pinned=True, poison=False, bias=None, d_shape=None,
              in_dtype=torch.bfloat16, out_dtype=torch.bfloat16):
    """One dg_run_host call of Runner r; returns (D on the host, status)."""
    l, m, k = a.shape
    n = b.shape[1]
    A_h, B_h = _host(a, pinned), _host(b, pinned)
    C_h = _host(c, pinned) if c is not None else None
    D_h = torch.zeros(d_shape or (l, m, n), dtype=out_elems_dtype)
    if pinned:
        D_h = D_h.pin_memory()
    A = torch.empty((l, m, k), dtype=in_dtype, device="cuda")
    B = torch.empty((l, n, k), dtype=in_dtype, device="cuda")
    C = torch.empty((l, m, n), dtype=torch.bfloat16, device="cuda") if c is not None else None
    D = torch.empty((l, m, n), dtype=out_dtype, device="cuda")
    if poison:
        # whatever the kernel reads before the uploads land is NaN
        for t in (A, B, C, D):
            if t is not None:
                t.view(torch.uint8).fill_(0xFF)
    torch.cuda.synchronize()
    r.plan.run_host(A_h, B_h, C_h, bias, D_h, A, B, C, D, r.ws, r.main, r.copy)
    rc = r.plan.check(r.ws, r.main, raise_on_error=False)
    return D_h, rc


def _shape_ok(sched, m, n, k, tp):
    if sched in (dg.AG_ROTATING_A, dg.RS_TILING_A_ROTATING_C) and m % tp:
        return False
    if sched in (dg.AG_ROTATING_B, dg.RS_TILING_B_ROTATING_C) and (n % tp or (n // tp) % 8):
        return False
    if sched in (dg.RS_TILING_A_ROTATING_C, dg.RS_TILING_B_ROTATING_C) and (k % tp or (k // tp) % 8):
        return False
    return True


@pytest.mark.parametrize("beta", [0.0, 1.0])
@pytest.mark.parametrize("cg", [1, 2])
@pytest.mark.parametrize("tp", [1, 2, 4, 8])
@pytest.mark.parametrize("sched", SCHEDS, ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_overlap_bit_equal_to_sequential_and_device(sched, tp, cg, beta):
    m, n, k, l = 768, 1024, 512, 2
    if not _shape_ok(sched, m, n, k, tp):
        pytest.skip("shape not divisible")
    a, b, c = host_inputs(m, n, k, l, seed=300 + 10 * sched + tp)
    c = c if beta != 0 else None
    opts = {dg.OPT_CTA_GROUP: cg}
    D_ov, rc = _run_host(Runner(m, n, k, l, tp, sched, 0.5, beta, options=opts), a, b, c)
    assert rc == dg.OK
    D_seq, rc = _run_host(Runner(m, n, k, l, tp, sched, 0.5, beta, options={**opts, dg.OPT_HOST_OVERLAP: 0}),
                          a, b, c)
    assert rc == dg.OK
    assert torch.equal(D_ov, D_seq)
    want, _ = Runner(m, n, k, l, tp, sched, 0.5, beta, options=opts).run(
        to_dev(a), to_dev(b), to_dev(c) if c is not None else None)
    assert torch.equal(D_ov, want.view(torch.int16).cpu())
    assert rel_err(D_ov.view(torch.bfloat16), oracle_full(a, b, c, 0.5, beta)) <= TOL


@pytest.mark.parametrize("sched", SCHEDS, ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_overlap_waits_for_late_uploads(sched):
    # the upload and copy streams start 40 ms late over NaN-filled device
    # buffers: every tile must still read its uploaded inputs
    m, n, k, l, tp = 1024, 1024, 512, 1, 4
    a, b, c = host_inputs(m, n, k, l, seed=320 + sched)
    r = Runner(m, n, k, l, tp, sched, 0.5, 1.0, options={dg.OPT_FAULT_DELAY_MS: 40, dg.OPT_TIMEOUT_MS: 5000})
    D_h, rc = _run_host(r, a, b, c, poison=True)
    assert rc == dg.OK
    want, _ = Runner(m, n, k, l, tp, sched, 0.5, 1.0).run(to_dev(a), to_dev(b), to_dev(c))
    assert torch.equal(D_h, want.view(torch.int16).cpu())


@pytest.mark.parametrize("sched", [dg.AG_ROTATING_A, dg.RS_TILING_B_ROTATING_C], ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_pageable_host_memory_takes_the_sequential_form(sched):
    m, n, k, l, tp = 512, 1024, 512, 1, 2
    a, b, c = host_inputs(m, n, k, l, seed=330 + sched)
    D_h, rc = _run_host(Runner(m, n, k, l, tp, sched, 0.5, 1.0), a, b, c, pinned=False)
    assert rc == dg.OK
    want, _ = Runner(m, n, k, l, tp, sched, 0.5, 1.0).run(to_dev(a), to_dev(b), to_dev(c))
    assert torch.equal(D_h, want.view(torch.int16).cpu())


def test_missing_upload_times_out_and_recovers():
    # uploads held back 400 ms against a 50 ms wait limit: the kernel gives up
    # (bounded), the download waits are released, dg_check reports the upload
    # wait; the next run without the delay is correct
    m, n, k, l, tp = 1024, 1024, 512, 1, 4
    a, b, c = host_inputs(m, n, k, l, seed=340)
    r = Runner(m, n, k, l, tp, dg.AG_ROTATING_A, 1.0, 0.0, options={dg.OPT_FAULT_DELAY_MS: 400, dg.OPT_TIMEOUT_MS: 50})
    _, rc = _run_host(r, a, b, None)
    assert rc == dg.ERR_TIMEOUT
    assert "upload wait" in dg.last_error()
    r.plan.set_option(dg.OPT_FAULT_DELAY_MS, 0)
    r.plan.set_option(dg.OPT_TIMEOUT_MS, 2000)
    D_h, rc = _run_host(r, a, b, None)
    assert rc == dg.OK
    want, _ = Runner(m, n, k, l, tp, dg.AG_ROTATING_A, 1.0, 0.0).run(to_dev(a), to_dev(b), None)
    assert torch.equal(D_h, want.view(torch.int16).cpu())


@pytest.mark.parametrize("sched", SCHEDS, ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_overlap_fp8_inputs_fp32_out_and_bias(sched):
    m, n, k, l, tp = 512, 1024, 512, 2, 4
    a, b, c = host_inputs_fp8(m, n, k, l, seed=350 + sched)
    bias = (torch.randn(n, device="cuda") * 0.5).to(torch.bfloat16)
    D = {}
    for ov in (1, 0):
        r = Runner(m, n, k, l, tp, sched, 0.5, 1.0, a_type=dg.TYPE_E4M3, b_type=dg.TYPE_E4M3, scale_a=0.5,
                   scale_b=2.0, options={dg.OPT_HOST_OVERLAP: ov, dg.OPT_OUT_TYPE: dg.TYPE_F32})
        D[ov], rc = _run_host(r, a, b, c, out_elems_dtype=torch.float32, bias=bias, in_dtype=torch.uint8,
                              out_dtype=torch.float32)
        assert rc == dg.OK
    assert torch.equal(D[0], D[1])
    assert torch.isfinite(D[1]).all()


@pytest.mark.parametrize("sched", [dg.RS_TILING_A_ROTATING_C, dg.RS_TILING_B_ROTATING_C],
                         ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_overlap_with_copy_engine_hand_off(sched):
    m, n, k, l, tp = 1024, 2048, 1024, 2, 4
    a, b, c = host_inputs(m, n, k, l, seed=360 + sched)
    D_h, rc = _run_host(Runner(m, n, k, l, tp, sched, 0.5, 1.0, options={dg.OPT_RS_CE_PARTIALS: 1}), a, b, c)
    assert rc == dg.OK
    want, _ = Runner(m, n, k, l, tp, sched, 0.5, 1.0).run(to_dev(a), to_dev(b), to_dev(c))
    assert torch.equal(D_h, want.view(torch.int16).cpu())


def test_back_to_back_calls_reuse_buffers():
    # consecutive calls on the same device buffers: a call's uploads must not
    # overwrite inputs the previous call's kernel still reads
    m, n, k, l, tp = 2048, 2048, 1024, 1, 8
    r = Runner(m, n, k, l, tp, dg.AG_ROTATING_A, 1.0, 0.0)
    ins = [host_inputs(m, n, k, l, seed=370 + i)[:2] for i in range(3)]
    A = torch.empty((l, m, k), dtype=torch.bfloat16, device="cuda")
    B = torch.empty((l, n, k), dtype=torch.bfloat16, device="cuda")
    D = torch.empty((l, m, n), dtype=torch.bfloat16, device="cuda")
    outs, keep = [], []
    for a, b in ins:
        D_h = torch.zeros((l, m, n), dtype=torch.int16).pin_memory()
        # the host inputs must outlive the asynchronous call: the library holds raw
        # pointers, so torch's pinned-memory cache would otherwise hand a freed block
        # to the next iteration while this call's upload still reads it
        A_h, B_h = _host(a), _host(b)
        keep += [A_h, B_h]
        r.plan.run_host(A_h, B_h, None, None, D_h, A, B, None, D, r.ws, r.main, r.copy)
        outs.append(D_h)
    r.plan.check(r.ws, r.main)
    for (a, b), D_h in zip(ins, outs):
        want, _ = Runner(m, n, k, l, tp, dg.AG_ROTATING_A, 1.0, 0.0).run(to_dev(a), to_dev(b), None)
        assert torch.equal(D_h, want.view(torch.int16).cpu())


@pytest.mark.parametrize("cg", [1, 2])
@pytest.mark.parametrize("tp", [2, 4, 8])
@pytest.mark.parametrize("sched", [dg.AG_ROTATING_A, dg.AG_ROTATING_B], ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_upload_frontier_order_on_device_runs(sched, tp, cg):
    # the block order of the upload frontier, asked for on a device-buffer run,
    # with late transfers over NaN-filled receive slots: the same bits
    m, n, k, l = 1024, 1536, 512, 2
    a, b, c = host_inputs(m, n, k, l, seed=380 + 10 * sched + tp)
    A, B, C = to_dev(a), to_dev(b), to_dev(c)
    ref, _ = Runner(m, n, k, l, tp, sched, 0.5, 1.0, options={dg.OPT_CTA_GROUP: cg}).run(A, B, C)
    r = Runner(m, n, k, l, tp, sched, 0.5, 1.0,
               options={dg.OPT_CTA_GROUP: cg, dg.OPT_TILE_ORDER: 1, dg.OPT_FAULT_DELAY_MS: 20,
                        dg.OPT_TIMEOUT_MS: 5000})
    info = r.plan.info()
    r.ws[info["off_slots"]:info["off_slots"] + info["slot_bytes"] * tp * (tp - 1) * l].view(torch.int16).fill_(0x7FC0)
    for _ in range(2):
        D, rc = r.run(A, B, C)
        assert rc == dg.OK
        assert torch.equal(D.view(torch.int16), ref.view(torch.int16))
