"""Full-size workloads, in the launch configuration the benchmark times.

The oracle cannot evaluate these problems whole, so:
* sampled entries D[rows, cols] (rows spread over every shard and batch,
  columns over every shard) are checked against the oracle evaluated on
  exactly those rows of A and B, drawn again on the CPU from the same seeded
  generator;
* AllGather schedules are compared bit for bit with the unsharded (tp=1) run
  of the same kernel, since the K order does not change;
* ReduceScatter schedules are compared with the unsharded run within the
  tolerance (the K order of the partial sums differs);
* D holds no NaN (every element written).
"""

import numpy as np
import pytest
import torch

from oracle import gemm as og
from reduce_scatter_gb300 import configs, dg, synth
from tests.gpu_common import TOL, Runner

pytestmark = pytest.mark.gpu

FULL = ["ag_a_tp2_blog", "ag_a_tp8_pr", "rs_a_tp8", "ag_b_tp4_batched", "rs_b_tp4_batched"]


def _dev_inputs(w):
    A = synth.tensor_bits_torch(w.seed, synth.STREAM_A, (w.l, w.m, w.k), w.dist_a, device="cuda").view(torch.bfloat16)
    B = synth.tensor_bits_torch(w.seed, synth.STREAM_B, (w.l, w.n, w.k), w.dist_b, device="cuda").view(torch.bfloat16)
    C = None
    if w.beta != 0:
        C = synth.tensor_bits_torch(w.seed, synth.STREAM_C, (w.l, w.m, w.n), w.dist_c, device="cuda").view(torch.bfloat16)
    return A, B, C


def _sample_check(w, D, nrows=48, ncols=48):
    rng = np.random.default_rng(12345)
    LM = w.l * w.m
    rows = np.unique(np.concatenate([rng.integers(0, LM, nrows), [0, LM - 1]]))
    cols = np.unique(np.concatenate([rng.integers(0, w.n, ncols), [0, w.n - 1]]))
    Dh = D.view(LM, w.n)[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()].float().cpu().numpy()
    worst = 0.0
    for b in range(w.l):
        rs = rows[(rows >= b * w.m) & (rows < (b + 1) * w.m)]
        if len(rs) == 0:
            continue
        a = og.bf16_bits_to_f64(synth.rows_bits_np(w.seed, synth.STREAM_A, (LM, w.k), rs, w.dist_a))
        bb = og.bf16_bits_to_f64(synth.rows_bits_np(w.seed, synth.STREAM_B, (w.l * w.n, w.k), cols + b * w.n, w.dist_b))
        c = None
        if w.beta != 0:
            c = og.bf16_bits_to_f64(synth.rows_bits_np(w.seed, synth.STREAM_C, (LM, w.n), rs, w.dist_c)[:, cols])
        want = og.gemm_entries(a, bb, c, w.alpha, w.beta)
        got = Dh[np.isin(rows, rs)].astype(np.float64)
        assert not np.any(np.isnan(got))
        worst = max(worst, float(np.abs(got - want).max() / np.abs(want).max()))
    assert worst <= TOL, worst
    return worst


@pytest.mark.parametrize("name", FULL)
def test_full_size(name):
    w = configs.WORKLOADS[name]
    A, B, C = _dev_inputs(w)
    r = Runner(w.m, w.n, w.k, w.l, w.tp, w.schedule, w.alpha, w.beta)
    D, _ = r.run(A, B, C)
    assert not torch.isnan(D.float()).any()
    _sample_check(w, D)
    del r
    ref_sched = w.schedule if w.schedule in (dg.AG_ROTATING_A, dg.AG_ROTATING_B) else dg.AG_ROTATING_A
    ref, _ = Runner(w.m, w.n, w.k, w.l, 1, ref_sched, w.alpha, w.beta).run(A, B, C)
    if w.schedule in (dg.AG_ROTATING_A, dg.AG_ROTATING_B):
        assert torch.equal(D.view(torch.int16), ref.view(torch.int16))
    else:
        err = (D.float() - ref.float()).abs().max().item() / ref.float().abs().max().item()
        assert err <= TOL, err


@pytest.mark.parametrize("name,op", [("ag_b_tp4_batched", None), ("rs_b_tp4_batched", "avg"),
                                     ("rs_a_tp8", "sum")])
def test_full_size_bias_f32_out(name, op):
    # the scaled ops' epilogue extras at full size: bias, fp32 D, the reduce op
    w = configs.WORKLOADS[name]
    A, B, C = _dev_inputs(w)
    bias_bits = synth.tensor_bits_np(w.seed, synth.STREAM_BIAS, (w.n,), ("uniform", -4.0, 4.0))
    bias = torch.from_numpy(bias_bits.view(np.int16)).cuda().view(torch.bfloat16)
    plan = dg.Plan(w.m, w.n, w.k, w.l, w.tp, w.schedule, w.alpha, w.beta, out_type="f32",
                   reduce_op=op or "sum")
    ws = torch.zeros(max(plan.workspace_bytes(), 256), dtype=torch.uint8, device="cuda")
    D = torch.full((w.l, w.m, w.n), float("nan"), dtype=torch.float32, device="cuda")
    main = torch.cuda.current_stream()
    plan.run_ex(A, B, C, bias, D, ws, main, torch.cuda.Stream())
    plan.check(ws, main)
    assert not torch.isnan(D).any()
    rng = np.random.default_rng(777)
    LM = w.l * w.m
    rows = np.unique(np.concatenate([rng.integers(0, LM, 40), [0, LM - 1]]))
    cols = np.unique(np.concatenate([rng.integers(0, w.n, 40), [0, w.n - 1]]))
    Dh = D.view(LM, w.n)[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()].cpu().numpy()
    bcols = og.bf16_bits_to_f64(bias_bits)[cols]
    for b in range(w.l):
        rs = rows[(rows >= b * w.m) & (rows < (b + 1) * w.m)]
        if len(rs) == 0:
            continue
        a = og.bf16_bits_to_f64(synth.rows_bits_np(w.seed, synth.STREAM_A, (LM, w.k), rs, w.dist_a))
        bb = og.bf16_bits_to_f64(synth.rows_bits_np(w.seed, synth.STREAM_B, (w.l * w.n, w.k), cols + b * w.n, w.dist_b))
        c = None
        if w.beta != 0:
            c = og.bf16_bits_to_f64(synth.rows_bits_np(w.seed, synth.STREAM_C, (LM, w.n), rs, w.dist_c)[:, cols])
        want = og.fused_gemm_entries(a, bb, c, w.alpha, w.beta, P=w.tp, reduce_op=op, bias_cols=bcols)
        got = Dh[np.isin(rows, rs)].astype(np.float64)
        # fp32 D: the fp32 accumulation error (about sqrt(K) * 2^-24 relative for these random
        # inputs) stays far inside 5e-4 of max|D|; a result rounded to bf16 on the way (up to
        # 2^-9 of each entry) would exceed it at the largest entries
        assert np.abs(got - want).max() / np.abs(want).max() <= 5e-4


@pytest.mark.parametrize("name", ["ag_a_tp8_pr", "rs_b_tp4_batched"])
def test_full_size_from_host_buffers(name):
    # the end-to-end call the benchmark times: pinned host inputs uploaded in
    # units that gate the tiles, D downloaded block by block; bit-equal to the
    # run on device buffers, and sampled entries against the oracle
    w = configs.WORKLOADS[name]
    A, B, C = _dev_inputs(w)
    r = Runner(w.m, w.n, w.k, w.l, w.tp, w.schedule, w.alpha, w.beta)
    ref, _ = r.run(A, B, C)
    A_h, B_h = A.cpu().pin_memory(), B.cpu().pin_memory()
    C_h = C.cpu().pin_memory() if C is not None else None
    D_h = torch.empty((w.l, w.m, w.n), dtype=torch.bfloat16).pin_memory()
    for t in (A, B, C):
        if t is not None:
            t.view(torch.int16).fill_(0x7FC0)  # NaN until the upload lands
    D = torch.empty_like(ref)
    r.plan.run_host(A_h, B_h, C_h, None, D_h, A, B, C, D, r.ws, r.main, r.copy)
    r.plan.check(r.ws, r.main)
    assert torch.equal(D_h.view(torch.int16), ref.view(torch.int16).cpu())
    _sample_check(w, D_h.cuda())


def test_operands_beyond_32_bit_element_counts():
    # B of 131072 x 32768 (4.3e9 elements, 8.6 GB) and D of 16384 x 131072 (2.1e9):
    # element offsets past 2^31 and 2^32 in every addressing path (TMA rows, the
    # epilogue's plain accesses, the shard transfers)
    from reduce_scatter_gb300.configs import Workload, N1, N002
    w = Workload("ag_a_tp8_wide", 0, 8, 16384, 131072, 32768, dist_a=N1, dist_b=N002)
    A, B, C = _dev_inputs(w)
    r = Runner(w.m, w.n, w.k, w.l, w.tp, w.schedule, w.alpha, w.beta)
    D, _ = r.run(A, B, C)
    assert not torch.isnan(D).any()
    _sample_check(w, D, nrows=24, ncols=24)


@pytest.mark.parametrize("cep", [0, 1])
def test_rs_partials_beyond_32_bit_element_counts(cep):
    # RS-TilingB with D of 16384 x 131072 (2.1e9 elements): the fp32 partial (8.6 GB), and
    # with the copy-engine hand-off the send and receive buffers, addressed past 2^31
    from reduce_scatter_gb300.configs import Workload, N1, N002
    w = Workload("rs_b_tp4_wide", 3, 4, 16384, 131072, 4096, dist_a=N1, dist_b=N002)
    A, B, C = _dev_inputs(w)
    r = Runner(w.m, w.n, w.k, w.l, w.tp, w.schedule, w.alpha, w.beta, options={dg.OPT_RS_CE_PARTIALS: cep})
    D, _ = r.run(A, B, C)
    assert not torch.isnan(D).any()
    _sample_check(w, D, nrows=24, ncols=24)
