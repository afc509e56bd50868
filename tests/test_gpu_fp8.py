"""The scaled variant with fp8 inputs (tcgen05 kind::f8f6f4) against the CPU
oracle: D = alpha * scale_a * scale_b * A B + beta * C with A, B in e4m3 or
e5m2 and C, D in bf16."""

import numpy as np
import pytest
import torch

from oracle import gemm as og
from reduce_scatter_gb300 import configs, dg, synth
from tests.gpu_common import TOL, Runner, host_inputs_fp8, oracle_fp8, rel_err, to_dev, to_dev_u8

pytestmark = pytest.mark.gpu

SCHEDS = [dg.AG_ROTATING_A, dg.AG_ROTATING_B, dg.RS_TILING_A_ROTATING_C, dg.RS_TILING_B_ROTATING_C]
FMTS = {"e4m3": dg.TYPE_E4M3, "e5m2": dg.TYPE_E5M2}


def _ok(sched, m, n, k, tp):
    if sched in (0, 1, 2) and m % tp:
        return False
    if sched != 2 and n % tp:
        return False
    if sched >= 2 and (k % tp or (k // tp) % 16):
        return False
    return True


@pytest.mark.parametrize("fmts", [("e4m3", "e4m3"), ("e5m2", "e5m2"), ("e4m3", "e5m2")], ids=lambda f: "x".join(f))
@pytest.mark.parametrize("tp", [1, 2, 4, 8])
@pytest.mark.parametrize("sched", SCHEDS, ids=lambda s: dg.SCHEDULE_NAMES[s])
@pytest.mark.parametrize("shape", [(512, 1024, 512, 1), (392, 776, 640, 2)], ids=lambda s: "x".join(map(str, s)))
def test_fp8_parity_vs_oracle(shape, sched, tp, fmts):
    m, n, k, l = shape
    if not _ok(sched, m, n, k, tp):
        pytest.skip("shape not divisible for this schedule/tp")
    fa, fb = fmts
    a, b, c = host_inputs_fp8(m, n, k, l, seed=tp + 10 * sched, fmt_a=fa, fmt_b=fb)
    A, B, C = to_dev_u8(a), to_dev_u8(b), to_dev(c)
    for alpha, beta, sa, sb in [(1.0, 0.0, 1.0, 1.0), (0.5, 1.0, 2.0, 0.02)]:
        r = Runner(m, n, k, l, tp, sched, alpha, beta, a_type=FMTS[fa], b_type=FMTS[fb], scale_a=sa, scale_b=sb)
        D, _ = r.run(A, B, C if beta else None)
        assert rel_err(D, oracle_fp8(a, b, c, fa, fb, alpha, beta, sa, sb)) <= TOL


@pytest.mark.parametrize("sched", [dg.AG_ROTATING_A, dg.AG_ROTATING_B], ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_fp8_allgather_bit_exact_vs_unsharded(sched):
    m, n, k, l = 1024, 1024, 640, 1
    a, b, c = host_inputs_fp8(m, n, k, l, seed=3)
    A, B, C = to_dev_u8(a), to_dev_u8(b), to_dev(c)
    kw = dict(a_type=dg.TYPE_E4M3, b_type=dg.TYPE_E4M3, scale_a=1.5, scale_b=0.25)
    ref, _ = Runner(m, n, k, l, 1, sched, 0.5, 1.0, **kw).run(A, B, C)
    for tp in (2, 4, 8):
        D, _ = Runner(m, n, k, l, tp, sched, 0.5, 1.0, **kw).run(A, B, C)
        assert torch.equal(D.view(torch.int16), ref.view(torch.int16)), tp


@pytest.mark.parametrize("epi", [0, 1, 2, 3, 4])
@pytest.mark.parametrize("sched", SCHEDS, ids=lambda s: dg.SCHEDULE_NAMES[s])
def test_fp8_all_ones_and_both_epilogues(sched, epi):
    m, n, l, tp = 512, 512, 1, 4
    for k in (256, 8192):
        one = 0x38  # e4m3 1.0
        A = torch.full((l, m, k), one, dtype=torch.uint8, device="cuda")
        B = torch.full((l, n, k), one, dtype=torch.uint8, device="cuda")
        r = Runner(m, n, k, l, tp, sched, 1.0, 0.0, options={dg.OPT_EPILOGUE: epi}, a_type=dg.TYPE_E4M3,
                   b_type=dg.TYPE_E4M3, scale_a=0.5, scale_b=0.25)
        D, _ = r.run(A, B, None)
        want = torch.tensor(k * 0.125).to(torch.bfloat16).float().item()
        assert torch.all(D.float() == want)


@pytest.mark.parametrize("name", ["ag_a_tp8_pr_e4m3", "rs_a_tp8_e4m3"])
def test_fp8_full_size_sampled(name):
    w = configs.WORKLOADS[name]
    A = synth.tensor_fp8_bits_torch(w.seed, synth.STREAM_A, (w.l, w.m, w.k), w.dist_a, w.in_type, device="cuda",
                                    chunk=1 << 28)
    B = synth.tensor_fp8_bits_torch(w.seed, synth.STREAM_B, (w.l, w.n, w.k), w.dist_b, w.in_type, device="cuda",
                                    chunk=1 << 28)
    r = Runner(w.m, w.n, w.k, w.l, w.tp, w.schedule, w.alpha, w.beta, a_type=dg.TYPE_E4M3, b_type=dg.TYPE_E4M3,
               scale_a=w.scale_a, scale_b=w.scale_b)
    D, _ = r.run(A, B, None)
    assert not torch.isnan(D.float()).any()
    rng = np.random.default_rng(7)
    rows = np.unique(np.concatenate([rng.integers(0, w.m, 40), [0, w.m - 1]]))
    cols = np.unique(np.concatenate([rng.integers(0, w.n, 40), [0, w.n - 1]]))
    a = og.fp8_bits_to_f64(synth.rows_fp8_bits_np(w.seed, synth.STREAM_A, (w.m, w.k), rows, w.dist_a, "e4m3"), "e4m3")
    b = og.fp8_bits_to_f64(synth.rows_fp8_bits_np(w.seed, synth.STREAM_B, (w.n, w.k), cols, w.dist_b, "e4m3"), "e4m3")
    want = og.gemm_entries(a, b, None, w.alpha * w.scale_a * w.scale_b, 0.0)
    got = D.view(w.m, w.n)[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()].float().cpu().numpy()
    assert np.abs(got - want).max() / np.abs(want).max() <= TOL
    if w.schedule == dg.AG_ROTATING_A:
        del r
        ref, _ = Runner(w.m, w.n, w.k, w.l, 1, w.schedule, w.alpha, w.beta, a_type=dg.TYPE_E4M3,
                        b_type=dg.TYPE_E4M3, scale_a=w.scale_a, scale_b=w.scale_b).run(A, B, None)
        assert torch.equal(D.view(torch.int16), ref.view(torch.int16))
