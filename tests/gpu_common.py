"""Helpers shared by the GPU tests: seeded inputs, one run through the C ABI,
and the comparison against the CPU oracle."""

from __future__ import annotations

import numpy as np
import torch

from oracle import gemm as og
from reduce_scatter_gb300 import dg, synth

TOL = 2e-2  # max|D - D_oracle| <= TOL * max|D_oracle| (bf16 inputs, fp32 accumulation)

UNIFORM = ("uniform", -1.0, 1.0)


def host_inputs(m, n, k, l, seed=1, da=UNIFORM, db=UNIFORM, dc=UNIFORM):
    a = synth.tensor_bits_np(seed, synth.STREAM_A, (l, m, k), da)
    b = synth.tensor_bits_np(seed, synth.STREAM_B, (l, n, k), db)
    c = synth.tensor_bits_np(seed, synth.STREAM_C, (l, m, n), dc)
    return a, b, c


def to_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def host_inputs_fp8(m, n, k, l, seed=1, fmt_a="e4m3", fmt_b="e4m3", da=("normal", 0.0, 1.0),
                    db=("normal", 0.0, 1.0), dc=UNIFORM):
    a = synth.tensor_fp8_bits_np(seed, synth.STREAM_A, (l, m, k), da, fmt_a)
    b = synth.tensor_fp8_bits_np(seed, synth.STREAM_B, (l, n, k), db, fmt_b)
    c = synth.tensor_bits_np(seed, synth.STREAM_C, (l, m, n), dc)
    return a, b, c


def to_dev_u8(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits)).cuda()


class Runner:
    """A plan, its workspace and two streams."""

    def __init__(self, m, n, k, l, tp, sched, alpha=1.0, beta=0.0, mode=dg.MODE_FUSED, options=None,
                 a_type=dg.TYPE_BF16, b_type=dg.TYPE_BF16, scale_a=1.0, scale_b=1.0):
        self.plan = dg.Plan(m, n, k, l, tp, sched, alpha, beta, a_type, b_type, scale_a, scale_b)
        self.plan.set_mode(mode)
        for opt, val in (options or {}).items():
            self.plan.set_option(opt, val)
        self.ws = torch.zeros(max(self.plan.workspace_bytes(), 256), dtype=torch.uint8, device="cuda")
        self.main = torch.cuda.current_stream()
        self.copy = torch.cuda.Stream()
        self.shape = (l, m, n)

    def run(self, A, B, C, D=None, check=True):
        if D is None:
            D = torch.full(self.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        self.plan.run(A, B, C, D, self.ws, self.main, self.copy)
        rc = self.plan.check(self.ws, self.main, raise_on_error=check)
        return D, rc


def oracle_full(a, b, c, alpha, beta):
    return og.gemm(og.bf16_bits_to_f64(a), og.bf16_bits_to_f64(b),
                   og.bf16_bits_to_f64(c) if beta != 0 else None, alpha, beta)


def oracle_fp8(a, b, c, fmt_a, fmt_b, alpha, beta, scale_a, scale_b):
    return og.scaled_gemm(og.fp8_bits_to_f64(a, fmt_a), og.fp8_bits_to_f64(b, fmt_b),
                          og.bf16_bits_to_f64(c) if beta != 0 else None, alpha, beta, scale_a, scale_b)


def rel_err(D: torch.Tensor, want: np.ndarray) -> float:
    got = D.float().cpu().numpy().astype(np.float64)
    assert not np.any(np.isnan(got)), "NaN in D (unwritten or poisoned output)"
    scale = max(np.abs(want).max(), 1e-30)
    return float(np.abs(got - want).max() / scale)
