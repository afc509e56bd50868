"""The torch-op front end: argument checks on CPU, and on the GPU the same
results as the C ABI (bit for bit) and as torch's matmul (within tolerance)."""

import numpy as np
import pytest
import torch

from reduce_scatter_gb300 import dg, ops
from tests.gpu_common import TOL, Runner, host_inputs, to_dev


def test_argument_checks_on_cpu():
    a = torch.zeros((64, 32), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        ops.fused_all_gather_matmul(a, a.t(), 2, gather_dim=2)
    with pytest.raises(ValueError):
        ops.fused_matmul_reduce_scatter(a, a.t(), 2, reduce_op="avg")
    with pytest.raises(ValueError):
        ops.fused_all_gather_matmul(a, a.t(), 2)  # not CUDA tensors
    with pytest.raises(TypeError):
        ops._in_type(torch.zeros(2, dtype=torch.float32))
    w = torch.zeros((48, 32), dtype=torch.bfloat16)          # (N, K) weight
    assert ops._k_major_b(w.t().unsqueeze(0)).data_ptr() == w.data_ptr()   # used in place


@pytest.mark.gpu
@pytest.mark.parametrize("sched,kw", [(dg.AG_ROTATING_A, dict(gather_dim=0)), (dg.AG_ROTATING_B, dict(gather_dim=1)),
                                      (dg.RS_TILING_A_ROTATING_C, dict(scatter_dim=0)),
                                      (dg.RS_TILING_B_ROTATING_C, dict(scatter_dim=1))])
def test_ops_match_the_abi_and_torch(sched, kw):
    m, n, k, l, tp = 1024, 768, 512, 2, 4
    a, b, c = host_inputs(m, n, k, l, seed=60 + sched)
    A, Bnk, C = to_dev(a), to_dev(b), to_dev(c)
    B = Bnk.transpose(1, 2)                                   # torch layout (L, K, N), a view
    ref, _ = Runner(m, n, k, l, tp, sched, 0.5, 1.0).run(A, Bnk, C)
    fn = ops.fused_all_gather_matmul if sched <= 1 else ops.fused_matmul_reduce_scatter
    D = fn(A, B, tp, alpha=0.5, beta=1.0, C=C, **kw)
    torch.cuda.synchronize()
    assert torch.equal(D.view(torch.int16), ref.view(torch.int16))
    want = (0.5 * torch.matmul(A.double(), B.double()) + C.double()).float()
    err = (D.float() - want).abs().max().item() / want.abs().max().item()
    assert err <= TOL
    # a B that is not a transposed K-major view is copied once, same result
    D2 = fn(A, B.contiguous(), tp, alpha=0.5, beta=1.0, C=C, **kw)
    torch.cuda.synchronize()
    assert torch.equal(D2.view(torch.int16), ref.view(torch.int16))


@pytest.mark.gpu
def test_scaled_ops_fp8():
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("no float8 in this torch")
    m, n, k, tp = 1024, 1024, 512, 4
    A = (torch.randn((m, k), device="cuda", generator=torch.Generator("cuda").manual_seed(1))).to(torch.float8_e4m3fn)
    W = (torch.randn((n, k), device="cuda", generator=torch.Generator("cuda").manual_seed(2))).to(torch.float8_e4m3fn)
    sa, sb = torch.tensor(0.5, device="cuda"), 0.25
    want = (torch.matmul(A.double(), W.double().t()) * 0.125).float()
    for fn, kw in ((ops.fused_all_gather_scaled_matmul, {}), (ops.fused_scaled_matmul_reduce_scatter, {})):
        D = fn(A, W.t(), sa, sb, tp, **kw)
        torch.cuda.synchronize()
        err = (D.float().squeeze(0) - want).abs().max().item() / want.abs().max().item()
        assert err <= TOL
