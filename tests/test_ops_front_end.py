"""The torch-op front end (the fused-op signatures of the torch symmetric-memory
module over the C ABI): argument rules and layouts on CPU; on the GPU every
result element by element against the CPU oracle (``oracle.gemm.fused_gemm``
on the exactly decoded inputs), and the same bits as the C ABI on the
flattened problem."""

import numpy as np
import pytest
import torch

from oracle import gemm as og
from reduce_scatter_gb300 import dg, ops
from tests.gpu_common import TOL, Runner


def test_argument_checks_on_cpu():
    a = torch.zeros((64, 32), dtype=torch.bfloat16)
    w = torch.zeros((48, 32), dtype=torch.bfloat16)           # (N, K) weight
    with pytest.raises(ValueError):
        ops.fused_all_gather_matmul(a, [w.t()], 1, 2)          # gather along K
    with pytest.raises(ValueError):
        ops.fused_all_gather_matmul(a, [w.t()], 0, 2, rotate="C")
    with pytest.raises(ValueError):
        ops.fused_all_gather_matmul(a, [w.t()], 0, 2)          # not CUDA tensors
    with pytest.raises(ValueError):
        ops.fused_all_gather_matmul(a[:63], [w.t()], 0, 2)     # 63 rows over 2 ranks
    with pytest.raises(ValueError):
        ops.fused_matmul_reduce_scatter(a, w.t(), "max", 0, 2)
    with pytest.raises(ValueError):
        ops.fused_matmul_reduce_scatter(a, w.t(), "sum", 2, 2)  # no such dimension
    with pytest.raises(ValueError):
        ops.fused_all_gather_scaled_matmul(a, [w.t()], 1.0, [1.0, 1.0], 0, 2)   # list lengths
    with pytest.raises(ValueError):
        ops.fused_all_gather_scaled_matmul(a, [w.t()], 1.0, [1.0], 0, 2, result_scales=[1.0, 2.0])
    with pytest.raises(ValueError):
        ops._out_type(torch.float16)
    assert ops._out_type(torch.float32) == dg.TYPE_F32
    if hasattr(torch, "float8_e5m2"):
        assert ops._out_type(torch.float8_e5m2) == dg.TYPE_E5M2
    with pytest.raises(TypeError):
        ops._in_type(torch.zeros(2, dtype=torch.float32))
    with pytest.raises(ValueError):
        ops._scale(torch.ones(2))
    assert ops._k_major_b(w.t()).data_ptr() == w.data_ptr()    # used in place
    assert ops._k_major_b(w.t().contiguous()).is_contiguous()


def test_layouts_on_cpu():
    # rank r's shard of the gathered / scattered dimension is the r-th block of rows
    t = torch.arange(2 * 8 * 3 * 4, dtype=torch.float32).view(2, 8, 3, 4)
    A2, lead = ops._rows(t, 1, "gather_dim", 4)
    assert lead == [8, 2, 3] and A2.shape == (48, 4)
    assert torch.equal(A2[:12], t[:, 0:2].movedim(1, 0).reshape(12, 4))   # rank 0: rows 0..1 of dim 1
    D = ops._unflatten(A2, lead, 1)
    assert torch.equal(D, t)
    sched, A2, lead, dim = ops._rs_layout(t, 3, 4)        # last dimension: N-slabs
    assert sched == dg.RS_TILING_B_ROTATING_C and dim is None and lead == [2, 8, 3]
    sched, A2, lead, dim = ops._rs_layout(t, 2, 3)
    assert sched == dg.RS_TILING_A_ROTATING_C and dim == 2
    for d in range(4):
        r = ops.restride_A_shard_for_fused_all_gather_matmul(t, d)
        assert torch.equal(r, t) and r.movedim(d, 0).is_contiguous()
        r = ops.restride_A_for_fused_matmul_reduce_scatter(t, d)
        assert torch.equal(r, t) and r.movedim(d, 0).is_contiguous()


def _randn(shape, seed, dtype=torch.bfloat16, std=1.0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return (torch.randn(shape, device="cuda", generator=g) * std).to(dtype)


def _f64(t):
    """Exact fp64 values of a bf16 or fp8 tensor, decoded by the oracle."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return og.bf16_bits_to_f64(t.view(torch.int16).numpy())
    if hasattr(torch, "float8_e4m3fn") and t.dtype == torch.float8_e4m3fn:
        return og.fp8_bits_to_f64(t.view(torch.uint8).numpy(), "e4m3")
    if hasattr(torch, "float8_e5m2") and t.dtype == torch.float8_e5m2:
        return og.fp8_bits_to_f64(t.view(torch.uint8).numpy(), "e5m2")
    raise TypeError(t.dtype)


def _oracle(A, W, *, alpha=1.0, beta=0.0, C=None, P=1, reduce_op=None, bias=None, k_slice=None):
    """The oracle's D for A (..., K) times the (N, K) weight W: every leading
    dimension of A flattened into rows, the result reshaped back.  ``k_slice``
    restricts the product to those K columns (one rank's K-slab)."""
    a = _f64(A).reshape(1, -1, A.shape[-1])
    w = _f64(W)[None]
    if k_slice is not None:
        a, w = a[:, :, k_slice], w[:, :, k_slice]
    c = None if C is None else _f64(C).reshape(1, -1, W.shape[0])
    D = og.fused_gemm(a, w, c, alpha, beta, P=P, reduce_op=reduce_op, bias=None if bias is None else _f64(bias))
    return D.reshape(*A.shape[:-1], W.shape[0])


def _rel(got, want):
    g = got.detach().double().cpu().numpy()
    assert g.shape == want.shape, (g.shape, want.shape)
    assert not np.isnan(g).any()
    return float(np.abs(g - want).max() / max(np.abs(want).max(), 1e-30))


@pytest.mark.gpu
@pytest.mark.parametrize("rotate", ["A", "B"])
@pytest.mark.parametrize("gather_dim", [0, 1])
def test_all_gather_matmul_multi_b(rotate, gather_dim):
    tp = 4
    A = _randn((4, 256, 512), 1)                      # (batch, seq, hidden): all ranks' shards
    Ws = [_randn((768, 512), 2, std=0.05), _randn((256, 512), 3, std=0.05)]   # (N, K) weights
    Bs = [W.t() for W in Ws]                          # torch layout (K, N), K-major views
    Ag, outs = ops.fused_all_gather_matmul(A, Bs, gather_dim, tp, rotate=rotate)
    torch.cuda.synchronize()
    assert Ag is A and len(outs) == 2
    sched = dg.AG_ROTATING_A if rotate == "A" else dg.AG_ROTATING_B
    A2 = A.movedim(gather_dim, 0).reshape(-1, 512).contiguous()
    for W, B, D in zip(Ws, Bs, outs):
        assert D.shape == (4, 256, W.shape[0])
        assert _rel(D, _oracle(A, W)) <= TOL
        # the same bits as the C ABI on the flattened problem
        ref, _ = Runner(A2.shape[0], W.shape[0], 512, 1, tp, sched).run(A2.unsqueeze(0), W.unsqueeze(0), None)
        flat = D.movedim(gather_dim, 0).reshape(-1, W.shape[0])
        assert torch.equal(flat.view(torch.int16), ref[0].view(torch.int16))


@pytest.mark.gpu
def test_all_gather_matmul_alpha_beta_c():
    tp = 2
    A = _randn((512, 256), 4)
    W = _randn((384, 256), 5, std=0.05)
    C = _randn((512, 384), 6)
    _, (D,) = ops.fused_all_gather_matmul(A, [W.t()], 0, tp, alpha=0.5, beta=1.0, Cs=[C])
    assert _rel(D, _oracle(A, W, alpha=0.5, beta=1.0, C=C)) <= TOL
    # a B that is not a K-major view is copied once: same bits
    _, (D2,) = ops.fused_all_gather_matmul(A, [W.t().contiguous()], 0, tp, alpha=0.5, beta=1.0, Cs=[C])
    assert torch.equal(D.view(torch.int16), D2.view(torch.int16))


@pytest.mark.gpu
@pytest.mark.parametrize("reduce_op", ["sum", "avg"])
@pytest.mark.parametrize("scatter_dim", [0, 1, 2])
def test_matmul_reduce_scatter(scatter_dim, reduce_op):
    tp = 4
    A = _randn((4, 256, 1024), 7)                     # all ranks' K-slabs along the last dimension
    W = _randn((512, 1024), 8, std=0.05)
    D = ops.fused_matmul_reduce_scatter(A, W.t(), reduce_op, scatter_dim, tp)
    assert D.shape == (4, 256, 512)
    assert _rel(D, _oracle(A, W, P=tp, reduce_op=reduce_op)) <= TOL
    # rank r's slab of scatter_dim is the r-th block: per-rank K-slab products reduce to it
    r = 1
    sl = [slice(None)] * 3
    sl[scatter_dim] = slice(r * D.shape[scatter_dim] // tp, (r + 1) * D.shape[scatter_dim] // tp)
    parts = sum(_oracle(A, W, k_slice=slice(q * 256, (q + 1) * 256)) for q in range(tp))
    if reduce_op == "avg":
        parts = parts / tp
    assert _rel(D[tuple(sl)], parts[tuple(sl)]) <= TOL


@pytest.mark.gpu
@pytest.mark.parametrize("reduce_op", ["sum", "avg"])
def test_scaled_ops_fp8_bias_f32(reduce_op):
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("no float8 in this torch")
    tp = 4
    A = _randn((2, 512, 512), 9, dtype=torch.float32).to(torch.float8_e4m3fn)
    W = _randn((1024, 512), 10, dtype=torch.float32).to(torch.float8_e4m3fn)
    bias = _randn((1024,), 11)
    sa, sb = torch.tensor(0.5, device="cuda"), 0.25
    _, (D,) = ops.fused_all_gather_scaled_matmul(A, [W.t()], sa, [sb], 1, tp, biases=[bias],
                                                 out_dtypes=[torch.float32])
    assert D.dtype == torch.float32 and D.shape == (2, 512, 1024)
    assert _rel(D, _oracle(A, W, alpha=0.125, bias=bias)) <= 5e-4
    Dr = ops.fused_scaled_matmul_reduce_scatter(A, W.t(), sa, sb, reduce_op, 1, tp, bias=bias,
                                                out_dtype=torch.float32)
    assert _rel(Dr, _oracle(A, W, alpha=0.125, P=tp, reduce_op=reduce_op, bias=bias)) <= 5e-4
    # bf16 output is the fp32 result rounded
    Db = ops.fused_scaled_matmul_reduce_scatter(A, W.t(), sa, sb, reduce_op, 1, tp, bias=bias,
                                                out_dtype=torch.bfloat16)
    assert Db.dtype == torch.bfloat16
    assert torch.equal(Db.view(torch.int16), Dr.to(torch.bfloat16).view(torch.int16))


@pytest.mark.gpu
def test_four_dim_gather_and_restride():
    # gather along a middle dimension of a 4-D A; a restrided A is read without a layout copy
    tp = 4
    A = _randn((2, 3, 256, 256), 12)
    W = _randn((512, 256), 13, std=0.05)
    _, (D,) = ops.fused_all_gather_matmul(A, [W.t()], 2, tp)
    assert D.shape == (2, 3, 256, 512) and _rel(D, _oracle(A, W)) <= TOL
    Ar = ops.restride_A_shard_for_fused_all_gather_matmul(A, 2)
    assert Ar.movedim(2, 0).is_contiguous()
    _, (Dr,) = ops.fused_all_gather_matmul(Ar, [W.t()], 2, tp)
    assert torch.equal(Dr.view(torch.int16), D.view(torch.int16))


@pytest.mark.gpu
def test_scaled_reduce_scatter_over_n_with_bias():
    # scatter_dim = the output's last dimension: the N-slab schedule, with a bias and fp32 D
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("no float8 in this torch")
    tp = 4
    A = _randn((2, 256, 512), 14, dtype=torch.float32).to(torch.float8_e4m3fn)
    W = _randn((1024, 512), 15, dtype=torch.float32).to(torch.float8_e4m3fn)
    bias = _randn((1024,), 16)
    D = ops.fused_scaled_matmul_reduce_scatter(A, W.t(), 0.5, 0.25, "sum", 2, tp, bias=bias,
                                               out_dtype=torch.float32)
    want = _oracle(A, W, alpha=0.125, P=tp, reduce_op="sum", bias=bias)
    assert D.shape == (2, 256, 1024) and _rel(D, want) <= 5e-4


@pytest.mark.gpu
def test_multi_b_moves_a_once_and_stays_current():
    # later Bs read the shards the first B's run moved: back-to-back calls with new A values
    # must each see their own A
    tp = 4
    Ws = [_randn((512, 1024), 20 + i, std=0.05) for i in range(3)]
    for seed in (30, 31):
        A = _randn((1024, 1024), seed)
        _, outs = ops.fused_all_gather_matmul(A, [W.t() for W in Ws], 0, tp)
        for W, D in zip(Ws, outs):
            ref, _ = Runner(1024, 512, 1024, 1, tp, dg.AG_ROTATING_A).run(A.unsqueeze(0), W.unsqueeze(0), None)
            assert torch.equal(D.view(torch.int16), ref[0].view(torch.int16)), seed


@pytest.mark.gpu
def test_scaled_ops_default_to_the_input_dtype():
    # out_dtype None: the torch op's default, the dtype of B (all-gather) or A (reduce-scatter);
    # for fp8 inputs an fp8 result, result_scale * value rounded to the format
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("no float8 in this torch")
    tp = 4
    A = _randn((512, 512), 17, dtype=torch.float32).to(torch.float8_e4m3fn)
    W = _randn((1024, 512), 18, dtype=torch.float32).to(torch.float8_e4m3fn)
    prod = _oracle(A, W, alpha=0.125)
    _, (D,) = ops.fused_all_gather_scaled_matmul(A, [W.t()], 0.5, [0.25], 0, tp, result_scales=[2.0])
    assert D.dtype == torch.float8_e4m3fn
    want = og.quantize_result(prod, "e4m3", 2.0)
    got = D.view(torch.uint8).cpu().numpy()
    assert np.mean(got == want) >= 0.99
    Dr = ops.fused_scaled_matmul_reduce_scatter(A, W.t(), 0.5, 0.25, "sum", 0, tp, result_scale=2.0)
    assert Dr.dtype == torch.float8_e4m3fn
    assert np.mean(Dr.view(torch.uint8).cpu().numpy() == want) >= 0.99
