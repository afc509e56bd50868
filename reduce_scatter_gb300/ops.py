"""torch-tensor front end of the C ABI, after the fused ops of
torch/distributed/_symmetric_memory (fused_all_gather_matmul,
fused_matmul_reduce_scatter and their scaled variants).

Every TP rank is emulated on the one GPU, so each call takes the tensors of
ALL virtual ranks (the unsharded A and B) and returns the whole D; the rank
layout, the rotation and the shard transfers are the library's.  This module
only marshals arguments: plans and workspaces are cached, outputs allocated
with torch, and every step of the computation runs in ``libdg.so``.

Conventions (torch's ``A @ B``):
  A: (M, K) or (L, M, K);  B: (K, N) or (L, K, N);  C, D: (M, N) or (L, M, N).
The kernels read B K-major, i.e. stored as (N, K).  If ``B`` is the
transposed view of a contiguous (N, K) tensor (``W.t()`` / ``W.mT``) it is
used in place; otherwise a K-major copy is made (one extra pass over B).
"""

from __future__ import annotations

import threading

import torch

from . import dg

_lock = threading.Lock()
_plans: dict = {}
_workspaces: dict = {}
_copy_streams: dict = {}

_FP8 = {}
for _name, _t in (("float8_e4m3fn", dg.TYPE_E4M3), ("float8_e5m2", dg.TYPE_E5M2)):
    if hasattr(torch, _name):
        _FP8[getattr(torch, _name)] = _t


def _in_type(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return dg.TYPE_BF16
    if t.dtype in _FP8:
        return _FP8[t.dtype]
    raise TypeError(f"inputs must be bfloat16 or float8 (e4m3fn / e5m2), got {t.dtype}")


def _batched(t: torch.Tensor, name: str) -> torch.Tensor:
    if t.dim() == 2:
        return t.unsqueeze(0)
    if t.dim() == 3:
        return t
    raise ValueError(f"{name} must be 2-D or 3-D (batch first), got shape {tuple(t.shape)}")


def _k_major_b(B: torch.Tensor) -> torch.Tensor:
    """(L, K, N) B as an (L, N, K) tensor with K contiguous, without a copy when possible."""
    Bt = B.transpose(-1, -2)
    if Bt.is_contiguous():
        return Bt
    return Bt.contiguous()


def _workspace(device: torch.device, nbytes: int) -> torch.Tensor:
    key = (device.index, nbytes)
    ws = _workspaces.get(key)
    if ws is None:
        ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws


def _copy_stream(device: torch.device) -> torch.cuda.Stream:
    s = _copy_streams.get(device.index)
    if s is None:
        s = torch.cuda.Stream(device=device)
        _copy_streams[device.index] = s
    return s


def _run(schedule: int, A, B, tp, alpha, beta, C, out, scale_a=1.0, scale_b=1.0):
    A3, B3 = _batched(A, "A"), _batched(B, "B")
    if not (A3.is_cuda and B3.is_cuda):
        raise ValueError("A and B must be CUDA tensors")
    L, M, K = A3.shape
    if B3.shape[0] != L or B3.shape[1] != K:
        raise ValueError(f"shape mismatch: A {tuple(A.shape)} @ B {tuple(B.shape)}")
    N = B3.shape[2]
    ta, tb = _in_type(A3), _in_type(B3)
    A3 = A3.contiguous()
    Bnk = _k_major_b(B3)
    dev = A3.device
    C3 = None
    if beta != 0.0:
        if C is None:
            raise ValueError("beta != 0 needs C")
        C3 = _batched(C, "C").to(torch.bfloat16).contiguous()
        if tuple(C3.shape) != (L, M, N):
            raise ValueError(f"C must be {(L, M, N)}, got {tuple(C3.shape)}")
    if out is None:
        out = torch.empty((L, M, N) if A.dim() == 3 else (M, N), dtype=torch.bfloat16, device=dev)
    D3 = _batched(out, "out")
    if tuple(D3.shape) != (L, M, N) or D3.dtype != torch.bfloat16 or not D3.is_contiguous():
        raise ValueError("out must be a contiguous bf16 tensor of the result's shape")
    key = (dev.index, schedule, M, N, K, L, tp, float(alpha), float(beta), ta, tb, float(scale_a), float(scale_b))
    with _lock:
        plan = _plans.get(key)
        if plan is None:
            plan = dg.Plan(M, N, K, L, tp, schedule, alpha, beta, ta, tb, scale_a, scale_b)
            _plans[key] = plan
        ws = _workspace(dev, plan.workspace_bytes())
        main = torch.cuda.current_stream(dev)
        plan.run(A3, Bnk, C3, D3, ws, main, _copy_stream(dev))
    return out


def fused_all_gather_matmul(A: torch.Tensor, B: torch.Tensor, tp: int, gather_dim: int = 0, *,
                            alpha: float = 1.0, beta: float = 0.0, C=None, out=None) -> torch.Tensor:
    """D = alpha * all_gather(A shards) @ B + beta * C over ``tp`` virtual ranks.

    ``gather_dim = 0``: A's rows are the sharded dimension and rotate between
    ranks (AllGather1D_TilingCD_RotatingA).  ``gather_dim = 1`` selects the
    other all-gather schedule, where B's columns rotate
    (AllGather1D_TilingCD_RotatingB).  M and N must divide by ``tp``.
    """
    sched = {0: dg.AG_ROTATING_A, 1: dg.AG_ROTATING_B}.get(gather_dim)
    if sched is None:
        raise ValueError("gather_dim must be 0 (rotate A) or 1 (rotate B)")
    return _run(sched, A, B, tp, alpha, beta, C, out)


def fused_matmul_reduce_scatter(A: torch.Tensor, B: torch.Tensor, tp: int, reduce_op: str = "sum",
                                scatter_dim: int = 0, *, alpha: float = 1.0, beta: float = 0.0, C=None,
                                out=None) -> torch.Tensor:
    """D = reduce_scatter(alpha * A_r @ B_r over ranks r) + beta * C.

    Rank r holds K-slab r of A and B; the partial products are summed with a
    rotating partial (the epilogue source), and rank j ends with slab j of D:
    M-slabs for ``scatter_dim = 0`` (ReduceScatter1D_TilingA_RotatingC), N-slabs
    for ``scatter_dim = 1`` (ReduceScatter1D_TilingB_RotatingC).  Only
    ``reduce_op = "sum"``.
    """
    if reduce_op != "sum":
        raise ValueError("reduce_op must be 'sum'")
    sched = {0: dg.RS_TILING_A_ROTATING_C, 1: dg.RS_TILING_B_ROTATING_C}.get(scatter_dim)
    if sched is None:
        raise ValueError("scatter_dim must be 0 (M-slabs) or 1 (N-slabs)")
    return _run(sched, A, B, tp, alpha, beta, C, out)


def _scale(s) -> float:
    # per-tensor scales: a Python number or a one-element tensor (read to the
    # host once; that read synchronizes with the tensor's stream)
    if isinstance(s, torch.Tensor):
        if s.numel() != 1:
            raise ValueError("only per-tensor (one-element) scales are supported")
        return float(s.item())
    return float(s)


def fused_all_gather_scaled_matmul(A: torch.Tensor, B: torch.Tensor, A_scale, B_scale, tp: int,
                                   gather_dim: int = 0, *, out=None) -> torch.Tensor:
    """fp8 (or bf16) all-gather matmul with per-tensor scales: A_scale * B_scale * (A @ B), bf16 out."""
    sched = {0: dg.AG_ROTATING_A, 1: dg.AG_ROTATING_B}.get(gather_dim)
    if sched is None:
        raise ValueError("gather_dim must be 0 or 1")
    return _run(sched, A, B, tp, 1.0, 0.0, None, out, _scale(A_scale), _scale(B_scale))


def fused_scaled_matmul_reduce_scatter(A: torch.Tensor, B: torch.Tensor, A_scale, B_scale, tp: int,
                                       reduce_op: str = "sum", scatter_dim: int = 0, *, out=None) -> torch.Tensor:
    """fp8 (or bf16) matmul-reduce-scatter with per-tensor scales, bf16 out."""
    if reduce_op != "sum":
        raise ValueError("reduce_op must be 'sum'")
    sched = {0: dg.RS_TILING_A_ROTATING_C, 1: dg.RS_TILING_B_ROTATING_C}.get(scatter_dim)
    if sched is None:
        raise ValueError("scatter_dim must be 0 or 1")
    return _run(sched, A, B, tp, 1.0, 0.0, None, out, _scale(A_scale), _scale(B_scale))


def clear_caches() -> None:
    """Drop cached plans, workspaces and copy streams."""
    with _lock:
        for p in _plans.values():
            p.close()
        _plans.clear()
        _workspaces.clear()
        _copy_streams.clear()
