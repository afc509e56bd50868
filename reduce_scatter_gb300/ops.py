"""torch-tensor front end of the C ABI with the signatures of the fused ops in
torch/distributed/_symmetric_memory/__init__.py: ``fused_all_gather_matmul``,
``fused_all_gather_scaled_matmul``, ``fused_matmul_reduce_scatter``,
``fused_scaled_matmul_reduce_scatter`` and the two ``restride_*`` helpers.

Every TP rank is emulated on the one GPU, so where the torch op takes one
rank's tensors and a process group, the call here takes ALL ``tp`` virtual
ranks' tensors at once and ``tp`` in place of the group name:

* all-gather ops: ``A`` is the ranks' shards concatenated along
  ``gather_dim`` (so it is also the gathered A, returned as the first
  result); each ``B`` in ``Bs`` is the ranks' local (K, N_r) weights
  concatenated along N.  Result i holds every rank's ``A @ Bs[i]``: rank r's
  is the r-th block of its last dimension.
* reduce-scatter ops: ``A`` (..., K) and ``B`` (K, N) are the ranks' K-slabs
  concatenated (A along its last dimension, B along its first).  The result,
  of shape ``[*A.shape[:-1], N]``, holds every rank's reduced slab: rank r's
  is the r-th block of ``scatter_dim``.  ``scatter_dim`` may also name the
  output's last dimension (N), which selects the N-slab schedule.

Leading dimensions are handled as in the torch module: the sharded dimension
is moved to the front and the rest flattened into the rows of an (M, K)
matrix (one copy of A unless ``A.movedim(dim, 0)`` is already contiguous;
``restride_A_shard_for_fused_all_gather_matmul`` /
``restride_A_for_fused_matmul_reduce_scatter`` give A that layout), and the
output is unflattened the same way.  B is read K-major: a ``W.t()`` view of a
contiguous (N, K) ``W`` is used in place, any other B is copied once.

This module only marshals arguments: plans, workspaces and copy streams are
cached, outputs allocated with torch, and every step of the computation runs
in ``libdg.so``.  Beyond the torch ops, the non-scaled calls accept
``alpha``/``beta`` and a C operand (the CUTLASS problem's epilogue), and the
all-gather calls ``rotate="B"`` (AllGather1D_TilingCD_RotatingB: the ranks
keep their rows of A and the B shards rotate instead).
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

_OUT_TYPES = {torch.bfloat16: dg.TYPE_BF16, torch.float32: dg.TYPE_F32}
_OUT_TYPES.update(_FP8)


def _in_type(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return dg.TYPE_BF16
    if t.dtype in _FP8:
        return _FP8[t.dtype]
    raise TypeError(f"inputs must be bfloat16 or float8 (e4m3fn / e5m2), got {t.dtype}")


def _out_type(dtype) -> int:
    if dtype not in _OUT_TYPES:
        raise ValueError(f"out_dtype must be bfloat16, float32 or a float8 type, got {dtype}")
    return _OUT_TYPES[dtype]


def _k_major_b(B: torch.Tensor) -> torch.Tensor:
    """(K, N) B as an (N, K) tensor with K contiguous, without a copy when possible."""
    if B.dim() != 2:
        raise ValueError("B must be a matrix")
    Bt = B.t()
    return Bt if Bt.is_contiguous() else Bt.contiguous()


def _rows(A: torch.Tensor, dim: int, what: str, tp: int = 1):
    """A (..., K) as an (M, K) matrix with dimension ``dim`` outermost, and the
    leading shape to unflatten the output with.  Rank r's shard of ``dim`` is
    then the r-th block of M/tp rows."""
    if A.dim() < 2:
        raise ValueError("A must be a matrix")
    if dim < 0 or dim >= A.dim() - 1:
        raise ValueError(f"invalid {what}")
    if A.shape[dim] % tp:
        raise ValueError(f"{what} extent {A.shape[dim]} is not divisible by tp={tp}")
    x = A.movedim(dim, 0)
    lead = list(x.shape[:-1])
    return x.reshape(-1, x.shape[-1]).contiguous(), lead


def _unflatten(D2: torch.Tensor, lead: list, dim: int) -> torch.Tensor:
    return D2.view(*lead, D2.shape[-1]).movedim(0, dim)


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


def _scale(s) -> float:
    # per-tensor scales: a Python number or a one-element tensor (read to the
    # host once; that read synchronizes with the tensor's stream)
    if s is None:
        return 1.0
    if isinstance(s, torch.Tensor):
        if s.numel() != 1:
            raise ValueError("only per-tensor (one-element) scales are supported")
        return float(s.item())
    return float(s)


_SLOT_LAYOUT = ("off_slots", "slot_bytes", "chunk_tiles", "chunks_per_shard", "tile_m", "elem_bytes")


def _gemm(schedule: int, A2: torch.Tensor, B: torch.Tensor, tp: int, *, alpha=1.0, beta=0.0, C2=None,
          bias=None, out_dtype=torch.bfloat16, reduce_op="sum", scale_a=1.0, scale_b=1.0, result_scale=1.0,
          after=None):
    """One run of the C ABI on an (M, K) A and a (K, N) B; returns (M, N) D and
    a handle for ``after``.

    ``after``: the handle of a run on the same A just before (AllGather
    RotatingA).  When this plan lays out its receive slots like that run's,
    this run reads the shards that run moved (GEMM_ONLY on its workspace), so
    the A shards cross once for several Bs.
    """
    if not (A2.is_cuda and B.is_cuda):
        raise ValueError("A and B must be CUDA tensors")
    M, K = A2.shape
    if B.shape[0] != K:
        raise ValueError(f"shape mismatch: A (.., {K}) @ B {tuple(B.shape)}")
    N = B.shape[1]
    ta, tb = _in_type(A2), _in_type(B)
    to = _out_type(out_dtype)
    op = dg.REDUCE_BY_NAME[reduce_op]
    Bnk = _k_major_b(B)
    dev = A2.device
    if beta != 0.0:
        if C2 is None:
            raise ValueError("beta != 0 needs C")
        C2 = C2.to(torch.bfloat16).contiguous()
        if tuple(C2.shape) != (M, N):
            raise ValueError(f"C must hold {M} x {N} values")
    else:
        C2 = None
    if bias is not None:
        bias = bias.to(device=dev, dtype=torch.bfloat16).contiguous()
        if bias.dim() != 1 or bias.shape[0] != N:
            raise ValueError(f"bias must be a vector of {N} values")
    D2 = torch.empty((M, N), dtype=out_dtype, device=dev)
    rs = float(result_scale) if to in (dg.TYPE_E4M3, dg.TYPE_E5M2) else 1.0
    key = (dev.index, schedule, M, N, K, tp, float(alpha), float(beta), ta, tb, float(scale_a), float(scale_b),
           to, op, rs)
    if Bnk.device != dev or (C2 is not None and C2.device != dev) or (bias is not None and bias.device != dev):
        raise ValueError("A, B, C and bias must be on the same device")
    with _lock, torch.cuda.device(dev):  # the library works on the current device
        plan = _plans.get(key)
        if plan is None:
            plan = dg.Plan(M, N, K, 1, tp, schedule, alpha, beta, ta, tb, scale_a, scale_b, out_type=to,
                           reduce_op=op, result_scale=rs)
            _plans[key] = plan
        info = plan.info()
        main = torch.cuda.current_stream(dev)
        reuse = (after is not None and schedule == dg.AG_ROTATING_A and tp > 1 and after["A"] is A2
                 and all(after["info"][f] == info[f] for f in _SLOT_LAYOUT)
                 and after["ws"].numel() >= plan.workspace_bytes())
        if reuse:
            ws = after["ws"]
            plan.set_mode(dg.MODE_GEMM_ONLY)
            try:
                plan.run_ex(A2, Bnk, C2, bias, D2, ws, main, _copy_stream(dev))
            finally:
                plan.set_mode(dg.MODE_FUSED)
        else:
            ws = _workspace(dev, plan.workspace_bytes())
            plan.run_ex(A2, Bnk, C2, bias, D2, ws, main, _copy_stream(dev))
    return D2, {"A": A2, "ws": ws, "info": info}


def _ag_schedule(rotate: str) -> int:
    sched = {"A": dg.AG_ROTATING_A, "B": dg.AG_ROTATING_B}.get(rotate)
    if sched is None:
        raise ValueError("rotate must be 'A' (AllGather1D_TilingCD_RotatingA) or 'B' (..._RotatingB)")
    return sched


def fused_all_gather_matmul(A: torch.Tensor, Bs, gather_dim: int, tp: int, *, rotate: str = "A",
                            alpha: float = 1.0, beta: float = 0.0, Cs=None):
    """``all_gather(A shards, gather_dim) @ B`` for every B in ``Bs``, over
    ``tp`` virtual ranks; returns ``(A, [outputs])`` like the torch op.

    The first B runs fused (its shard transfers overlapped with the GEMM);
    with rotate="A" the later Bs read the A shards that run moved, so A
    crosses once for all Bs as in the torch op.  ``Cs`` (one per B, shaped
    like its output) enters as ``beta * C`` when ``beta != 0``.
    """
    sched = _ag_schedule(rotate)
    Bs = list(Bs)
    if Cs is not None and len(Cs) != len(Bs):
        raise ValueError("len(Cs) must be the same as len(Bs)")
    A2, lead = _rows(A, gather_dim, "gather_dim", tp)
    outs, prev = [], None
    for i, B in enumerate(Bs):
        C2 = None
        if beta != 0.0:
            if Cs is None:
                raise ValueError("beta != 0 needs Cs")
            C2, _ = _rows(Cs[i], gather_dim, "gather_dim")
        D2, prev = _gemm(sched, A2, B, tp, alpha=alpha, beta=beta, C2=C2, after=prev)
        outs.append(_unflatten(D2, lead, gather_dim))
    return A, outs


def fused_all_gather_scaled_matmul(A: torch.Tensor, Bs, A_scale, B_scales, gather_dim: int, tp: int,
                                   biases=None, result_scales=None, out_dtypes=None, use_fast_accum=None, *,
                                   rotate: str = "A"):
    """fp8 (or bf16) all-gather matmuls with per-tensor scales:
    ``A_scale * B_scales[i] * (A @ Bs[i]) + biases[i]``; returns ``(A, [outputs])``.

    ``out_dtypes[i]``: None (the dtype of ``Bs[i]``, as in the torch op),
    bfloat16, float32 or a float8 type; an fp8 output holds
    ``result_scales[i] * value`` rounded to the format (nearest, saturating).
    ``use_fast_accum`` is accepted and has no effect: the tensor cores always
    accumulate in fp32.
    """
    sched = _ag_schedule(rotate)
    Bs = list(Bs)
    n = len(Bs)
    B_scales = list(B_scales)
    biases = [None] * n if biases is None else list(biases)
    result_scales = [None] * n if result_scales is None else list(result_scales)
    out_dtypes = [None] * n if out_dtypes is None else list(out_dtypes)
    use_fast_accum = [False] * n if use_fast_accum is None else list(use_fast_accum)
    for name, lst in (("B_scales", B_scales), ("biases", biases), ("result_scales", result_scales),
                      ("out_dtypes", out_dtypes), ("use_fast_accum", use_fast_accum)):
        if len(lst) != n:
            raise ValueError(f"len({name}) must be the same as len(Bs)")
    sa = _scale(A_scale)
    A2, lead = _rows(A, gather_dim, "gather_dim", tp)
    outs, prev = [], None
    for B, sb, bias, rsc, dt in zip(Bs, B_scales, biases, result_scales, out_dtypes):
        D2, prev = _gemm(sched, A2, B, tp, bias=bias, out_dtype=dt if dt is not None else B.dtype, scale_a=sa,
                         scale_b=_scale(sb), result_scale=_scale(rsc), after=prev)
        outs.append(_unflatten(D2, lead, gather_dim))
    return A, outs


def _rs_layout(A: torch.Tensor, scatter_dim: int, tp: int):
    if A.dim() < 2:
        raise ValueError("A must be a matrix")
    if scatter_dim < 0 or scatter_dim >= A.dim():
        raise ValueError("invalid scatter_dim")
    if scatter_dim == A.dim() - 1:
        # the output's last dimension (N) is scattered: N-slabs
        return dg.RS_TILING_B_ROTATING_C, A.reshape(-1, A.shape[-1]).contiguous(), list(A.shape[:-1]), None
    A2, lead = _rows(A, scatter_dim, "scatter_dim", tp)
    return dg.RS_TILING_A_ROTATING_C, A2, lead, scatter_dim


def _rs_result(D2: torch.Tensor, lead: list, dim) -> torch.Tensor:
    if dim is None:
        return D2.view(*lead, D2.shape[-1])
    return _unflatten(D2, lead, dim)


def fused_matmul_reduce_scatter(A: torch.Tensor, B: torch.Tensor, reduce_op: str, scatter_dim: int, tp: int, *,
                                alpha: float = 1.0, beta: float = 0.0, C=None) -> torch.Tensor:
    """``reduce_scatter(A_r @ B_r over the tp ranks, reduce_op, scatter_dim)``:
    every rank's product over its K-slab, summed ("sum") or averaged ("avg")
    through the rotating partial, each rank ending with its slab.

    ``alpha`` scales every rank's product; ``beta * C`` (C shaped like the
    result) enters once.
    """
    if reduce_op not in ("sum", "avg"):
        raise ValueError("reduce_op must be sum or avg")
    sched, A2, lead, dim = _rs_layout(A, scatter_dim, tp)
    C2 = None
    if beta != 0.0:
        if C is None:
            raise ValueError("beta != 0 needs C")
        C2 = C.reshape(-1, C.shape[-1]) if dim is None else _rows(C, dim, "scatter_dim")[0]
    D2, _ = _gemm(sched, A2, B, tp, alpha=alpha, beta=beta, C2=C2, reduce_op=reduce_op)
    return _rs_result(D2, lead, dim)


def fused_scaled_matmul_reduce_scatter(A: torch.Tensor, B: torch.Tensor, A_scale, B_scale, reduce_op: str,
                                       scatter_dim: int, tp: int, bias=None, result_scale=None, out_dtype=None,
                                       use_fast_accum: bool = False) -> torch.Tensor:
    """fp8 (or bf16) matmul-reduce-scatter with per-tensor scales: each rank's
    ``A_scale * B_scale * (A_r @ B_r) + bias``, reduced over the ranks (so a
    "sum" carries tp copies of the bias, an "avg" one, as in the torch module's
    reference composition).  ``out_dtype``: None (A's dtype, as in the torch
    op), bfloat16, float32 or a float8 type (then ``result_scale * value``
    rounded to the format; the partials stay fp32 until the last step);
    ``use_fast_accum`` has no effect.
    """
    if reduce_op not in ("sum", "avg"):
        raise ValueError("reduce_op must be sum or avg")
    sched, A2, lead, dim = _rs_layout(A, scatter_dim, tp)
    D2, _ = _gemm(sched, A2, B, tp, bias=bias, out_dtype=out_dtype if out_dtype is not None else A.dtype,
                  reduce_op=reduce_op, scale_a=_scale(A_scale), scale_b=_scale(B_scale),
                  result_scale=_scale(result_scale))
    return _rs_result(D2, lead, dim)


def _dim_outermost(t: torch.Tensor, dim: int) -> torch.Tensor:
    """A copy of ``t`` (same shape and values) whose memory holds dimension
    ``dim`` outermost and the others in their order, so that
    ``result.movedim(dim, 0)`` is contiguous."""
    if dim < 0 or dim >= t.dim():
        raise ValueError("invalid dim")
    buf = torch.empty((t.shape[dim], *[s for d, s in enumerate(t.shape) if d != dim]), dtype=t.dtype,
                      device=t.device)
    out = buf.movedim(0, dim)
    out.copy_(t)
    return out


def restride_A_shard_for_fused_all_gather_matmul(t: torch.Tensor, gather_dim: int) -> torch.Tensor:
    """``t`` laid out so that the all-gather ops read it without a layout copy."""
    return _dim_outermost(t, gather_dim)


def restride_A_for_fused_matmul_reduce_scatter(t: torch.Tensor, scatter_dim: int) -> torch.Tensor:
    """``t`` laid out so that the reduce-scatter ops read it without a layout copy."""
    return _dim_outermost(t, scatter_dim)


def clear_caches() -> None:
    """Drop cached plans, workspaces and copy streams."""
    with _lock:
        for p in _plans.values():
            p.close()
        _plans.clear()
        _workspaces.clear()
        _copy_streams.clear()
