"""CPU oracle of the four tensor-parallel schedules, rank by rank, step by step.

TEST INFRASTRUCTURE ONLY (see ``oracle/gemm.py``).  Small cases only: it
walks the virtual ranks and steps with Python loops over fp64 numpy blocks.

The pages name the schedules without defining them ("Distributed GEMM",
CUTLASS example 65 README, section "Trying out other schedules": the
All Gather + GEMM schedules ``AllGather1D_TilingCD_RotatingA`` and
``AllGather1D_TilingCD_RotatingB``, the GEMM + Reduce Scatter schedules
``ReduceScatter1D_TilingA_RotatingC`` and ``ReduceScatter1D_TilingB_RotatingC``).
The reading taken here, with P = TP virtual ranks, rank r, step s:

* AG-RotatingA.  Rank r holds rows M_r of A and columns N_r of B and owns
  D[:, N_r].  At step s it computes D[M_j, N_r], j = (r + s) mod P, with the
  A shard it has just received.  The rotation ``(step + rank) % group_size``
  is that of ``_pipelined_all_gather_and_consume`` in
  ``torch/distributed/_symmetric_memory/__init__.py``; the per-step local
  problem M/P x N/P x K is the "Local GEMM Problem Size" the CUTLASS
  pull request #1907 "Distributed GEMM" prints for TP=8 and TP=4.
* AG-RotatingB.  Same sharding; rank r owns D[M_r, :] and at step s computes
  D[M_r, N_j], j = (r + s) mod P, with the B shard it has just received.
* RS-TilingA-RotatingC.  Rank r holds columns K_r of A and rows K_r of B.  At
  step s it computes the partial for M-slab j = (r + s + 1) mod P and adds it
  to the rotating partial X_j it receives:
  X_j <- alpha * A[M_j, K_r] B[K_r, :] + (beta * C[M_j, :] if s == 0 else X_j).
  The last step (s = P - 1, j = r) leaves rank r its own slab: "produce
  chunk (rank + step) % group_size, own chunk last" in
  ``_pipelined_produce_and_all2all`` of the same torch module, with the
  separate ``reduce_fn`` replaced by the epilogue source ("use the epilogue
  source as the communication buffer", pull request #1907 description).
* RS-TilingB-RotatingC.  The same with N-slabs: X_j covers D[:, N_j].

Layouts as in ``oracle/gemm.py``: A (L, M, K), B stored (L, N, K), C and D
(L, M, N).  P must divide the sharded extents (the torch module raises on
shapes not divisible by the group size).

Parity status: pinned (tests/test_oracle_pins.py checks every schedule and
P against ``oracle.gemm.gemm``, the unsharded definition, and checks the
rotation tables against brute-force coverage and the printed local sizes).
"""

from __future__ import annotations

import numpy as np

AG_ROTATING_A = "AllGather1D_TilingCD_RotatingA"
AG_ROTATING_B = "AllGather1D_TilingCD_RotatingB"
RS_TILING_A_ROTATING_C = "ReduceScatter1D_TilingA_RotatingC"
RS_TILING_B_ROTATING_C = "ReduceScatter1D_TilingB_RotatingC"
SCHEDULES = (AG_ROTATING_A, AG_ROTATING_B, RS_TILING_A_ROTATING_C, RS_TILING_B_ROTATING_C)


def _slab(extent: int, P: int, j: int) -> slice:
    if extent % P:
        raise ValueError(f"extent {extent} not divisible by TP={P}")
    w = extent // P
    return slice(j * w, (j + 1) * w)


def slab_index(schedule: str, P: int, r: int, s: int) -> int:
    """Index j of the shard (AG) or output slab (RS) rank r handles at step s."""
    if schedule in (AG_ROTATING_A, AG_ROTATING_B):
        return (r + s) % P
    if schedule in (RS_TILING_A_ROTATING_C, RS_TILING_B_ROTATING_C):
        return (r + s + 1) % P
    raise ValueError(schedule)


def local_problem(schedule: str, m: int, n: int, k: int, l: int, P: int) -> tuple:
    """Per-rank, per-step GEMM extents (M, N, K, L)."""
    if schedule in (AG_ROTATING_A, AG_ROTATING_B):
        return (m // P, n // P, k, l)
    if schedule == RS_TILING_A_ROTATING_C:
        return (m // P, n, k // P, l)
    if schedule == RS_TILING_B_ROTATING_C:
        return (m, n // P, k // P, l)
    raise ValueError(schedule)


def step_blocks(schedule: str, m: int, n: int, k: int, P: int, r: int, s: int) -> dict:
    """Index ranges rank r touches at step s.

    Returns ``{"rows": slice over M, "cols": slice over N, "k": slice over K,
    "recv": which operand arrived from another rank ("A", "B", "C" or None)}``.
    """
    j = slab_index(schedule, P, r, s)
    full_m, full_n, full_k = slice(0, m), slice(0, n), slice(0, k)
    if schedule == AG_ROTATING_A:
        return {"rows": _slab(m, P, j), "cols": _slab(n, P, r), "k": full_k,
                "recv": "A" if j != r else None}
    if schedule == AG_ROTATING_B:
        return {"rows": _slab(m, P, r), "cols": _slab(n, P, j), "k": full_k,
                "recv": "B" if j != r else None}
    if schedule == RS_TILING_A_ROTATING_C:
        return {"rows": _slab(m, P, j), "cols": full_n, "k": _slab(k, P, r),
                "recv": "C" if s > 0 else None}
    if schedule == RS_TILING_B_ROTATING_C:
        return {"rows": full_m, "cols": _slab(n, P, j), "k": _slab(k, P, r),
                "recv": "C" if s > 0 else None}
    raise ValueError(schedule)


def run_schedule(schedule: str, A: np.ndarray, B_nk: np.ndarray, C, alpha: float,
                 beta: float, P: int, *, bias=None, reduce_op: str = "sum") -> np.ndarray:
    """D assembled from what every virtual rank computes at every step (fp64).

    For the RS schedules the partial X_j is carried from step to step exactly
    as the rotation prescribes; D receives X_j from the step that ends on the
    slab's owner.  ``bias`` (N,), if given, enters every block a rank
    computes (each rank's product carries it, as aten._scaled_mm adds it in
    the torch module's compositions); ``reduce_op`` "avg" weighs each rank's
    contribution to a rotating partial by 1/P, so the finished partial is
    the mean over ranks (torch.mean in ``_fused_matmul_reduce_scatter_impl``),
    beta C still entering once.
    """
    if reduce_op not in ("sum", "avg"):
        raise ValueError(f"reduce_op must be 'sum' or 'avg', got {reduce_op!r}")
    A = np.asarray(A, np.float64)
    B_nk = np.asarray(B_nk, np.float64)
    L, m, k = A.shape
    n = B_nk.shape[1]
    Cf = None if C is None else np.asarray(C, np.float64)
    bv = None if bias is None else np.asarray(bias, np.float64)
    D = np.full((L, m, n), np.nan)
    if schedule in (AG_ROTATING_A, AG_ROTATING_B):
        for s in range(P):
            for r in range(P):
                b = step_blocks(schedule, m, n, k, P, r, s)
                rows, cols = b["rows"], b["cols"]
                blk = np.float64(alpha) * np.matmul(A[:, rows, :], np.swapaxes(B_nk[:, cols, :], 1, 2))
                if bv is not None:
                    blk = blk + bv[cols]
                if beta != 0.0:
                    blk = blk + np.float64(beta) * Cf[:, rows, cols]
                D[:, rows, cols] = blk
        return D
    # ReduceScatter: one rotating partial per output slab.
    weight = np.float64(1.0) if reduce_op == "sum" else np.float64(1.0) / np.float64(P)
    X = {}
    for s in range(P):
        for r in range(P):
            j = slab_index(schedule, P, r, s)
            b = step_blocks(schedule, m, n, k, P, r, s)
            rows, cols, ks = b["rows"], b["cols"], b["k"]
            part = np.float64(alpha) * np.matmul(A[:, rows, ks], np.swapaxes(B_nk[:, cols, ks], 1, 2))
            if bv is not None:
                part = part + bv[cols]
            part = weight * part
            if s == 0:
                src = np.float64(beta) * Cf[:, rows, cols] if beta != 0.0 else 0.0
            else:
                src = X[j]
            X[j] = part + src
            if s == P - 1:
                assert j == r
                D[:, rows, cols] = X[j]
    return D


def rs_accumulation_order(schedule: str, P: int, j: int) -> list:
    """Ranks whose K-slabs are added into output slab j, in order."""
    order = []
    for s in range(P):
        for r in range(P):
            if slab_index(schedule, P, r, s) == j:
                order.append(r)
    return order
