"""CPU oracle for the tensor-parallel GEMM: the plain definition in fp64.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this
module; only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` use it.  It shares no code with the device path.

What every schedule computes ("Distributed GEMM", CUTLASS example 65 README,
section "Getting started": the ``--m --n --k --l --alpha --beta`` problem,
checked against "a single-device GEMM")::

    D[l, i, j] = alpha * sum_k A[l, i, k] * B[l, k, j] + beta * C[l, i, j]

Layouts (the pages do not fix them; this is the reading the device path
implements): A is (L, M, K) row-major; B is stored as (L, N, K), i.e. its
transpose, K innermost ("TN"); C and D are (L, M, N) row-major.

The bf16 inputs are widened exactly to fp64 and the sum is taken in fp64 by
one library matrix product (numpy ``matmul`` on float64), then scaled and
offset elementwise.  When ``beta == 0`` C is not read at all (BLAS
convention; the pages are silent), so NaNs in C do not reach D.

Parity status: pinned (tests/test_oracle_pins.py: ``bf16_bits_to_f64`` against
the format's definition on hand-decoded patterns and torch's own widening of
all 65,536 codes; ``gemm``: brute-force triple loop,
closed forms, the statistical mean printed on the all_gather+matmul blog
page, schedule invariance; ``fused_gemm``: a loop-by-loop restatement of the
torch module's per-rank composition, closed forms, schedule invariance with
a bias and both reduce ops; ``f64_to_fp8_bits``: every code round-trips,
midpoints go to the even code, saturation, torch's own conversion).
"""

from __future__ import annotations

import numpy as np


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16/int16) to float64."""
    b = np.asarray(bits)
    u = b.astype(np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def gemm(A: np.ndarray, B_nk: np.ndarray, C, alpha: float, beta: float) -> np.ndarray:
    """``alpha * A @ B + beta * C`` in fp64.

    A: (L, M, K); B_nk: (L, N, K) (B stored transposed); C: (L, M, N) or
    ``None`` (only allowed when ``beta == 0``).  All float64.  Returns (L, M, N).
    """
    A = np.asarray(A, dtype=np.float64)
    B_nk = np.asarray(B_nk, dtype=np.float64)
    if A.ndim != 3 or B_nk.ndim != 3:
        raise ValueError("A and B must be 3-D (L, rows, K)")
    L, M, K = A.shape
    if B_nk.shape[0] != L or B_nk.shape[2] != K:
        raise ValueError(f"shape mismatch A{A.shape} B{B_nk.shape}")
    D = np.float64(alpha) * np.matmul(A, np.swapaxes(B_nk, 1, 2))
    if beta != 0.0:
        if C is None:
            raise ValueError("beta != 0 needs C")
        D = D + np.float64(beta) * np.asarray(C, dtype=np.float64)
    return D


def gemm_entries(A_rows: np.ndarray, B_rows: np.ndarray, C_block, alpha: float,
                 beta: float) -> np.ndarray:
    """The same definition on a sample: rows i of A against rows j of B.

    A_rows: (R, K) fp64 rows of A (any batch), B_rows: (S, K) fp64 rows of the
    stored (N, K) B of the same batch, C_block: (R, S) or ``None``.  Returns
    the (R, S) block ``D[rows, cols]``.  Used to check outputs of problems too
    large to evaluate in full.
    """
    D = np.float64(alpha) * (np.asarray(A_rows, np.float64) @ np.asarray(B_rows, np.float64).T)
    if beta != 0.0:
        D = D + np.float64(beta) * np.asarray(C_block, dtype=np.float64)
    return D


def flops(m: int, n: int, k: int, l: int) -> float:
    """Algorithmic flop count of the whole problem: 2*M*N*K*L."""
    return 2.0 * m * n * k * l


# ------------------------------------------------------------ scaled fp8 GEMM
#
# The scaled variants on the pages (fused_all_gather_scaled_matmul and
# fused_scaled_matmul_reduce_scatter in torch/distributed/_symmetric_memory,
# which call aten._scaled_mm with A_scale and B_scale) multiply the fp8 product
# by the per-tensor scales:  D = alpha * scale_a * scale_b * (A B) + beta * C.
# Here in fp64 on the exactly decoded fp8 values.

# OCP fp8 formats: (mantissa bits, exponent bias); e4m3 is the "fn" variant
# (no infinities; S.1111.111 is NaN), e5m2 is IEEE-like (infinities, NaNs).
_FP8 = {"e4m3": (3, 7), "e5m2": (2, 15)}


def fp8_bits_to_f64(bits, fmt: str) -> np.ndarray:
    """Exact value of each fp8 code (uint8) in float64."""
    man, bias = _FP8[fmt]
    b = np.asarray(bits).astype(np.int64) & 0xFF
    sign = np.where(b & 0x80, -1.0, 1.0)
    exp_field = (b >> man) & ((1 << (7 - man)) - 1)
    mant = b & ((1 << man) - 1)
    sub = np.ldexp(mant.astype(np.float64), 1 - bias - man)
    nrm = np.ldexp(1.0 + mant / float(1 << man), exp_field - bias)
    val = sign * np.where(exp_field == 0, sub, nrm)
    top = (1 << (7 - man)) - 1
    if fmt == "e4m3":
        val = np.where((exp_field == top) & (mant == (1 << man) - 1), np.nan, val)
    else:
        val = np.where((exp_field == top) & (mant == 0), sign * np.inf, val)
        val = np.where((exp_field == top) & (mant != 0), np.nan, val)
    return val


def scaled_gemm(A, B_nk, C, alpha: float, beta: float, scale_a: float, scale_b: float) -> np.ndarray:
    """alpha * scale_a * scale_b * A @ B + beta * C in fp64 (A, B already decoded)."""
    A = np.asarray(A, dtype=np.float64)
    B_nk = np.asarray(B_nk, dtype=np.float64)
    D = (np.float64(alpha) * np.float64(scale_a) * np.float64(scale_b)) * np.matmul(A, np.swapaxes(B_nk, 1, 2))
    if beta != 0.0:
        D = D + np.float64(beta) * np.asarray(C, dtype=np.float64)
    return D


# ------------------------------------------------- bias and the reduce op
#
# The scaled fused ops of torch/distributed/_symmetric_memory/__init__.py take
# a per-column ``bias`` that aten._scaled_mm adds to every rank's product, and
# fused_matmul_reduce_scatter reduces the ranks' products with ``reduce_op``
# "sum" (torch.sum over ranks) or "avg" (torch.mean over ranks).  Their
# reference compositions (_fused_all_gather_scaled_matmul_fallback and
# _fused_scaled_matmul_reduce_scatter_fallback: one _scaled_mm per rank, then
# all-gather / reduce_scatter_tensor) fix what the result is.  In the
# reduce-scatter ops every rank adds the bias before the reduction; the ranks'
# K-slabs partition K, so sum_r A_r B_r = A B and
#
#   all-gather:            D = alpha A B + bias + beta C
#   reduce-scatter, sum:   D = alpha A B + P bias + beta C
#   reduce-scatter, avg:   D = (alpha A B + P bias) / P + beta C
#
# beta C belongs to the CUTLASS problem (``--beta``), not to the torch ops; it
# enters once, after the reduction.


def fused_gemm(A, B_nk, C, alpha: float, beta: float, *, P: int = 1, reduce_op=None,
               bias=None) -> np.ndarray:
    """The fused op's result in fp64, from its composition above.

    ``reduce_op`` None for the all-gather ops, "sum" or "avg" for the
    reduce-scatter ops over ``P`` ranks; ``bias`` None or an (N,) vector added
    to each output row of every rank's product.  A, B_nk, C as in ``gemm``.
    """
    if reduce_op not in (None, "sum", "avg"):
        raise ValueError(f"reduce_op must be None, 'sum' or 'avg', got {reduce_op!r}")
    A = np.asarray(A, dtype=np.float64)
    B_nk = np.asarray(B_nk, dtype=np.float64)
    D = np.float64(alpha) * np.matmul(A, np.swapaxes(B_nk, 1, 2))
    if bias is not None:
        copies = 1 if reduce_op is None else P
        D = D + np.float64(copies) * np.asarray(bias, dtype=np.float64)
    if reduce_op == "avg":
        D = D / np.float64(P)
    if beta != 0.0:
        if C is None:
            raise ValueError("beta != 0 needs C")
        D = D + np.float64(beta) * np.asarray(C, dtype=np.float64)
    return D


def fused_gemm_entries(A_rows, B_rows, C_block, alpha: float, beta: float, *, P: int = 1, reduce_op=None,
                       bias_cols=None) -> np.ndarray:
    """``fused_gemm`` on a sample: rows i of A against rows j of the stored
    (N, K) B (any one batch), ``C_block`` (R, S) or None, ``bias_cols`` the
    bias at those columns j (S,) or None.  Returns the (R, S) block of D."""
    if reduce_op not in (None, "sum", "avg"):
        raise ValueError(f"reduce_op must be None, 'sum' or 'avg', got {reduce_op!r}")
    D = np.float64(alpha) * (np.asarray(A_rows, np.float64) @ np.asarray(B_rows, np.float64).T)
    if bias_cols is not None:
        copies = 1 if reduce_op is None else P
        D = D + np.float64(copies) * np.asarray(bias_cols, dtype=np.float64)
    if reduce_op == "avg":
        D = D / np.float64(P)
    if beta != 0.0:
        D = D + np.float64(beta) * np.asarray(C_block, dtype=np.float64)
    return D


# ------------------------------------------------------- fp8 results
#
# fp8 outputs of the scaled ops (aten._scaled_mm with an fp8 out_dtype and a
# result scale): the fp32 result times the result scale, rounded to the
# nearest fp8 value -- ties to the even code -- and saturated at the largest
# finite magnitude.  Written here as a nearest-neighbour search over the 256
# codes of the format, decoded by fp8_bits_to_f64.


def f64_to_fp8_bits(x, fmt: str) -> np.ndarray:
    """The fp8 code nearest to each value (ties to the even code), saturating
    at the largest finite magnitude; the sign of zero is kept."""
    codes = np.arange(128, dtype=np.int64)
    vals = fp8_bits_to_f64(codes, fmt)
    ok = np.isfinite(vals)
    pos_codes, pos_vals = codes[ok], vals[ok]           # ascending with the code
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    i = np.clip(np.searchsorted(pos_vals, a), 1, len(pos_vals) - 1)
    lo, hi = pos_vals[i - 1], pos_vals[i]
    take_hi = (a - lo > hi - a) | ((a - lo == hi - a) & (pos_codes[i] % 2 == 0))
    code = np.where(take_hi, pos_codes[i], pos_codes[i - 1])
    code = np.where(a >= pos_vals[-1], pos_codes[-1], code)
    code = np.where(a <= pos_vals[0], pos_codes[0], code)
    return (code | (np.signbit(x).astype(np.int64) << 7)).astype(np.uint8)


def quantize_result(D, fmt: str, result_scale: float = 1.0) -> np.ndarray:
    """fp8 codes of result_scale * D (the definition above)."""
    return f64_to_fp8_bits(np.float64(result_scale) * np.asarray(D, dtype=np.float64), fmt)
