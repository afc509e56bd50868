"""Checks that pin the CPU oracle to facts outside itself.

Each check takes the oracle functions as arguments and raises
``AssertionError`` when they disagree with the fact it encodes.
``test_oracle_pins.py`` runs them on the real oracle;
``test_oracle_mutations.py`` runs them on oracles with planted mistakes and
expects at least one check to fail for every mistake.
"""

from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np

from reduce_scatter_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _bits_to_f64(bits):
    return synth.bf16_bits_to_f32_np(bits).astype(np.float64)


def _rand(seed, stream, shape, dist=("uniform", -1.0, 1.0)):
    return _bits_to_f64(synth.tensor_bits_np(seed, stream, shape, dist))


def _int_valued(seed, stream, shape, lo=-8, hi=8):
    """Small integers (exact in bf16); products and sums stay exact in fp64."""
    rng = np.random.default_rng(seed * 131 + stream)
    return rng.integers(lo, hi + 1, size=shape).astype(np.float64)


def brute_gemm(A, B_nk, C, alpha, beta):
    """Triple loop in Python floats (fp64), written apart from the oracle."""
    L, M, K = A.shape
    N = B_nk.shape[1]
    D = [[[0.0] * N for _ in range(M)] for _ in range(L)]
    for l in range(L):
        for i in range(M):
            for j in range(N):
                acc = 0.0
                for kk in range(K):
                    acc += float(A[l, i, kk]) * float(B_nk[l, j, kk])
                v = float(alpha) * acc
                if beta != 0.0:
                    v = v + float(beta) * float(C[l, i, j])
                D[l][i][j] = v
    return np.array(D, dtype=np.float64)


# ----------------------------------------------------------------- gemm pins

BRUTE_SHAPES = [(1, 1, 1, 1), (1, 3, 5, 7), (2, 4, 3, 9), (1, 8, 16, 5), (3, 2, 6, 4)]


def check_brute_force_exact(gemm):
    """Integer-valued inputs: every order of summation is exact, so equal bits."""
    for idx, (L, M, N, K) in enumerate(BRUTE_SHAPES):
        for alpha, beta in [(1.0, 0.0), (0.5, 1.0), (-2.0, 0.25), (0.0, 3.0)]:
            A = _int_valued(idx, 1, (L, M, K))
            B = _int_valued(idx, 2, (L, N, K))
            C = _int_valued(idx, 3, (L, M, N))
            got = gemm(A, B, C, alpha, beta)
            want = brute_gemm(A, B, C, alpha, beta)
            assert got.shape == want.shape, (got.shape, want.shape)
            assert np.array_equal(got, want), (L, M, N, K, alpha, beta)


def check_brute_force_random(gemm):
    """bf16 uniform inputs: agreement within the fp64 summation error bound."""
    for idx, (L, M, N, K) in enumerate(BRUTE_SHAPES):
        A = _rand(100 + idx, 1, (L, M, K))
        B = _rand(100 + idx, 2, (L, N, K))
        C = _rand(100 + idx, 3, (L, M, N))
        got = gemm(A, B, C, 0.75, -1.5)
        want = brute_gemm(A, B, C, 0.75, -1.5)
        # |error| <= gamma_K * sum|a||b| with gamma_K ~ K * 2^-53, plus the scaling steps.
        bound = (K + 4) * 2.0 ** -52 * (np.abs(A) @ np.abs(np.swapaxes(B, 1, 2)) * 0.75 + 1.5 * np.abs(C) + 1.0)
        assert np.all(np.abs(got - want) <= bound)


def check_closed_forms(gemm):
    L, M, N = 2, 5, 7
    for K in (1, 16, 256, 8192):
        ones_a = np.ones((L, M, K))
        ones_b = np.ones((L, N, K))
        C = _int_valued(7, 3, (L, M, N))
        # all-ones: D = K * alpha + beta * C
        D = gemm(ones_a, ones_b, C, 1.0, 0.0)
        assert np.array_equal(D, np.full((L, M, N), float(K)))
        D = gemm(ones_a, ones_b, C, 0.5, 1.0)
        assert np.array_equal(D, 0.5 * K + C)
    # identity B (N = K): D = alpha * A + beta * C
    K = 12
    A = _rand(8, 1, (L, M, K))
    C = _rand(8, 3, (L, M, K))
    eye = np.broadcast_to(np.eye(K), (L, K, K)).copy()
    assert np.array_equal(gemm(A, eye, None, 1.0, 0.0), A)
    assert np.array_equal(gemm(A, eye, C, 2.0, 0.5), 2.0 * A + 0.5 * C)
    # one-hot B: column n of D is column perm[n] of A
    N, K = 9, 6
    A = _rand(9, 1, (L, M, K))
    perm = np.array([3, 0, 5, 5, 1, 2, 4, 0, 3])
    onehot = np.zeros((L, N, K))
    onehot[:, np.arange(N), perm] = 1.0
    D = gemm(A, onehot, None, 1.0, 0.0)
    assert np.array_equal(D, A[:, :, perm])
    # alpha = 0 leaves beta * C; beta = 0 ignores NaNs in C
    Cn = np.full((L, M, N), np.nan)
    D = gemm(A, onehot, Cn, 1.0, 0.0)
    assert not np.any(np.isnan(D))
    Cr = _rand(9, 3, (L, M, N))
    assert np.array_equal(gemm(A, onehot, Cr, 0.0, 1.5), 1.5 * Cr)


def check_printed_mean(gemm):
    """The blog's printed output.mean() for U[0,1) inputs with K = 8192."""
    with open(os.path.join(GOLDEN, "blog_allgather_matmul_mean.json")) as f:
        g = json.load(f)
    K = g["gemm"]["k"]
    M, N = 96, 80
    dist = ("uniform", 0.0, 1.0)
    A = _bits_to_f64(synth.tensor_bits_np(1, 1, (1, M, K), dist))
    B = _bits_to_f64(synth.tensor_bits_np(1, 2, (1, N, K), dist))
    mean = float(gemm(A, B, None, 1.0, 0.0).mean())
    # Standard error of the mean of M*N entries that share rows and columns:
    # var(D_ij) = K * (E[a^2]E[b^2] - E[a]^2E[b]^2) = K * (1/9 - 1/16); rows and
    # columns are shared, so take the conservative sqrt(var / min(M, N)) * 3
    # plus the 2048-vs-printed gap.
    se = math.sqrt(K * (1.0 / 9 - 1.0 / 16) / min(M, N))
    assert abs(mean - g["printed_mean"]) <= 3 * se + abs(g["printed_mean"] - K / 4), (mean, se)
    # a dropped or doubled factor would move the mean by K/4 or more
    assert abs(mean - K / 4) < K / 64


# ------------------------------------------------------------- schedule pins


def check_schedule_invariance(run_schedule, gemm, schedules):
    """Every schedule and TP gives the unsharded D (the torch module's
    fallbacks define each fused op as collective-then-matmul)."""
    for P in (1, 2, 4, 8):
        L, M, N, K = 2, 2 * P, 3 * P, 4 * P
        A = _int_valued(P, 1, (L, M, K))
        B = _int_valued(P, 2, (L, N, K))
        C = _int_valued(P, 3, (L, M, N))
        for alpha, beta in [(1.0, 0.0), (0.5, 1.0), (2.0, -0.5)]:
            want = gemm(A, B, C, alpha, beta)
            for sched in schedules:
                got = run_schedule(sched, A, B, C, alpha, beta, P)
                assert np.array_equal(got, want), (sched, P, alpha, beta)
        # random bf16 inputs: equal up to fp64 rounding of the RS partial sums
        A = _rand(P, 1, (L, M, K))
        B = _rand(P, 2, (L, N, K))
        C = _rand(P, 3, (L, M, N))
        want = gemm(A, B, C, 0.5, 1.0)
        for sched in schedules:
            got = run_schedule(sched, A, B, C, 0.5, 1.0, P)
            assert np.allclose(got, want, rtol=0, atol=1e-12 * (np.abs(want).max() + 1)), (sched, P)


def check_rotation_tables(slab_index, step_blocks, schedules):
    """Rotation invariants the pages' loops fix, for P = 1..8:

    * each rank handles every shard / slab exactly once;
    * at every step the P ranks handle P distinct shards / slabs;
    * AG: step 0 consumes the local shard (no wait for a transfer);
    * RS: the last step ends on the owner's slab ("own chunk last"), and the
      partial of slab j moves from rank r at step s to rank r - 1 at step s+1
      (a ring, so each hand-off is one neighbour transfer);
    * the blocks of all (rank, step) pairs tile the (M, N, K) volume exactly once.
    """
    ag = schedules[:2]
    for P in range(1, 9):
        for sched in schedules:
            for r in range(P):
                js = [slab_index(sched, P, r, s) for s in range(P)]
                assert sorted(js) == list(range(P)), (sched, P, r, js)
            for s in range(P):
                js = [slab_index(sched, P, r, s) for r in range(P)]
                assert sorted(js) == list(range(P)), (sched, P, s)
            if sched in ag:
                assert all(slab_index(sched, P, r, 0) == r for r in range(P))
            else:
                assert all(slab_index(sched, P, r, P - 1) == r for r in range(P))
                for s in range(P - 1):
                    for r in range(P):
                        j = slab_index(sched, P, r, s)
                        assert slab_index(sched, P, (r - 1) % P, s + 1) == j
            m, n, k = 2 * P, 3 * P, 5 * P
            cover = np.zeros((m, n, k), dtype=np.int64)
            for r in range(P):
                for s in range(P):
                    b = step_blocks(sched, m, n, k, P, r, s)
                    cover[b["rows"], b["cols"], b["k"]] += 1
            assert np.all(cover == 1), (sched, P)


def check_printed_local_sizes(local_problem, schedule_ag_a):
    with open(os.path.join(GOLDEN, "pr1907_distgemm_printout.json")) as f:
        g = json.load(f)
    for run in g["runs"]:
        m, n, k, l = run["problem"]
        assert tuple(local_problem(schedule_ag_a, m, n, k, l, run["tp"])) == tuple(run["local_problem"])


def all_shapes():
    return list(itertools.product([1, 2], [1, 3], [2, 5]))


# ------------------------------------------------ bias and reduce-op pins


def brute_fused(A, B_nk, C, alpha, beta, P, reduce_op, bias):
    """The torch module's composition by loops, written apart from the oracle:
    each rank r takes the product over its own K-slab (all of K for the
    all-gather ops, reduce_op None), scales it by alpha and adds the bias (one
    aten._scaled_mm per rank); the ranks' results are summed or averaged;
    beta * C enters once."""
    L, M, K = A.shape
    N = B_nk.shape[1]
    ranks = 1 if reduce_op is None else P
    w = K // ranks
    D = np.zeros((L, M, N))
    for l in range(L):
        for i in range(M):
            for j in range(N):
                total = 0.0
                for r in range(ranks):
                    acc = 0.0
                    for kk in range(r * w, (r + 1) * w):
                        acc += float(A[l, i, kk]) * float(B_nk[l, j, kk])
                    v = float(alpha) * acc
                    if bias is not None:
                        v += float(bias[j])
                    total += v
                if reduce_op == "avg":
                    total /= P
                if beta != 0.0:
                    total += float(beta) * float(C[l, i, j])
                D[l, i, j] = total
    return D


def check_bias_reduce_brute_force(fused_gemm):
    """Integer-valued inputs, P a power of two: every result is exact."""
    for idx, (L, M, N) in enumerate([(1, 3, 5), (2, 4, 3)]):
        for P in (1, 2, 4):
            K = 2 * P
            A = _int_valued(40 + idx, 1, (L, M, K))
            B = _int_valued(40 + idx, 2, (L, N, K))
            C = _int_valued(40 + idx, 3, (L, M, N))
            bias = _int_valued(40 + idx, 4, (N,))
            for op in (None, "sum", "avg"):
                for alpha, beta, bv in [(1.0, 0.0, bias), (0.5, 1.0, bias), (2.0, -0.5, None)]:
                    got = fused_gemm(A, B, C, alpha, beta, P=P, reduce_op=op, bias=bv)
                    want = brute_fused(A, B, C, alpha, beta, P, op, bv)
                    assert np.array_equal(got, want), (L, M, N, P, op, alpha, beta, bv is None)


def check_bias_reduce_closed_forms(fused_gemm):
    L, M, N, K, P = 2, 3, 4, 8, 4
    bias = _int_valued(50, 4, (N,))
    C = _int_valued(50, 3, (L, M, N))
    zeros_a = np.zeros((L, M, K))
    B = _int_valued(50, 2, (L, N, K))
    # A = 0: only the bias copies and beta * C remain
    assert np.array_equal(fused_gemm(zeros_a, B, C, 1.0, 0.0, P=P, reduce_op=None, bias=bias),
                          np.broadcast_to(bias, (L, M, N)))
    assert np.array_equal(fused_gemm(zeros_a, B, C, 1.0, 0.5, P=P, reduce_op="sum", bias=bias),
                          P * bias + 0.5 * C)
    assert np.array_equal(fused_gemm(zeros_a, B, C, 1.0, 0.5, P=P, reduce_op="avg", bias=bias),
                          bias + 0.5 * C)
    # all-ones operands: alpha K plus the bias (AG), P bias (sum); avg is sum / P
    ones_a, ones_b = np.ones((L, M, K)), np.ones((L, N, K))
    assert np.array_equal(fused_gemm(ones_a, ones_b, None, 0.5, 0.0, P=P, reduce_op=None, bias=bias),
                          np.broadcast_to(0.5 * K + bias, (L, M, N)))
    s = fused_gemm(ones_a, ones_b, None, 0.5, 0.0, P=P, reduce_op="sum", bias=bias)
    assert np.array_equal(s, np.broadcast_to(0.5 * K + P * bias, (L, M, N)))
    assert np.array_equal(fused_gemm(ones_a, ones_b, None, 0.5, 0.0, P=P, reduce_op="avg", bias=bias), s / P)
    # no bias and no reduction: the plain definition
    A = _rand(51, 1, (L, M, K))
    Br = _rand(51, 2, (L, N, K))
    plain = np.float64(0.75) * np.matmul(A, np.swapaxes(Br, 1, 2)) + 1.5 * C
    assert np.array_equal(fused_gemm(A, Br, C, 0.75, 1.5), plain)


def check_schedule_bias_reduce(run_schedule, fused_gemm, schedules):
    """Every schedule and TP, with a bias and both reduce ops, gives the
    composition's result (exact on integer inputs)."""
    for P in (1, 2, 4, 8):
        L, M, N, K = 2, 2 * P, 3 * P, 4 * P
        A = _int_valued(60 + P, 1, (L, M, K))
        B = _int_valued(60 + P, 2, (L, N, K))
        C = _int_valued(60 + P, 3, (L, M, N))
        bias = _int_valued(60 + P, 4, (N,))
        for sched in schedules[:2]:
            got = run_schedule(sched, A, B, C, 0.5, 1.0, P, bias=bias)
            assert np.array_equal(got, fused_gemm(A, B, C, 0.5, 1.0, P=P, reduce_op=None, bias=bias)), (sched, P)
        for sched in schedules[2:]:
            for op in ("sum", "avg"):
                got = run_schedule(sched, A, B, C, 0.5, 1.0, P, bias=bias, reduce_op=op)
                want = fused_gemm(A, B, C, 0.5, 1.0, P=P, reduce_op=op, bias=bias)
                assert np.array_equal(got, want), (sched, P, op)


# ------------------------------------------------------- bf16 input decoding

# bfloat16 is the upper half of an IEEE-754 binary32: 1 sign bit, 8 exponent
# bits (bias 127) and 7 stored mantissa bits.  Hand-decoded patterns with the
# value each must widen to (NaN marked by None).
BF16_PATTERNS = [
    (0x0000, 0.0), (0x8000, -0.0), (0x3F80, 1.0), (0xBF80, -1.0), (0x4000, 2.0), (0xC040, -3.0),
    (0x3F00, 0.5), (0x4049, 3.140625), (0x0080, 2.0 ** -126),           # smallest normal
    (0x0001, 2.0 ** -133), (0x807F, -127 * 2.0 ** -133),               # subnormals
    (0x7F7F, (2.0 - 2.0 ** -7) * 2.0 ** 127),                            # largest finite
    (0x7F80, math.inf), (0xFF80, -math.inf), (0x7FC0, None), (0xFFC1, None),
]


def check_bf16_decode(decode, torch_decode):
    """``decode`` (bit patterns -> float64) against the format's definition on
    hand-written patterns (both as uint16 and as int16 input, so that a
    sign-extension slip shows), and against ``torch_decode`` (a library
    widening) on all 65,536 codes."""
    for bits, want in BF16_PATTERNS:
        for dtype in (np.uint16, np.int16):
            arr = np.array([bits], dtype=np.uint16).astype(dtype)
            got = float(np.asarray(decode(arr), dtype=np.float64).reshape(-1)[0])
            if want is None:
                assert math.isnan(got), (hex(bits), got)
            else:
                assert got == want and math.copysign(1.0, got) == math.copysign(1.0, want), (hex(bits), got, want)
    codes = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):  # signalling-NaN codes widen to quiet NaNs
        got = np.asarray(decode(codes), dtype=np.float64)
    want = np.asarray(torch_decode(codes), dtype=np.float64)
    assert got.shape == want.shape
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))
