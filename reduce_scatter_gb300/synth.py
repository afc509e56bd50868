"""Seeded synthetic inputs for the communication-fused TP GEMM.

This module only draws numbers. It holds none of the GEMM's arithmetic, so
both the CPU oracle (through its callers in ``tests/`` and ``bench.py``) and
the device path may take their inputs from it.

Generator
---------
Every tensor element is drawn from a counter-based SplitMix64 stream
(Steele, Lea and Flood, "Fast Splittable Pseudorandom Number Generators",
OOPSLA 2014; the mixing constants are those of Vigna's public-domain
``splitmix64.c``).  Element ``i`` (row-major flat index) of the tensor with
key ``key`` gets ``mix64(key + (i + 1) * GAMMA)``.  ``key`` is
``mix64(seed * 2**16 + stream)``, so each tensor (A, B, C) has its own
stream and any subset of elements can be drawn without drawing the rest.

From the 64-bit output ``z``:

* ``u24 = z >> 40`` gives a uniform on [0, 1) with 24 bits: ``u24 * 2**-24``.
* ``uniform(lo, hi)``: ``lo + (hi - lo) * u`` in fp64, rounded to fp32 and
  then to bf16 (both round-to-nearest-even).  A value that rounds up to
  ``hi`` is replaced by the largest bf16 below ``hi``, so the range stays
  half-open.
* ``normal(mean, std)``: Box-Muller on the pair of elements ``2i`` and
  ``2i+1`` of the stream: ``u1 = (u24(2i) + 1) * 2**-24`` in (0, 1],
  ``u2 = u24(2i+1) * 2**-24``;  ``mean + std * sqrt(-2 ln u1) cos(2 pi u2)``
  in fp64, rounded to fp32 and then bf16.

bf16 values travel as their uint16 bit patterns (numpy ``uint16`` or
torch ``int16``), so nothing here depends on a bf16 dtype.

Two back ends compute the same bits: numpy (uint64 arithmetic) for the CPU
side and torch (int64 two's-complement wrap-around, logical shifts by
masking) for tensors made directly on the device.  ``tests/test_synth.py``
checks that they agree bit for bit.
"""

from __future__ import annotations

import math

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB
_U64 = (1 << 64) - 1

# Tensor stream ids.
STREAM_A = 1
STREAM_B = 2
STREAM_C = 3
STREAM_BIAS = 4


def _mix64_int(z: int) -> int:
    z &= _U64
    z = ((z ^ (z >> 30)) * MIX1) & _U64
    z = ((z ^ (z >> 27)) * MIX2) & _U64
    return z ^ (z >> 31)


def stream_key(seed: int, stream: int) -> int:
    """64-bit key of tensor ``stream`` under ``seed``."""
    return _mix64_int(((seed & 0xFFFFFFFFFFFF) << 16) + (stream & 0xFFFF))


# ---------------------------------------------------------------- numpy side


def _mix64_np(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * np.uint64(MIX1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(MIX2)
        return z ^ (z >> np.uint64(31))


def raw_np(key: int, idx: np.ndarray) -> np.ndarray:
    """SplitMix64 outputs for flat indices ``idx`` (any integer array)."""
    i = np.asarray(idx, dtype=np.uint64)
    with np.errstate(over="ignore"):
        x = np.uint64(key) + (i + np.uint64(1)) * np.uint64(GAMMA)
    return _mix64_np(x)


def f32_to_bf16_bits_np(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16, nearest-even, returned as uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))
    return (b >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32_np(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _bf16_below(hi: float) -> int:
    """Bits of the largest bf16 strictly below ``hi`` (``hi`` a bf16 value)."""
    hb = int(f32_to_bf16_bits_np(np.array([hi], np.float32))[0])
    if hi > 0:
        return hb - 1
    if hi == 0:
        return 0x8001  # smallest negative subnormal
    return hb + 1


def uniform_bits_np(seed: int, stream: int, idx: np.ndarray, lo: float, hi: float) -> np.ndarray:
    z = raw_np(stream_key(seed, stream), idx)
    u = (z >> np.uint64(40)).astype(np.float64) * (2.0 ** -24)
    v = (lo + (hi - lo) * u).astype(np.float32)
    bits = f32_to_bf16_bits_np(v)
    over = bf16_bits_to_f32_np(bits) >= np.float32(hi)
    if np.any(over):
        bits = np.where(over, np.uint16(_bf16_below(hi)), bits)
    return bits


def normal_bits_np(seed: int, stream: int, idx: np.ndarray, mean: float, std: float) -> np.ndarray:
    i = np.asarray(idx, dtype=np.uint64)
    key = stream_key(seed, stream)
    z1 = raw_np(key, i * np.uint64(2))
    z2 = raw_np(key, i * np.uint64(2) + np.uint64(1))
    u1 = ((z1 >> np.uint64(40)).astype(np.float64) + 1.0) * (2.0 ** -24)
    u2 = (z2 >> np.uint64(40)).astype(np.float64) * (2.0 ** -24)
    n = np.sqrt(-2.0 * np.log(u1)) * np.cos((2.0 * math.pi) * u2)
    v = (mean + std * n).astype(np.float32)
    return f32_to_bf16_bits_np(v)


def draw_bits_np(seed: int, stream: int, idx: np.ndarray, dist: tuple) -> np.ndarray:
    """``dist`` is ``("uniform", lo, hi)`` or ``("normal", mean, std)``."""
    kind = dist[0]
    if kind == "uniform":
        return uniform_bits_np(seed, stream, idx, float(dist[1]), float(dist[2]))
    if kind == "normal":
        return normal_bits_np(seed, stream, idx, float(dist[1]), float(dist[2]))
    raise ValueError(f"unknown distribution {dist!r}")


def tensor_bits_np(seed: int, stream: int, shape: tuple, dist: tuple) -> np.ndarray:
    """Whole tensor of ``shape`` (row-major) as uint16 bf16 bits."""
    n = int(np.prod(shape)) if len(shape) else 1
    return draw_bits_np(seed, stream, np.arange(n, dtype=np.uint64), dist).reshape(shape)


def rows_bits_np(seed: int, stream: int, shape: tuple, rows: np.ndarray, dist: tuple) -> np.ndarray:
    """Selected rows of a tensor viewed as ``(prod(shape[:-1]), shape[-1])``.

    ``rows`` indexes the flattened leading dimensions.  Returns
    ``(len(rows), shape[-1])`` uint16 bits equal to the same rows of
    ``tensor_bits_np(seed, stream, shape, dist)``.
    """
    cols = int(shape[-1])
    rows = np.asarray(rows, dtype=np.uint64)
    idx = rows[:, None] * np.uint64(cols) + np.arange(cols, dtype=np.uint64)[None, :]
    return draw_bits_np(seed, stream, idx.reshape(-1), dist).reshape(len(rows), cols)


# ---------------------------------------------------------------- torch side


def _s64(v: int) -> int:
    """Unsigned 64-bit constant as the signed int64 with the same bits."""
    v &= _U64
    return v - (1 << 64) if v >= (1 << 63) else v


def _lsr(t, k: int):
    """Logical right shift of an int64 tensor."""
    return (t >> k) & ((1 << (64 - k)) - 1)


def _mix64_t(z):
    z = (z ^ _lsr(z, 30)) * _s64(MIX1)
    z = (z ^ _lsr(z, 27)) * _s64(MIX2)
    return z ^ _lsr(z, 31)


def _raw_t(key: int, idx):
    return _mix64_t((idx + 1) * _s64(GAMMA) + _s64(key))


def _f32_to_bf16_bits_t(v):
    import torch

    b = v.to(torch.float32).view(torch.int32).to(torch.int64) & 0xFFFFFFFF
    b = b + 0x7FFF + ((b >> 16) & 1)
    b = (b >> 16) & 0xFFFF
    return b.to(torch.int32).to(torch.int16)  # wraps to the same 16 bits


def _draw_t(seed: int, stream: int, idx, dist: tuple):
    import torch

    key = stream_key(seed, stream)
    kind = dist[0]
    if kind == "uniform":
        lo, hi = float(dist[1]), float(dist[2])
        u = _lsr(_raw_t(key, idx), 40).to(torch.float64) * (2.0 ** -24)
        v = (lo + (hi - lo) * u).to(torch.float32)
        bits = _f32_to_bf16_bits_t(v)
        back = ((bits.to(torch.int64) & 0xFFFF) << 16).to(torch.int32)
        over = back.view(torch.float32) >= hi
        below = _bf16_below(hi)
        below_s = below - 0x10000 if below >= 0x8000 else below
        return torch.where(over, torch.full_like(bits, below_s), bits)
    if kind == "normal":
        mean, std = float(dist[1]), float(dist[2])
        z1 = _raw_t(key, idx * 2)
        z2 = _raw_t(key, idx * 2 + 1)
        u1 = (_lsr(z1, 40).to(torch.float64) + 1.0) * (2.0 ** -24)
        u2 = _lsr(z2, 40).to(torch.float64) * (2.0 ** -24)
        n = torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)
        return _f32_to_bf16_bits_t(mean + std * n)
    raise ValueError(f"unknown distribution {dist!r}")


def tensor_bits_torch(seed: int, stream: int, shape: tuple, dist: tuple, device="cpu",
                      chunk: int = 1 << 26):
    """Same bits as :func:`tensor_bits_np`, as an int16 torch tensor on ``device``.

    Drawn in chunks of ``chunk`` elements to bound the int64 temporaries.
    """
    import torch

    n = 1
    for d in shape:
        n *= int(d)
    out = torch.empty(n, dtype=torch.int16, device=device)
    for start in range(0, n, chunk):
        stop = min(n, start + chunk)
        idx = torch.arange(start, stop, dtype=torch.int64, device=device)
        out[start:stop] = _draw_t(seed, stream, idx, dist)
    return out.view(*shape)


def bf16_view(t):
    """Reinterpret an int16 bit tensor as ``torch.bfloat16`` (no copy)."""
    import torch

    return t.view(torch.bfloat16)


# ------------------------------------------------------------------- fp8 inputs
#
# fp8 tensors are the same seeded fp32 draws rounded to an OCP fp8 format:
# e4m3 (the "fn" variant: bias 7, 3 mantissa bits, no infinities, largest
# finite 448) or e5m2 (bias 15, 2 mantissa bits, largest finite 57344).
# Rounding is to nearest, ties to even, on the value's own quantum (the
# subnormal quantum below the smallest normal); magnitudes beyond the largest
# finite value saturate to it.  All steps are exact float64 arithmetic on
# powers of two, so the numpy and torch versions give the same bits.

FP8_FORMATS = {"e4m3": (3, 7, 448.0), "e5m2": (2, 15, 57344.0)}


def f32_to_fp8_bits_np(x: np.ndarray, fmt: str) -> np.ndarray:
    man, bias, top = FP8_FORMATS[fmt]
    v = np.asarray(x, dtype=np.float32).astype(np.float64)
    sign = np.signbit(v)
    a = np.minimum(np.abs(v), top)
    _, e = np.frexp(np.where(a > 0, a, 1.0))          # a = f * 2**e, f in [0.5, 1)
    E = np.maximum(e - 1, 1 - bias)                  # exponent of the value's binade
    quantum = np.ldexp(1.0, E - man)
    q = np.minimum(np.rint(a / quantum) * quantum, top)
    _, e2 = np.frexp(np.where(q > 0, q, 1.0))
    E2 = e2 - 1
    normal = q >= np.ldexp(1.0, 1 - bias)
    sub_code = np.rint(q / np.ldexp(1.0, 1 - bias - man))
    mant = np.rint((q / np.ldexp(1.0, E2) - 1.0) * (1 << man))
    norm_code = (E2 + bias) * (1 << man) + mant
    code = np.where(normal, norm_code, sub_code).astype(np.int64)
    code = np.where(q == 0, 0, code)
    return (code | (sign.astype(np.int64) << 7)).astype(np.uint8)


def fp8_bits_to_f32_np(bits: np.ndarray, fmt: str) -> np.ndarray:
    """Decode (finite codes only; used by the generator's own checks)."""
    man, bias, _ = FP8_FORMATS[fmt]
    b = np.asarray(bits, dtype=np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    ef = (b >> man) & ((1 << (7 - man)) - 1)
    mf = b & ((1 << man) - 1)
    val = np.where(ef == 0, np.ldexp(mf.astype(np.float64), 1 - bias - man),
                   np.ldexp(1.0 + mf / (1 << man), ef - bias))
    return (sign * val).astype(np.float32)


def _f32_to_fp8_bits_t(v, fmt: str):
    import torch

    man, bias, top = FP8_FORMATS[fmt]
    v = v.to(torch.float32).to(torch.float64)
    sign = torch.signbit(v)
    a = torch.clamp(v.abs(), max=top)
    _, e = torch.frexp(torch.where(a > 0, a, torch.ones_like(a)))
    E = torch.clamp(e - 1, min=1 - bias).to(torch.float64)
    quantum = torch.pow(2.0, E - man)
    q = torch.clamp(torch.round(a / quantum) * quantum, max=top)
    _, e2 = torch.frexp(torch.where(q > 0, q, torch.ones_like(q)))
    E2 = (e2 - 1).to(torch.float64)
    normal = q >= 2.0 ** (1 - bias)
    sub_code = torch.round(q / 2.0 ** (1 - bias - man))
    mant = torch.round((q / torch.pow(2.0, E2) - 1.0) * (1 << man))
    norm_code = (E2 + bias) * (1 << man) + mant
    code = torch.where(normal, norm_code, sub_code).to(torch.int64)
    code = torch.where(q == 0, torch.zeros_like(code), code)
    code = code | (sign.to(torch.int64) << 7)
    return code.to(torch.uint8)


def _draw_f32_np(seed, stream, idx, dist):
    """fp32 value of a draw before its final rounding (uniform or normal)."""
    kind = dist[0]
    if kind == "uniform":
        lo, hi = float(dist[1]), float(dist[2])
        z = raw_np(stream_key(seed, stream), idx)
        u = (z >> np.uint64(40)).astype(np.float64) * (2.0 ** -24)
        return (lo + (hi - lo) * u).astype(np.float32)
    if kind == "normal":
        mean, std = float(dist[1]), float(dist[2])
        i = np.asarray(idx, dtype=np.uint64)
        key = stream_key(seed, stream)
        z1 = raw_np(key, i * np.uint64(2))
        z2 = raw_np(key, i * np.uint64(2) + np.uint64(1))
        u1 = ((z1 >> np.uint64(40)).astype(np.float64) + 1.0) * (2.0 ** -24)
        u2 = (z2 >> np.uint64(40)).astype(np.float64) * (2.0 ** -24)
        n = np.sqrt(-2.0 * np.log(u1)) * np.cos((2.0 * math.pi) * u2)
        return (mean + std * n).astype(np.float32)
    raise ValueError(f"unknown distribution {dist!r}")


def tensor_fp8_bits_np(seed: int, stream: int, shape: tuple, dist: tuple, fmt: str) -> np.ndarray:
    n = int(np.prod(shape)) if len(shape) else 1
    return f32_to_fp8_bits_np(_draw_f32_np(seed, stream, np.arange(n, dtype=np.uint64), dist), fmt).reshape(shape)


def rows_fp8_bits_np(seed: int, stream: int, shape: tuple, rows: np.ndarray, dist: tuple, fmt: str) -> np.ndarray:
    cols = int(shape[-1])
    rows = np.asarray(rows, dtype=np.uint64)
    idx = rows[:, None] * np.uint64(cols) + np.arange(cols, dtype=np.uint64)[None, :]
    return f32_to_fp8_bits_np(_draw_f32_np(seed, stream, idx.reshape(-1), dist), fmt).reshape(len(rows), cols)


def _draw_f32_t(seed: int, stream: int, idx, dist: tuple):
    import torch

    key = stream_key(seed, stream)
    kind = dist[0]
    if kind == "uniform":
        lo, hi = float(dist[1]), float(dist[2])
        u = _lsr(_raw_t(key, idx), 40).to(torch.float64) * (2.0 ** -24)
        return (lo + (hi - lo) * u).to(torch.float32)
    if kind == "normal":
        mean, std = float(dist[1]), float(dist[2])
        u1 = (_lsr(_raw_t(key, idx * 2), 40).to(torch.float64) + 1.0) * (2.0 ** -24)
        u2 = _lsr(_raw_t(key, idx * 2 + 1), 40).to(torch.float64) * (2.0 ** -24)
        n = torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)
        return (mean + std * n).to(torch.float32)
    raise ValueError(f"unknown distribution {dist!r}")


def tensor_fp8_bits_torch(seed: int, stream: int, shape: tuple, dist: tuple, fmt: str, device="cpu",
                          chunk: int = 1 << 26):
    """Same bits as :func:`tensor_fp8_bits_np`, as a uint8 torch tensor on ``device``."""
    import torch

    n = 1
    for d in shape:
        n *= int(d)
    out = torch.empty(n, dtype=torch.uint8, device=device)
    for start in range(0, n, chunk):
        stop = min(n, start + chunk)
        idx = torch.arange(start, stop, dtype=torch.int64, device=device)
        out[start:stop] = _f32_to_fp8_bits_t(_draw_f32_t(seed, stream, idx, dist), fmt)
    return out.view(*shape)
