"""The seeded input generator: both back ends give the same bits, subsets
equal slices of the whole, and the distributions have the stated shape."""

import numpy as np
import pytest
import torch

from reduce_scatter_gb300 import synth


def test_splitmix64_reference_values():
    # SplitMix64 from state 0: the first outputs of Vigna's splitmix64.c
    # (x += gamma; z = mix(x)), a standard published sequence.
    z = synth.raw_np(0, np.arange(3, dtype=np.uint64))
    assert [int(v) for v in z] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_bf16_rne():
    x = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, -2.5, 65504.0, 1e-40], np.float32)
    bits = synth.f32_to_bf16_bits_np(x)
    assert [int(b) for b in bits] == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x4780, 0x0001]


@pytest.mark.parametrize("dist", [("uniform", -1.0, 1.0), ("uniform", 0.0, 1.0), ("normal", 0.0, 1.0),
                                  ("normal", 0.0, 0.02)])
def test_numpy_and_torch_agree(dist):
    shape = (3, 37, 129)
    a = synth.tensor_bits_np(1, 2, shape, dist)
    b = synth.tensor_bits_torch(1, 2, shape, dist, chunk=1000).numpy().view(np.uint16)
    assert np.array_equal(a, b)


def test_rows_subset_equals_slice():
    dist = ("normal", 0.0, 1.0)
    full = synth.tensor_bits_np(5, 1, (2, 50, 33), dist).reshape(100, 33)
    rows = np.array([0, 17, 49, 50, 99])
    sub = synth.rows_bits_np(5, 1, (2, 50, 33), rows, dist)
    assert np.array_equal(sub, full[rows])


def test_streams_and_seeds_differ():
    d = ("uniform", -1.0, 1.0)
    a = synth.tensor_bits_np(1, 1, (64,), d)
    assert not np.array_equal(a, synth.tensor_bits_np(1, 2, (64,), d))
    assert not np.array_equal(a, synth.tensor_bits_np(2, 1, (64,), d))


def test_uniform_range_and_mean():
    for lo, hi in [(-1.0, 1.0), (0.0, 1.0)]:
        v = synth.bf16_bits_to_f32_np(synth.tensor_bits_np(3, 1, (200000,), ("uniform", lo, hi)))
        assert v.min() >= lo and v.max() < hi
        assert abs(v.mean() - (lo + hi) / 2) < 0.01 * (hi - lo)


def test_normal_moments():
    v = synth.bf16_bits_to_f32_np(synth.tensor_bits_np(3, 2, (200000,), ("normal", 0.0, 0.02))).astype(np.float64)
    assert abs(v.mean()) < 0.001
    assert abs(v.std() - 0.02) < 0.0005


@pytest.mark.parametrize("fmt,tdt", [("e4m3", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2)])
def test_fp8_quantizer_matches_torch_casts_in_range(fmt, tdt):
    top = synth.FP8_FORMATS[fmt][2]
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.normal(0, 1, 20000), rng.normal(0, 0.02, 20000), rng.normal(0, 100, 5000),
                        rng.uniform(-top, top, 5000), [0.0, -0.0, top, -top, 2.0 ** -9, 2.0 ** -10,
                                                       2.0 ** -17, 1.0625, 1.1875]]).astype(np.float32)
    x = x[np.abs(x) <= top]
    ours = synth.f32_to_fp8_bits_np(x, fmt)
    theirs = torch.from_numpy(x).to(tdt).view(torch.uint8).numpy()
    assert np.array_equal(ours, theirs)
    # saturation beyond the largest finite value (torch gives NaN there instead)
    assert synth.f32_to_fp8_bits_np(np.array([1e6, -1e6], np.float32), fmt).tolist() == \
        synth.f32_to_fp8_bits_np(np.array([top, -top], np.float32), fmt).tolist()


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("dist", [("normal", 0.0, 1.0), ("normal", 0.0, 0.02), ("uniform", -1.0, 1.0)])
def test_fp8_numpy_and_torch_agree(fmt, dist):
    shape = (2, 31, 77)
    a = synth.tensor_fp8_bits_np(4, 1, shape, dist, fmt)
    b = synth.tensor_fp8_bits_torch(4, 1, shape, dist, fmt, chunk=999).numpy()
    assert np.array_equal(a, b)
    rows = np.array([0, 5, 61])
    sub = synth.rows_fp8_bits_np(4, 1, shape, rows, dist, fmt)
    assert np.array_equal(sub, a.reshape(62, 77)[rows])
