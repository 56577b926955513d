"""Pins of the seeded input generator (no GPU)."""

import math

import numpy as np
import pytest
import torch

from exact_attention_95_gb300 import inputs


def test_splitmix64_reference_words():
    # First outputs of SplitMix64 seeded with 0, as published with the
    # generator's reference implementation.
    w = inputs.splitmix64(0, 0, 3)
    assert [int(x) for x in w] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_stream_offsets_are_consistent():
    a = inputs.splitmix64(1234, 0, 100)
    b = inputs.splitmix64(1234, 40, 60)
    np.testing.assert_array_equal(a[40:], b)
    x = inputs.normals(77, 0, 1000)
    y = inputs.normals(77, 500, 500)
    np.testing.assert_array_equal(x[500:], y)


def test_normals_statistics():
    x = inputs.normals(5, 0, 1 << 18)
    assert abs(x.mean()) < 0.01
    assert abs(x.var() - 1) < 0.01
    assert abs((np.abs(x) < 1).mean() - math.erf(1 / math.sqrt(2))) < 0.005


def test_bf16_rounding_is_round_to_nearest_even():
    # Compare with torch's fp32 -> bf16 conversion (RNE) on values exactly
    # representable in fp32 (no double rounding possible), including ties.
    vals = np.array([1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, -1 - 2 ** -8, 1 + 2 ** -9, 3.14159,
                     -2.71828, 1e-3, 65504.0, 1 + 2 ** -8 + 2 ** -20], dtype=np.float64)
    mine = inputs.round_to_bf16_bits(vals)
    ref = torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy()
    np.testing.assert_array_equal(mine.view(np.int16), ref)
    # Ties to even: 1 + 2^-8 lies halfway between 1 and 1 + 2^-7 -> 1.
    assert inputs.bf16_bits_to_f64(inputs.round_to_bf16_bits(np.array([1 + 2 ** -8])))[0] == 1.0


def test_bf16_rounding_single_step_from_fp64():
    # A value just above a tie in fp64 but that rounds to the tie in fp32 must
    # round up (single rounding), where fp64->fp32->bf16 would round to even.
    v = np.array([1 + 2 ** -8 + 2 ** -40])
    assert inputs.bf16_bits_to_f64(inputs.round_to_bf16_bits(v))[0] == 1 + 2 ** -7


def test_make_tensor_bf16_and_mul():
    t = inputs.make_tensor(99, (2, 3, 16, 8), "bf16")
    t8 = inputs.make_tensor(99, (2, 3, 16, 8), "bf16", mul=8.0)
    np.testing.assert_array_equal(inputs.to_f64(t) * 8, inputs.to_f64(t8))
    ref = inputs.round_to_bf16_bits(inputs.normals(99, 0, t.size)).reshape(t.shape)
    np.testing.assert_array_equal(t, ref)
    # chunked generation is identical to one pass
    t2 = inputs.make_tensor(99, (2, 3, 16, 8), "bf16", chunk=50)
    np.testing.assert_array_equal(t, t2)


def test_workloads_and_seeds():
    w = inputs.WORKLOADS["c3"]
    assert (w.B, w.Hq, w.N, w.d, w.causal, w.q_mul) == (2, 32, 4096, 128, True, 8.0)
    assert inputs.tensor_seed(3, "dO") == 0x5EED0000 + 48 + 3
    assert w.fwd_flops() == 4 * 4096 ** 2 * 128 * 32 * 2 / 2
    assert inputs.WORKLOADS["c4"].shape("K") == (1, 8, 16384, 128)


def test_sample_rows():
    r = inputs.sample_rows(3, 1000, 64, must=[0, 1, 999])
    assert len(r) == 64 and len(set(r.tolist())) == 64
    assert {0, 1, 999} <= set(r.tolist())
    np.testing.assert_array_equal(r, inputs.sample_rows(3, 1000, 64, must=[0, 1, 999]))
    assert len(inputs.sample_rows(1, 5, 64)) == 5


def test_make_tensor_rejects_inexact_multiplier():
    with pytest.raises(ValueError):
        inputs.make_tensor(1, (4,), "bf16", mul=3.0)


def test_blocky_tensor_is_exact_and_seeded():
    a = inputs.make_blocky_tensor(7, (2, 3, 300, 16), exps=(-2, 0, 3))
    b = inputs.make_blocky_tensor(7, (2, 3, 300, 16), exps=(-2, 0, 3))
    assert np.array_equal(a, b)
    base = inputs.bf16_bits_to_f64(inputs.make_tensor(7, (2, 3, 300, 16), "bf16"))
    x = inputs.bf16_bits_to_f64(a)
    # Each 128-row block is the base times one power of two from the set.
    ratio = x.reshape(6, 300, 16) / base.reshape(6, 300, 16)
    for h in range(6):
        for t in range(3):
            r = np.unique(ratio[h, 128 * t:128 * (t + 1)])
            assert r.size == 1 and r[0] in (0.25, 1.0, 8.0)


def test_random_block_mask_density_and_seed():
    m = inputs.random_block_mask(11, 2, 64, 0.5)
    assert m.dtype == np.uint8 and m.shape == (2, 64, 64)
    assert np.array_equal(m, inputs.random_block_mask(11, 2, 64, 0.5))
    assert abs(m.mean() - 0.5) < 0.02
    assert inputs.random_block_mask(11, 1, 8, 0.0).sum() == 0
    assert inputs.random_block_mask(11, 1, 8, 1.0).sum() == 64
