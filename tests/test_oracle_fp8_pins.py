"""Pins of the reference e4m3 block quantizer (CPU only).

Checked against the e4m3 format itself, not against the quantizer's own
formula: every one of the 256 codes decodes to its value and re-encodes to
itself; the landmark values (largest finite 448, smallest normal 2^-6,
smallest subnormal 2^-9, the 8 values of the binade [1, 2)); ties round to
even; saturation at 448; and a block's dequantized values stay within half a
unit in the last place of the input.
"""

import numpy as np

from oracle import fp8


def test_all_codes_roundtrip():
    codes = np.arange(256, dtype=np.uint8)
    vals = fp8.decode_e4m3(codes)
    ok = ~np.isnan(vals)
    assert ok.sum() == 254  # S.1111.111 is NaN for both signs; no infinities
    # Every finite code is a fixed point of rounding and re-encodes to itself
    # (codes 0x00 and 0x80 are +0 and -0).
    assert np.array_equal(fp8.round_e4m3(vals[ok]), vals[ok])
    assert np.array_equal(fp8.encode_e4m3(vals[ok]), codes[ok])


def test_landmarks():
    assert fp8.decode_e4m3(np.array([0x7E]))[0] == 448.0          # 0.1111.110
    assert fp8.decode_e4m3(np.array([0x08]))[0] == 2.0 ** -6      # smallest normal
    assert fp8.decode_e4m3(np.array([0x01]))[0] == 2.0 ** -9      # smallest subnormal
    assert list(fp8.decode_e4m3(np.arange(0x38, 0x40))) == [1 + k / 8 for k in range(8)]
    assert fp8.decode_e4m3(np.array([0xB8]))[0] == -1.0


def test_rounding_ties_and_saturation():
    # Ties go to the even mantissa: 1 + 1/16 lies between 1 and 1.125 -> 1;
    # 1 + 3/16 lies between 1.125 and 1.25 -> 1.25.
    assert fp8.round_e4m3(1.0625) == 1.0
    assert fp8.round_e4m3(1.1875) == 1.25
    assert fp8.round_e4m3(-1.0625) == -1.0
    # Subnormal ties: 1.5 * 2^-9 -> 2 * 2^-9 (even), 0.5 * 2^-9 -> 0.
    assert fp8.round_e4m3(1.5 * 2.0 ** -9) == 2.0 ** -8
    assert fp8.round_e4m3(0.5 * 2.0 ** -9) == 0.0
    # Past the largest finite value: saturate (also the halfway point 464).
    assert fp8.round_e4m3(500.0) == 448.0 and fp8.round_e4m3(-1e9) == -448.0
    assert fp8.round_e4m3(460.0) == 448.0


def test_block_quantization_error_bound_and_layout():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((3, 300, 64)) * np.array([1.0, 20.0, 1e-3])[:, None, None]
    codes, scales = fp8.quantize_blocks(x)
    assert scales.shape == (3, 3) and codes.shape == x.shape
    y = fp8.dequantize_blocks(codes, scales)
    # Each element within half a spacing of its binade (relative 2^-4), or
    # below the subnormal spacing.
    rel = np.abs(y - x) / np.maximum(np.abs(x), 1e-300)
    small = np.abs(x) / np.repeat(scales, 128, axis=1)[:, :300, None] < 2.0 ** -6
    assert np.all((rel <= 2.0 ** -4 + 1e-12) | small)
    # The block maximum maps to +-448 exactly.
    for t in range(3):
        blk = codes[:, t * 128:(t + 1) * 128]
        assert np.all(np.abs(fp8.decode_e4m3(blk)).max(axis=(1, 2)) == 448.0)
    ct, st = fp8.quantize_blocks(x, transpose=True)
    assert ct.shape == (3, 64, 300) and np.array_equal(ct.transpose(0, 2, 1), codes)
    assert np.array_equal(fp8.dequantize_blocks(ct, st, transpose=True), y)
