"""Reference FP8 (e4m3) block quantization, written from the number format.

TEST INFRASTRUCTURE ONLY (part of the oracle): used by the tests to check the
library's quantizer bit for bit and to dequantize FP8 inputs for the fp64
attention oracle.  Shares no code with the CUDA path.

The FP8 attention of "LLM 注意力与计算内核精读笔记 · 02 FlashAttention" §10
(FA3: FP8 tensor cores with block-level quantization, a per-block scale being
steadier than a per-tensor one, §12.2) leaves the format details open; the
readings taken here:
  - e4m3 in the OCP layout: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa
    bits; largest finite value 448 = 1.75 * 2^8; subnormals k * 2^-9; no
    infinities.
  - Rounding to nearest, ties to even; values beyond 448 saturate to +-448.
  - A block is 128 consecutive rows of one head; its scale is amax / 448
    (1 for an all-zero block), and x is stored as e4m3(x / scale).  The
    division and the scale are fp32 operations (IEEE, round to nearest), as
    in the kernel that produces the codes, so both round the same quotient.
"""

import numpy as np

E4M3_MAX = 448.0
BLOCK = 128


def round_e4m3(x):
    """Nearest e4m3 value (ties to even, saturating) of each element, as float64."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    out = np.zeros_like(a)
    nz = a > 0
    # Binade exponent, at least -6 (the subnormal binade shares the quantum 2^-9).
    e = np.full(a.shape, -6.0)
    e[nz] = np.maximum(np.floor(np.log2(a[nz])), -6.0)
    q = np.exp2(e - 3.0)  # spacing of representable values in the binade
    r = np.round(a / q) * q  # numpy rounds half to even
    out = np.minimum(r, E4M3_MAX)
    return np.copysign(out, x)


def encode_e4m3(v):
    """8-bit codes of e4m3-representable values v (as produced by round_e4m3)."""
    v = np.asarray(v, dtype=np.float64)
    sign = (np.signbit(v)).astype(np.uint8) << 7
    a = np.abs(v)
    code = np.zeros(a.shape, dtype=np.uint8)
    sub = a < 2.0 ** -6
    # Subnormal: exponent field 0, mantissa a / 2^-9.
    code[sub] = np.round(a[sub] / 2.0 ** -9).astype(np.uint8)
    nrm = ~sub
    e = np.floor(np.log2(a[nrm]))
    mant = np.round((a[nrm] / np.exp2(e) - 1.0) * 8.0)
    code[nrm] = ((e + 7).astype(np.uint8) << 3) | mant.astype(np.uint8)
    return code | sign


def decode_e4m3(code):
    """Value of each 8-bit e4m3 code (NaN for the code S.1111.111)."""
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    ex = (c >> 3) & 0xF
    m = c & 7
    val = np.where(ex == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(ex - 7.0))
    val = np.where((ex == 15) & (m == 7), np.nan, val)
    return s * val


def quantize_blocks(x, transpose=False):
    """Block quantization of x [BH, N, d] (float64): per 128-row block of a head,
    scale = amax / 448 (1 if the block is zero) and codes = e4m3(x / scale).
    Returns (codes [BH, N, d] or, with transpose, [BH, d, N]; scales [BH, T])."""
    x = np.asarray(x, dtype=np.float32)
    BH, N, d = x.shape
    T = -(-N // BLOCK)
    scales = np.ones((BH, T), dtype=np.float32)
    codes = np.zeros((BH, N, d), dtype=np.uint8)
    for t in range(T):
        blk = x[:, t * BLOCK:(t + 1) * BLOCK, :]
        amax = np.abs(blk).max(axis=(1, 2))
        sc = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
        scales[:, t] = sc
        q = (blk / sc[:, None, None]).astype(np.float32)  # fp32 quotient, round to nearest
        codes[:, t * BLOCK:(t + 1) * BLOCK, :] = encode_e4m3(round_e4m3(q.astype(np.float64)))
    if transpose:
        codes = np.ascontiguousarray(codes.transpose(0, 2, 1))
    return codes, scales


def dequantize_blocks(codes, scales, transpose=False):
    """Inverse of quantize_blocks (exact in float64)."""
    c = np.asarray(codes)
    if transpose:
        c = c.transpose(0, 2, 1)
    v = decode_e4m3(c)
    BH, N, d = v.shape
    rep = np.repeat(np.asarray(scales, dtype=np.float64), BLOCK, axis=1)[:, :N]
    return v * rep[:, :, None]
