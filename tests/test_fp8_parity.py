"""FP8 (e4m3) quantizer and forward vs the oracle.

The quantizer is integer work decided by floating point: its codes and
scales must equal the reference quantizer's bit for bit (both divide in fp32
and round the same quotient).  The FP8 forward is compared with the fp64
attention oracle evaluated on the dequantized inputs (codes x block scales,
as produced by the reference quantizer), under a bound derived from its one
deliberate rounding, P to e4m3 before P V:

  each P' = P r_j (r_j = sv_j / max sv <= 1) is held as e4m3 with the row's
  exponent offset so that the largest P' of a row lies in [2^4, 2^8]; a normal
  e4m3 value is off by at most 2^-4 relative, a subnormal one by at most
  min(P', 2^-10).  In units of w = exp(s - max s) that is, per key,
      e_k = max(2^-4 w_k, min(w_k, 2^-14 / r_j)),
  so |O - O_ref| <= (sum_k e_k |v_k| + |O_ref| sum_k e_k) / sum_k w_k, the
  second term for the divisor's correction by the rounding of each tile's
  largest P'.  The test allows 1.25x that plus 1e-5 (fp32 sums, ex2).
LSE does not see the P rounding (row sums are fp32): max-abs 1e-3.
"""

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8 as ofp8
import exact_attention_95_gb300 as pkg
from exact_attention_95_gb300 import inputs

from parity import LSE_TOL, f64, to_dev

pytestmark = pytest.mark.gpu


def _bits_to_f32(bits):
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


@pytest.mark.parametrize("shape,transpose", [
    ((1, 2, 300, 128), False), ((1, 2, 300, 128), True),
    ((2, 3, 1000, 64), False), ((2, 3, 1000, 64), True),
    ((1, 1, 77, 128), True), ((1, 4, 4096, 128), True), ((1, 4, 4096, 128), False),
])
def test_quantize_bit_exact(shape, transpose):
    bits = inputs.make_blocky_tensor(0xF8 + shape[2] + shape[3], shape, exps=(-3, 0, 2, 5))
    if shape[2] > 128:
        bits[0, 0, 128:256] = 0  # an all-zero block: scale 1, codes 0
    X = to_dev(bits)
    codes, scales = pkg.attn_quantize_fp8(X, transpose=transpose)
    torch.cuda.synchronize()
    B, H, N, d = shape
    x = _bits_to_f32(bits).reshape(B * H, N, d)
    rc, rs = ofp8.quantize_blocks(x, transpose=transpose)
    got = codes.cpu().numpy().reshape(B * H, *codes.shape[2:])
    if transpose:
        ldt = pkg.attn_fp8_vt_stride(N)
        assert got.shape == (B * H, d, ldt)
        assert np.all(got[:, :, N:] == 0), "pad columns must be zero"
        got = got[:, :, :N]
    assert np.array_equal(scales.cpu().numpy().reshape(B * H, -1), rs), "scales differ"
    diff = np.argwhere(got != rc)
    assert diff.size == 0, f"{len(diff)} codes differ, first at {diff[:3].tolist()}"


def _fp8_inputs(B, Hq, Hkv, N, seed, exps=(-1, 0, 1)):
    """Seeded bf16 inputs with per-block magnitudes, quantized by the reference
    quantizer: device codes/scales for the kernel, fp64 dequantized tensors for
    the oracle."""
    dev, host = {}, {}
    for name, H in (("Q", Hq), ("K", Hkv), ("V", Hkv)):
        bits = inputs.make_blocky_tensor(seed + inputs.TENSOR_IDS[name], (B, H, N, 128), exps=exps)
        x = _bits_to_f32(bits).reshape(B * H, N, 128)
        tr = name == "V"
        c, s = ofp8.quantize_blocks(x, transpose=tr)
        host[name] = ofp8.dequantize_blocks(c, s, transpose=tr).reshape(B, H, N, 128)
        host["s" + name] = s.reshape(B, H, -1).astype(np.float64)
        if tr:
            ldt = pkg.attn_fp8_vt_stride(N)
            cp = np.zeros((B * H, 128, ldt), dtype=np.uint8)
            cp[:, :, :N] = c
            c = cp.reshape(B, H, 128, ldt)
        else:
            c = c.reshape(B, H, N, 128)
        dev[name] = torch.from_numpy(np.ascontiguousarray(c)).cuda()
        dev["s" + name] = torch.from_numpy(s.reshape(B, H, -1).astype(np.float32)).cuda()
    return dev, host


def _o_bound_rows(q, k, v, sv, scale, causal, rows, oref):
    """Bound for query rows `rows` of one head: q [R, d] those rows, k, v [N, d],
    sv [T] the head's V block scales, oref [R, d] the reference rows."""
    N = k.shape[0]
    keep = (np.arange(N)[None, :] <= np.asarray(rows)[:, None]) if causal else np.ones((len(rows), N), dtype=bool)
    s = np.where(keep, scale * (q @ k.T), -np.inf)
    w = np.exp(s - s.max(axis=1, keepdims=True))
    rinv = np.repeat(sv.max() / sv, 128)[:N]
    e = np.where(keep, np.maximum(2.0 ** -4 * w, np.minimum(w, 2.0 ** -14 * rinv[None, :])), 0.0)
    den = w.sum(axis=1, keepdims=True)
    return 1.25 * (e @ np.abs(v) + np.abs(oref) * e.sum(axis=1, keepdims=True)) / den + 1e-5


def _o_bound(Qd, Kd, Vd, sV, scale, causal, Oref):
    """Per-element bound on |O - O_ref| from the e4m3 rounding of P (see above)."""
    B, Hq, N, d = Qd.shape
    G = Hq // Kd.shape[1]
    bound = np.zeros_like(Oref)
    for b in range(B):
        for h in range(Hq):
            bound[b, h] = _o_bound_rows(Qd[b, h], Kd[b, h // G], Vd[b, h // G], sV[b, h // G], scale, causal,
                                        np.arange(N), Oref[b, h])
    return bound


FWD_CASES = [
    # B, Hq, Hkv, N, causal
    (1, 2, 1, 300, True),
    (1, 2, 2, 300, False),
    (2, 4, 2, 1000, True),
    (1, 2, 1, 128, True),
    (1, 1, 1, 77, False),
    (1, 2, 2, 1536, True),
    (1, 2, 1, 1, True),     # one query and one key
    (1, 1, 1, 16, True),    # one partial tile
    (2, 4, 1, 257, True),   # GQA 4:1, a tile of one row at the end
]


@pytest.mark.parametrize("case", FWD_CASES, ids=lambda c: "B%dHq%dHkv%dN%d_c%d" % c)
def test_fwd_fp8_parity(case):
    B, Hq, Hkv, N, causal = case
    dev, host = _fp8_inputs(B, Hq, Hkv, N, seed=0xF800 + N + 7 * Hq)
    scale = 1.0 / np.sqrt(128)
    O, L = pkg.attn_fwd_fp8(dev["Q"], dev["sQ"], dev["K"], dev["sK"], dev["V"], dev["sV"], scale, causal,
                            out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert pkg.attn_last_device_status() == pkg.ATTN_OK
    Oref, Lref = oracle.fwd(host["Q"], host["K"], host["V"], scale, causal)
    err = np.abs(f64(O) - Oref)
    bound = _o_bound(host["Q"], host["K"], host["V"], host["sV"], scale, causal, Oref)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert np.all(err <= bound), f"O err {err[worst]:.3e} > bound {bound[worst]:.3e} at {worst}"
    # The rounding errors are independent across keys: on average far inside the worst case.
    assert err.mean() <= 0.5 * bound.mean(), (err.mean(), bound.mean())
    err_l = np.abs(f64(L) - Lref).max()
    assert err_l <= LSE_TOL, f"LSE max-abs {err_l:.3e}"


def test_fwd_fp8_large_logits_bf16_out():
    # Peaked rows (Q x 8): one key dominates; its rounding cancels in O / (l - corr).
    B, Hq, Hkv, N = 1, 2, 1, 640
    dev, host = _fp8_inputs(B, Hq, Hkv, N, seed=0xF8F8, exps=(2, 3))
    scale = 1.0 / np.sqrt(128)
    O, L = pkg.attn_fwd_fp8(dev["Q"], dev["sQ"], dev["K"], dev["sK"], dev["V"], dev["sV"], scale, True)
    torch.cuda.synchronize()
    Oref, Lref = oracle.fwd(host["Q"], host["K"], host["V"], scale, True)
    bound = _o_bound(host["Q"], host["K"], host["V"], host["sV"], scale, True, Oref)
    half_ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(Oref), 2.0 ** -126))) - 8)
    err = np.abs(f64(O) - Oref)
    assert np.all(err <= bound + half_ulp), float((err - bound - half_ulp).max())
    assert np.abs(f64(L) - Lref).max() <= LSE_TOL


def test_fwd_fp8_equals_quantizer_roundtrip():
    # The library quantizer feeds the library forward: same result as the
    # reference quantizer's codes (bit-identical inputs give identical outputs).
    B, Hq, Hkv, N = 1, 2, 1, 384
    dev, host = _fp8_inputs(B, Hq, Hkv, N, seed=0xF877)
    tensors = {}
    for name, H in (("Q", Hq), ("K", Hkv), ("V", Hkv)):
        bits = inputs.make_blocky_tensor(0xF877 + inputs.TENSOR_IDS[name], (B, H, N, 128), exps=(-1, 0, 1))
        tensors[name] = pkg.attn_quantize_fp8(to_dev(bits), transpose=(name == "V"))
    a = pkg.attn_fwd_fp8(dev["Q"], dev["sQ"], dev["K"], dev["sK"], dev["V"], dev["sV"], None, True)
    b = pkg.attn_fwd_fp8(tensors["Q"][0], tensors["Q"][1], tensors["K"][0], tensors["K"][1], tensors["V"][0],
                         tensors["V"][1], None, True)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_fwd_fp8_bench_workload_sampled_rows():
    """The FP8 benchmark's launch: the c3 tensors (B2 H32 N4096 d128, causal,
    Q x8) quantized by the library, bf16 O.  Checked on 128 seeded rows of each
    of four heads; the codes of those heads are also compared with the
    reference quantizer's."""
    w = inputs.WORKLOADS["c3"]
    t = inputs.workload_tensors(w, names=("Q", "K", "V"))
    g = {k: to_dev(v) for k, v in t.items()}
    qc, qs = pkg.attn_quantize_fp8(g["Q"])
    kc, ks = pkg.attn_quantize_fp8(g["K"])
    vc, vs = pkg.attn_quantize_fp8(g["V"], transpose=True)
    O, L = pkg.attn_fwd_fp8(qc, qs, kc, ks, vc, vs, w.scale, w.causal)
    torch.cuda.synchronize()
    assert pkg.attn_last_device_status() == pkg.ATTN_OK
    assert torch.isfinite(O).all() and torch.isfinite(L).all()
    dev_codes = {"Q": (qc, qs), "K": (kc, ks), "V": (vc, vs)}
    for b, h in ((0, 0), (0, 13), (1, 7), (1, 31)):
        deq, sv = {}, None
        for name in ("Q", "K", "V"):
            tr = name == "V"
            x = _bits_to_f32(t[name][b, h])[None]
            c, s = ofp8.quantize_blocks(x, transpose=tr)
            dc, ds = dev_codes[name]
            assert np.array_equal(dc[b, h].cpu().numpy(), c[0]), f"{name} codes of head ({b},{h})"
            assert np.array_equal(ds[b, h].cpu().numpy(), s[0])
            deq[name] = ofp8.dequantize_blocks(c, s, transpose=tr)[0]
            if tr:
                sv = s[0].astype(np.float64)
        rows = inputs.sample_rows(0xF8C3 + 64 * b + h, w.N, 128, must=[0, 1, 127, 128, w.N - 1])
        Oref, Lref = oracle.fwd_rows(deq["Q"][None, None], deq["K"][None, None], deq["V"][None, None], w.scale,
                                     w.causal, rows)
        Oref = Oref.reshape(len(rows), w.d)
        Lref = Lref.reshape(len(rows))
        bound = _o_bound_rows(deq["Q"][rows], deq["K"], deq["V"], sv, w.scale, w.causal, rows, Oref)
        half_ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(Oref), 2.0 ** -126))) - 8)
        Og = f64(O[b, h])[rows]
        err = np.abs(Og - Oref)
        assert np.all(err <= bound + half_ulp), f"head ({b},{h}): {float((err - bound - half_ulp).max()):.3e}"
        assert np.abs(f64(L[b, h])[rows] - Lref).max() <= LSE_TOL
