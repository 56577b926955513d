"""bf16 output against fp32 output of the same kernels, bit for bit.

Every forward kernel stages bf16 O rows through shared memory and stores
them a row piece at a time; the fp32 output path stores each thread's row
directly.  Both round the same fp32 product O/l, so the bf16 output must
equal the fp32 output rounded to nearest even, element by element, and LSE
must be identical -- on ragged lengths (partial warps of rows), on the
persistent, one-tile, packed-split, block-sparse and FP8 kernels.
"""
import numpy as np
import pytest
import torch

import exact_attention_95_gb300 as pkg

from parity import make, to_dev

pytestmark = pytest.mark.gpu


def _same(a32, L32, a16, L16):
    torch.cuda.synchronize()
    assert pkg.attn_last_device_status() == pkg.ATTN_OK
    assert a16.dtype == torch.bfloat16 and a32.dtype == torch.float32
    assert torch.equal(a16, a32.to(torch.bfloat16))
    assert torch.equal(L16, L32)


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal", [
    (1, 4, 2, 700, 128, True),    # persistent, ragged last pair
    (2, 2, 1, 333, 64, False),    # persistent, d = 64
    (1, 2, 2, 100, 128, True),    # one query tile
    (1, 3, 3, 129, 64, True),     # a tile of one row
])
def test_dense_bf16_equals_rounded_fp32(B, Hq, Hkv, N, d, causal):
    t = make(B, Hq, Hkv, N, d, seed=0xE900 + N + d, names=("Q", "K", "V"))
    g = {k: to_dev(v) for k, v in t.items()}
    O32, L32 = pkg.attn_fwd(g["Q"], g["K"], g["V"], None, causal, out_dtype=torch.float32)
    O16, L16 = pkg.attn_fwd(g["Q"], g["K"], g["V"], None, causal)
    _same(O32, L32, O16, L16)


def test_split_packed_bf16_equals_rounded_fp32():
    # 8 query heads on 2 kv heads, 5 query rows each: packed one-tile rows;
    # one split writes O directly, several go through the merge.
    t = make(1, 8, 2, 5, 128, seed=0xE9A0, names=("Q",))
    kv = make(1, 8, 2, 3000, 128, seed=0xE9A1, names=("K", "V"))
    g = {"Q": to_dev(t["Q"]), "K": to_dev(kv["K"]), "V": to_dev(kv["V"])}
    for splits in (1, 4):
        O32, L32 = pkg.attn_fwd_split(g["Q"], g["K"], g["V"], None, True, num_splits=splits,
                                      out_dtype=torch.float32)
        O16, L16 = pkg.attn_fwd_split(g["Q"], g["K"], g["V"], None, True, num_splits=splits)
        _same(O32, L32, O16, L16)


def test_masked_bf16_equals_rounded_fp32():
    B, Hq, Hkv, N, d = 1, 2, 1, 555, 128
    t = make(B, Hq, Hkv, N, d, seed=0xE9B0, names=("Q", "K", "V"))
    g = {k: to_dev(v) for k, v in t.items()}
    T = (N + 127) // 128
    m = (np.random.default_rng(3).random((Hq, T, T)) < 0.6).astype(np.uint8)
    gm = torch.from_numpy(m).cuda()
    for causal in (False, True):
        O32, L32 = pkg.attn_fwd_masked(g["Q"], g["K"], g["V"], gm, None, causal, out_dtype=torch.float32)
        O16, L16 = pkg.attn_fwd_masked(g["Q"], g["K"], g["V"], gm, None, causal)
        _same(O32, L32, O16, L16)


def test_fp8_bf16_equals_rounded_fp32():
    t = make(2, 4, 2, 700, 128, seed=0xE9C0, names=("Q", "K", "V"))
    g = {k: to_dev(v) for k, v in t.items()}
    qc, qs = pkg.attn_quantize_fp8(g["Q"])
    kc, ks = pkg.attn_quantize_fp8(g["K"])
    vc, vs = pkg.attn_quantize_fp8(g["V"], transpose=True)
    for causal in (False, True):
        O32, L32 = pkg.attn_fwd_fp8(qc, qs, kc, ks, vc, vs, None, causal, out_dtype=torch.float32)
        O16, L16 = pkg.attn_fwd_fp8(qc, qs, kc, ks, vc, vs, None, causal)
        _same(O32, L32, O16, L16)


def test_tensor_map_cache_follows_shape():
    # The library caches TMA tensor maps by every encoding argument: the same
    # base pointer with another length must not reuse the longer map.
    t = make(1, 1, 1, 900, 128, seed=0xE9D0, names=("Q", "K", "V"))
    g = {k: to_dev(v) for k, v in t.items()}
    full = pkg.attn_fwd(g["Q"], g["K"], g["V"], None, True, out_dtype=torch.float32)
    for n in (900, 333, 129, 900):
        pre = {k: v[:, :, :n] for k, v in g.items()}  # contiguous prefix views, same base pointers
        fresh = {k: v.clone() for k, v in pre.items()}
        a = pkg.attn_fwd(pre["Q"], pre["K"], pre["V"], None, True, out_dtype=torch.float32)
        b = pkg.attn_fwd(fresh["Q"], fresh["K"], fresh["V"], None, True, out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
        # Causal: a prefix of the queries sees exactly the same keys.
        assert torch.equal(a[0], full[0][:, :, :n]) and torch.equal(a[1], full[1][:, :, :n])
