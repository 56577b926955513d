"""Split-key forward with separate query and key lengths vs the fp64 oracle.

attn_fwd_split computes the same function as the oracle's forward for
Nq != Nk (causal mask aligned to the bottom-right corner; rows with no kept
key give O = 0, LSE = -inf) and splits the key range into parts whose partial
(O, LSE) pairs are merged.  Compared element by element against the oracle,
for decode-like shapes (one query row, long key range), ragged lengths, more
splits than tiles, GQA, and Nq > Nk.
"""

import numpy as np
import pytest
import torch

import oracle
import exact_attention_95_gb300 as pkg
from exact_attention_95_gb300 import inputs

from parity import LSE_TOL, check_o, f64, to_dev

pytestmark = pytest.mark.gpu


def _make(B, Hq, Hkv, Nq, Nk, d, seed, q_mul=1.0):
    t = {
        "Q": inputs.make_tensor(seed + 0, (B, Hq, Nq, d), "bf16", q_mul),
        "K": inputs.make_tensor(seed + 1, (B, Hkv, Nk, d), "bf16"),
        "V": inputs.make_tensor(seed + 2, (B, Hkv, Nk, d), "bf16"),
    }
    return t, {k: to_dev(v) for k, v in t.items()}


def _check(O, L, Oref, Lref, bf16_out=False):
    empty = np.isneginf(Lref)
    assert np.array_equal(np.isneginf(L), empty), "rows without keys must have LSE = -inf"
    assert np.all(O[empty] == 0.0), "rows without keys must have O = 0"
    err_o, ok = check_o(O, Oref, bf16_out=bf16_out)
    assert ok, f"O max-abs {err_o:.3e}"
    if (~empty).any():
        err_l = np.abs(L[~empty] - Lref[~empty]).max()
        assert err_l <= LSE_TOL, f"LSE max-abs {err_l:.3e}"


CASES = [
    # B, Hq, Hkv, Nq, Nk, d, causal, splits
    (1, 4, 2, 1, 4096, 128, False, 0),
    (1, 4, 2, 1, 4096, 128, True, 8),
    (1, 4, 2, 3, 4096, 128, True, 32),
    (2, 2, 1, 130, 1000, 64, False, 3),
    (2, 2, 1, 130, 1000, 64, True, 1),
    (2, 2, 1, 130, 1000, 64, True, 3),
    (1, 2, 2, 777, 777, 128, True, 5),
    (1, 2, 1, 300, 100, 128, True, 2),   # Nq > Nk: the first rows keep no key
    (1, 2, 1, 300, 100, 128, False, 1),
    (1, 1, 1, 64, 200, 64, False, 4),    # more splits than tiles
    (1, 1, 1, 128, 1024, 128, False, 8),  # one tile per split
    (1, 8, 8, 256, 8192, 128, True, 0),
    # GQA packing: the G query heads of a kv head share one tile when G * Nq <= 128.
    (2, 8, 2, 16, 700, 64, True, 3),
    (1, 16, 1, 8, 1000, 128, True, 0),    # exactly 128 packed rows
    (1, 16, 1, 9, 1000, 128, True, 2),    # 144 rows: not packed
    (1, 4, 1, 20, 10, 64, True, 1),       # packed, Nq > Nk: rows i < 10 keep no key
    (1, 32, 8, 1, 131072, 128, True, 0),  # the decode benchmark shape
    # Few rows per kv head (decoding shapes), d = 64 and 128.
    (2, 4, 4, 3, 1000, 64, True, 0),      # Hq == Hkv, 3 query rows
    (1, 8, 1, 1, 5000, 64, False, 0),     # 8 packed rows, d = 64
    (1, 2, 2, 8, 300, 128, True, 2),      # Hq == Hkv, 8 rows, bottom-right causal
    (1, 6, 2, 2, 2000, 128, True, 0),     # 6 packed rows
    (1, 4, 2, 1, 1, 128, False, 0),       # a single key
    # More parts than one warp's lanes: the merge reads the parts' LSEs in
    # chunks of 32 and their O rows in batches of 16.
    (1, 4, 2, 2, 9000, 64, True, 40),
    (1, 2, 1, 1, 9000, 128, False, 71),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B%dHq%dHkv%dNq%dNk%dd%d_c%d_s%d" % c)
def test_fwd_split_parity(case):
    B, Hq, Hkv, Nq, Nk, d, causal, splits = case
    t, g = _make(B, Hq, Hkv, Nq, Nk, d, seed=9000 + Nq + Nk + d)
    scale = 1.0 / np.sqrt(d)
    O, L = pkg.attn_fwd_split(g["Q"], g["K"], g["V"], scale, causal, num_splits=splits,
                              out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert pkg.attn_last_device_status() == pkg.ATTN_OK
    f = {k: inputs.to_f64(v) for k, v in t.items()}
    Oref, Lref = oracle.fwd(f["Q"], f["K"], f["V"], scale, causal)
    _check(f64(O), f64(L), Oref, Lref)


def test_fwd_split_bf16_out_large_logits():
    t, g = _make(1, 4, 1, 5, 3000, 128, seed=321, q_mul=8.0)
    scale = 1.0 / np.sqrt(128)
    O, L = pkg.attn_fwd_split(g["Q"], g["K"], g["V"], scale, True, num_splits=6)
    torch.cuda.synchronize()
    f = {k: inputs.to_f64(v) for k, v in t.items()}
    Oref, Lref = oracle.fwd(f["Q"], f["K"], f["V"], scale, True)
    _check(f64(O), f64(L), Oref, Lref, bf16_out=True)


def test_fwd_split_one_split_equals_attn_fwd():
    # With Nq == Nk and one split the same kernel writes the same bits.
    t, g = _make(1, 4, 2, 640, 640, 128, seed=55)
    a = pkg.attn_fwd(g["Q"], g["K"], g["V"], None, True)
    b = pkg.attn_fwd_split(g["Q"], g["K"], g["V"], None, True, num_splits=1)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_fwd_split_repeatable_and_split_invariant():
    t, g = _make(1, 2, 2, 17, 2048, 64, seed=77)
    ref = pkg.attn_fwd_split(g["Q"], g["K"], g["V"], None, True, num_splits=4, out_dtype=torch.float32)
    for _ in range(3):
        o, l = pkg.attn_fwd_split(g["Q"], g["K"], g["V"], None, True, num_splits=4, out_dtype=torch.float32)
        assert torch.equal(o, ref[0]) and torch.equal(l, ref[1])
    # Different split counts give the same function up to rounding.
    for s in (1, 2, 16):
        o, l = pkg.attn_fwd_split(g["Q"], g["K"], g["V"], None, True, num_splits=s, out_dtype=torch.float32)
        assert (o - ref[0]).abs().max().item() < 1e-3
        assert (l - ref[1]).abs().max().item() < 1e-4
