"""Block-sparse forward and backward vs the fp64 oracle's masked entry points.

A uint8 mask [1 or Hq, T, T] (T = ceil(N/128)) removes 128 x 128 blocks on
top of the causal rule (Block-Sparse FlashAttention, "从Online-Softmax到
FlashAttention V1/V2/V3" 0x04).  Random masks (shared and per head), query
tiles with every block removed (O = 0, LSE = -inf, dQ = 0), key tiles no
kept block reaches (dK = dV = 0), GQA, causal and not; an all-ones mask gives
the dense results.
"""

import numpy as np
import pytest
import torch

import oracle
import exact_attention_95_gb300 as pkg
from exact_attention_95_gb300 import inputs

from parity import GRAD_TOL, LSE_TOL, check_o, f64, make, rel_err, to_dev

pytestmark = pytest.mark.gpu


def _mask(heads, N, density, seed, kill_q=None, kill_k=None):
    T = (N + 127) // 128
    rng = np.random.default_rng(seed)
    m = (rng.random((heads, T, T)) < density).astype(np.uint8)
    if kill_q is not None:
        m[:, kill_q, :] = 0
    if kill_k is not None:
        m[:, :, kill_k] = 0
    return m


CASES = [
    # B, Hq, Hkv, N, d, causal, mask heads, density, query tile to kill, key tile to kill
    (1, 2, 1, 640, 128, True, 1, 0.5, None, None),
    (2, 4, 2, 777, 64, False, 4, 0.6, 1, None),
    (1, 2, 2, 1024, 128, True, 2, 0.35, 3, 0),
    (1, 4, 1, 300, 128, False, 4, 0.7, None, 2),
    (1, 1, 1, 2048, 64, True, 1, 0.25, 5, 7),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B%dHq%dHkv%dN%dd%d_c%d_mh%d_p%.2f_q%s_k%s" % c)
def test_blocksparse_fwd_bwd_parity(case):
    B, Hq, Hkv, N, d, causal, mh, dens, kq, kk = case
    t = make(B, Hq, Hkv, N, d, seed=7000 + N + d)
    g = {k: to_dev(v) for k, v in t.items()}
    m = _mask(mh, N, dens, seed=N + mh, kill_q=kq, kill_k=kk)
    gm = torch.from_numpy(m).cuda()
    scale = 1.0 / np.sqrt(d)
    O, L = pkg.attn_fwd_masked(g["Q"], g["K"], g["V"], gm, scale, causal, out_dtype=torch.float32)
    Ob = O.to(torch.bfloat16)
    dQ, dK, dV = pkg.attn_bwd_masked(g["Q"], g["K"], g["V"], Ob, g["dO"], L, gm, scale, causal)
    torch.cuda.synchronize()
    assert pkg.attn_last_device_status() == pkg.ATTN_OK
    f = {k: inputs.to_f64(v) for k, v in t.items()}
    ref = oracle.bwd_masked(f["Q"], f["K"], f["V"], f["dO"], scale, causal, m)
    Oref, Lref = ref["O"], ref["LSE"]
    Og, Lg = f64(O), f64(L)
    empty = np.isneginf(Lref)
    assert np.array_equal(np.isneginf(Lg), empty)
    assert np.all(Og[empty] == 0.0)
    err_o, ok = check_o(Og, Oref, bf16_out=False)
    assert ok, f"O max-abs {err_o:.3e}"
    if (~empty).any():
        assert np.abs(Lg[~empty] - Lref[~empty]).max() <= LSE_TOL
    if kq is not None:
        assert np.all(empty[:, :, kq * 128:(kq + 1) * 128])
    # The backward reads the forward's bf16 O, as a training step would.
    for name, got in (("dQ", dQ), ("dK", dK), ("dV", dV)):
        e = rel_err(f64(got), ref[name])
        assert e <= GRAD_TOL, f"{name} rel err {e:.3e}"
    if kk is not None:
        assert torch.all(dK[:, :, kk * 128:(kk + 1) * 128] == 0) and torch.all(dV[:, :, kk * 128:(kk + 1) * 128] == 0)


def test_all_ones_mask_equals_dense():
    B, Hq, Hkv, N, d = 1, 4, 2, 700, 128
    t = make(B, Hq, Hkv, N, d, seed=4321)
    g = {k: to_dev(v) for k, v in t.items()}
    T = (N + 127) // 128
    ones = torch.ones(1, T, T, dtype=torch.uint8, device="cuda")
    for causal in (False, True):
        Od, Ld = pkg.attn_fwd(g["Q"], g["K"], g["V"], None, causal)
        Om, Lm = pkg.attn_fwd_masked(g["Q"], g["K"], g["V"], ones, None, causal)
        assert torch.equal(Od, Om) and torch.equal(Ld, Lm)
        gd = pkg.attn_bwd(g["Q"], g["K"], g["V"], Od, g["dO"], Ld, None, causal)
        gm = pkg.attn_bwd_masked(g["Q"], g["K"], g["V"], Od, g["dO"], Ld, ones, None, causal)
        for a, b in zip(gd, gm):
            assert (a.float() - b.float()).abs().max().item() <= 2e-2 * a.float().abs().max().item()


def test_blocksparse_bench_workload_two_heads():
    """The block-sparse benchmark's launch: the c3 tensors (B2 H32 N4096 d128,
    causal, Q x8) with its density-1/2 mask shared by all heads; forward with
    bf16 O and the backward reading it.  Two whole heads against the oracle."""
    import bench
    w = inputs.WORKLOADS["c3"]
    t = inputs.workload_tensors(w)
    g = {k: to_dev(v) for k, v in t.items()}
    T = (w.N + 127) // 128
    m = inputs.random_block_mask(bench.SPARSE_MASK_SEED, 1, T, 0.5)
    gm = torch.from_numpy(m).cuda()
    O, L = pkg.attn_fwd_masked(g["Q"], g["K"], g["V"], gm, w.scale, w.causal)
    dQ, dK, dV = pkg.attn_bwd_masked(g["Q"], g["K"], g["V"], O, g["dO"], L, gm, w.scale, w.causal)
    torch.cuda.synchronize()
    assert pkg.attn_last_device_status() == pkg.ATTN_OK
    for b, h in ((0, 0), (1, 31)):
        f = {k: inputs.to_f64(v[b:b + 1, h:h + 1]) for k, v in t.items()}
        ref = oracle.bwd_masked(f["Q"], f["K"], f["V"], f["dO"], w.scale, w.causal, m)
        Og, Lg = f64(O[b:b + 1, h:h + 1]), f64(L[b:b + 1, h:h + 1])
        empty = np.isneginf(ref["LSE"])
        assert np.array_equal(np.isneginf(Lg), empty)
        err_o, ok = check_o(Og, ref["O"], bf16_out=True)
        assert ok, f"head ({b},{h}) O max-abs {err_o:.3e}"
        assert np.abs(Lg[~empty] - ref["LSE"][~empty]).max() <= LSE_TOL
        # The oracle's gradients use its own O; the GPU's use its bf16 O (as a
        # training step does): both within the gradient tolerance.
        for name, got in (("dQ", dQ), ("dK", dK), ("dV", dV)):
            e = rel_err(f64(got[b:b + 1, h:h + 1]), ref[name])
            assert e <= GRAD_TOL, f"head ({b},{h}) {name} rel err {e:.3e}"
    assert torch.isfinite(dQ).all() and torch.isfinite(dK).all() and torch.isfinite(dV).all()
