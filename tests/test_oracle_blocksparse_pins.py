"""Pins of the oracle's block-sparse forward and backward (CPU only).

Block-Sparse FlashAttention ("从Online-Softmax到FlashAttention V1/V2/V3", 0x04)
skips the blocks a block mask zeroes: their keys take no part in the softmax
of those queries.  The oracle's masked entry points are pinned against things
other than themselves: brute force with an explicit element mask, a
block-diagonal mask that must equal independent attention inside each block,
invariance to the contents of masked blocks, empty rows, an all-ones mask,
and central finite differences for the backward.
"""

import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(20261203)


def _rand(*shape):
    return RNG.standard_normal(shape)


def _brute(Q, K, V, scale, elem_mask):
    """Attention with an explicit keep-mask [Hq or 1, Nq, Nk], one head at a time."""
    B, Hq, Nq, d = Q.shape
    Hkv, Nk = K.shape[1], K.shape[2]
    G = Hq // Hkv
    O = np.zeros((B, Hq, Nq, d))
    L = np.full((B, Hq, Nq), -np.inf)
    for b in range(B):
        for h in range(Hq):
            m = elem_mask[0 if elem_mask.shape[0] == 1 else h]
            s = Q[b, h] @ K[b, h // G].T * scale
            s = np.where(m, s, -np.inf)
            for i in range(Nq):
                row = s[i]
                if np.all(np.isneginf(row)):
                    continue
                e = np.exp(row - row.max())
                O[b, h, i] = (e / e.sum()) @ V[b, h // G]
                L[b, h, i] = row.max() + np.log(e.sum())
    return O, L


def _elem_mask(bmask, Nq, Nk, bsize, causal):
    hm = bmask.shape[0]
    m = np.zeros((hm, Nq, Nk), dtype=bool)
    for h in range(hm):
        for i in range(Nq):
            for j in range(Nk):
                keep = bmask[h, i // bsize, j // bsize] != 0
                if causal and j > i + (Nk - Nq):
                    keep = False
                m[h, i, j] = keep
    return m


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("heads_mask", [1, 4])
def test_masked_forward_equals_brute_force(causal, heads_mask):
    B, Hq, Hkv, Nq, Nk, d, bs = 2, 4, 2, 11, 13, 5, 3
    Q, K, V = _rand(B, Hq, Nq, d), _rand(B, Hkv, Nk, d), _rand(B, Hkv, Nk, d)
    nqb, nkb = -(-Nq // bs), -(-Nk // bs)
    bmask = (RNG.random((heads_mask, nqb, nkb)) < 0.6).astype(np.uint8)
    O, L = oracle.fwd_masked(Q, K, V, 0.4, causal, bmask, bsize=bs)
    Ob, Lb = _brute(Q, K, V, 0.4, _elem_mask(bmask, Nq, Nk, bs, causal))
    assert np.allclose(O, Ob, rtol=0, atol=1e-12)
    assert np.array_equal(np.isneginf(L), np.isneginf(Lb))
    fin = np.isfinite(Lb)
    assert np.allclose(L[fin], Lb[fin], rtol=0, atol=1e-12)


def test_block_diagonal_mask_is_independent_blocks():
    # With only diagonal blocks kept, each query block attends to its own key
    # block alone: the output equals plain attention on each block separately.
    B, Hq, N, d, bs = 1, 2, 12, 4, 4
    Q, K, V = _rand(B, Hq, N, d), _rand(B, Hq, N, d), _rand(B, Hq, N, d)
    bmask = np.eye(N // bs, dtype=np.uint8)[None]
    O, L = oracle.fwd_masked(Q, K, V, 0.5, False, bmask, bsize=bs)
    for k in range(N // bs):
        sl = slice(k * bs, (k + 1) * bs)
        Ok, Lk = oracle.fwd(Q[:, :, sl], K[:, :, sl], V[:, :, sl], 0.5, False)
        assert np.allclose(O[:, :, sl], Ok, rtol=0, atol=1e-13)
        assert np.allclose(L[:, :, sl], Lk, rtol=0, atol=1e-13)


def test_masked_blocks_have_no_influence():
    B, Hq, N, d, bs = 1, 2, 16, 3, 4
    Q, K, V = _rand(B, Hq, N, d), _rand(B, Hq, N, d), _rand(B, Hq, N, d)
    bmask = np.ones((1, 4, 4), dtype=np.uint8)
    bmask[0, 1, 2] = bmask[0, 3, 0] = 0
    O1, L1 = oracle.fwd_masked(Q, K, V, 0.7, False, bmask, bsize=bs)
    K2, V2 = K.copy(), V.copy()
    # Keys 8..11 are masked for queries 4..7 only: changing them must leave those rows alone.
    K2[:, :, 8:12] += 5.0
    V2[:, :, 8:12] -= 3.0
    O2, L2 = oracle.fwd_masked(Q, K2, V2, 0.7, False, bmask, bsize=bs)
    assert np.allclose(O1[:, :, 4:8], O2[:, :, 4:8], rtol=0, atol=1e-14)
    assert np.allclose(L1[:, :, 4:8], L2[:, :, 4:8], rtol=0, atol=1e-14)
    assert not np.allclose(O1[:, :, 0:4], O2[:, :, 0:4])  # unmasked rows do change


def test_fully_masked_rows_and_all_ones_mask():
    B, Hq, N, d, bs = 1, 1, 8, 3, 4
    Q, K, V, dO = _rand(B, Hq, N, d), _rand(B, Hq, N, d), _rand(B, Hq, N, d), _rand(B, Hq, N, d)
    bmask = np.array([[[0, 0], [1, 1]]], dtype=np.uint8)
    O, L = oracle.fwd_masked(Q, K, V, 0.3, False, bmask, bsize=bs)
    assert np.all(O[:, :, :4] == 0.0) and np.all(np.isneginf(L[:, :, :4]))
    g = oracle.bwd_masked(Q, K, V, dO, 0.3, False, bmask, bsize=bs)
    assert np.all(g["dQ"][:, :, :4] == 0.0)
    ones = np.ones((1, 2, 2), dtype=np.uint8)
    Om, Lm = oracle.fwd_masked(Q, K, V, 0.3, True, ones, bsize=bs)
    Od, Ld = oracle.fwd(Q, K, V, 0.3, True)
    assert np.array_equal(Om, Od) and np.array_equal(Lm, Ld)
    gm = oracle.bwd_masked(Q, K, V, dO, 0.3, True, ones, bsize=bs)
    gd = oracle.bwd(Q, K, V, dO, 0.3, True)
    for k in ("dQ", "dK", "dV"):
        assert np.array_equal(gm[k], gd[k])


@pytest.mark.parametrize("causal", [False, True])
def test_masked_backward_finite_differences(causal):
    B, Hq, Hkv, N, d, bs = 1, 2, 1, 6, 3, 2
    Q, K, V, dO = _rand(B, Hq, N, d), _rand(B, Hkv, N, d), _rand(B, Hkv, N, d), _rand(B, Hq, N, d)
    bmask = np.array([[[1, 0, 1], [1, 1, 0], [0, 1, 1]]], dtype=np.uint8)
    scale, h = 0.6, 1e-5
    g = oracle.bwd_masked(Q, K, V, dO, scale, causal, bmask, bsize=bs)

    def loss(Qx, Kx, Vx):
        O, _ = oracle.fwd_masked(Qx, Kx, Vx, scale, causal, bmask, bsize=bs)
        return float((O * dO).sum())

    for name, X in (("dQ", Q), ("dK", K), ("dV", V)):
        num = np.zeros_like(X)
        it = np.nditer(X, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += h
            Xm[idx] -= h
            args_p = [Q, K, V]
            args_m = [Q, K, V]
            k = {"dQ": 0, "dK": 1, "dV": 2}[name]
            args_p[k], args_m[k] = Xp, Xm
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        err = np.abs(num - g[name]).max() / max(np.abs(g[name]).max(), 1e-12)
        assert err < 1e-6, (name, err)
