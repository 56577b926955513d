"""Pins of the fp64 oracle to facts that do not come from the oracle itself.

Each test states what fixes the expected value: a number printed on the pages
(the worked example, the causal-mask matrices), a closed form, an invariant of
the mathematics, or finite differences of the oracle's own forward (which pins
the backward to the forward independently of how the backward is written).
"""

import math

import numpy as np
import pytest

import oracle


def _rng(seed):
    return np.random.default_rng(seed)


def _d1_problem(scores, values):
    """A d=1 attention row: q=1, k_j=s_j, v_j=values_j, scale=1."""
    n = len(scores)
    Q = np.ones((1, 1, 1, 1))
    K = np.asarray(scores, dtype=np.float64).reshape(1, 1, n, 1)
    V = np.asarray(values, dtype=np.float64).reshape(1, 1, n, 1)
    return Q, K, V


# --------------------------------------------------------------------------
# The worked example ("02 FlashAttention", §8 and exercise 2)
# --------------------------------------------------------------------------

def test_worked_example_forward(golden_example):
    g = golden_example
    Q, K, V = _d1_problem(g["scores"], g["values"])
    O, L = oracle.fwd(Q, K, V, scale=1.0, causal=False)
    assert abs(O[0, 0, 0, 0] - g["split_a.block2.O"][0]) <= 5e-4
    # The page's 0.7518 is a1*1 + a3*1 summed from the probabilities it printed
    # to 4 decimals, so it carries two half-units of rounding: 1e-4.
    assert abs(O[0, 0, 0, 0] - g["softmax.O"][0]) <= 1e-4
    # LSE is not printed on the page; it follows from the printed scores.
    assert abs(L[0, 0, 0] - math.log(sum(math.exp(s) for s in g["scores"]))) <= 1e-12


def test_worked_example_softmax(golden_example):
    a = oracle.softmax3(golden_example["scores"])
    np.testing.assert_allclose(a, golden_example["softmax"], atol=5e-5, rtol=0)
    assert abs(a.sum() - 1.0) < 1e-15


@pytest.mark.parametrize("split", ["split_a", "split_b"])
def test_worked_example_online_merge(golden_example, split):
    g = golden_example
    O, m, l, Ot = oracle.online_row(g["scores"], g["values"], [int(x) for x in g[split]])
    for blk in (1, 2):
        for key, col in (("m", m), ("l", l), ("O", Ot[:, 0])):
            name = f"{split}.block{blk}.{key}"
            if name in g:
                assert abs(col[blk - 1] - g[name][0]) <= 5e-4, name
    assert abs(O[0] - g[f"{split}.block2.O"][0]) <= 5e-4


def test_worked_example_inblock_probabilities(golden_example):
    # Block 1 of split_a: P~ = exp(s - m~) against the in-block max.
    s = np.array(golden_example["scores"][:2])
    p = np.exp(s - s.max())
    np.testing.assert_allclose(p, golden_example["split_a.block1.P"], atol=5e-4)
    # The oracle's online merge with one block of two values must give
    # O = sum(P~ v) / sum(P~) for that block.
    O, m, l, _ = oracle.online_row(s, [1.0, 0.0], [2])
    assert abs(l[0] - p.sum()) < 1e-15 and abs(O[0] - p[0] / p.sum()) < 1e-15


# --------------------------------------------------------------------------
# Online softmax equals the 3-pass form (exercise 1 invariant, exercise 6)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("block", [1, 2, 3, 8, 32, 128])
def test_online_equals_three_pass_fp64(block):
    r = _rng(block)
    n, dv = 300, 4
    s = r.normal(size=n) * 3.0
    v = r.normal(size=(n, dv))
    sizes = [block] * (n // block) + ([n % block] if n % block else [])
    O, m, l, Ot = oracle.online_row(s, v, sizes)
    a = oracle.softmax3(s)
    ref = a @ v
    np.testing.assert_allclose(O, ref, rtol=1e-12, atol=1e-13)
    # Prefix invariant: after each block, l = sum_{k<=j} exp(s_k - m) and
    # O is the softmax of the prefix applied to the prefix of v.
    end = 0
    for t, nb in enumerate(sizes):
        end += nb
        pre = s[:end]
        assert m[t] == pre.max()
        assert abs(l[t] - np.exp(pre - m[t]).sum()) <= 1e-12 * l[t]
        np.testing.assert_allclose(Ot[t], oracle.softmax3(pre) @ v[:end], rtol=1e-11, atol=1e-13)


@pytest.mark.parametrize("block", [2, 8, 32, 128])
def test_blocked_softmax_fp32_study(block):
    # "02 FlashAttention" exercise 6: naive and online softmax agree to ~1e-7 in fp32.
    x = _rng(100 + block).normal(size=1024).astype(np.float32) * 4
    naive = oracle.softmax3_f32(x)
    online = oracle.online_softmax_f32(x, block)
    assert np.abs(naive - online).max() < 1e-6
    exact = oracle.softmax3(x.astype(np.float64))
    assert np.abs(online - exact).max() < 1e-6


# --------------------------------------------------------------------------
# Closed forms of the forward
# --------------------------------------------------------------------------

def test_single_key():
    r = _rng(1)
    Q = r.normal(size=(2, 3, 1, 8))
    K = r.normal(size=(2, 3, 1, 8))
    V = r.normal(size=(2, 3, 1, 8))
    for causal in (False, True):
        O, L = oracle.fwd(Q, K, V, 0.7, causal)
        np.testing.assert_array_equal(O, V)
        np.testing.assert_allclose(L, 0.7 * np.einsum("bhnd,bhnd->bhn", Q, K), rtol=1e-14)


def test_zero_query_gives_means():
    r = _rng(2)
    N, d = 9, 4
    Q = np.zeros((1, 1, N, d))
    K = r.normal(size=(1, 1, N, d))
    V = r.normal(size=(1, 1, N, d))
    O, L = oracle.fwd(Q, K, V, 0.5, False)
    np.testing.assert_allclose(O[0, 0], np.broadcast_to(V[0, 0].mean(0), (N, d)), rtol=1e-13)
    np.testing.assert_allclose(L, math.log(N), rtol=1e-14)
    O, L = oracle.fwd(Q, K, V, 0.5, True)
    prefix = np.cumsum(V[0, 0], axis=0) / np.arange(1, N + 1)[:, None]
    np.testing.assert_allclose(O[0, 0], prefix, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(L[0, 0], np.log(np.arange(1, N + 1)), rtol=1e-14)


def test_constant_values():
    r = _rng(3)
    Q, K = r.normal(size=(1, 2, 7, 5)), r.normal(size=(1, 2, 7, 5))
    O, _ = oracle.fwd(Q, K, np.ones((1, 2, 7, 5)), 0.3, True)
    np.testing.assert_allclose(O, 1.0, rtol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_one_hot_match_closed_form(causal):
    # q_i = c e_{pi(i)}, k_j = e_j: s_ij = scale*c if j == pi(i) else 0, so
    # O_i = (e^{scale c} v_{pi(i)} + sum_{other kept j} v_j) / (e^{scale c} + #others).
    # A transposed S (K Q^T) or a wrong head/batch index moves the weight elsewhere.
    N, c, scale = 6, 3.0, 0.8
    perm = [2, 0, 1, 5, 3, 4] if not causal else [0, 0, 1, 2, 1, 3]
    r = _rng(4)
    Q = np.zeros((1, 1, N, N))
    for i, p in enumerate(perm):
        Q[0, 0, i, p] = c
    K = np.eye(N).reshape(1, 1, N, N)
    V = r.normal(size=(1, 1, N, N))
    O, L = oracle.fwd(Q, K, V, scale, causal)
    for i in range(N):
        kept = [j for j in range(N) if not causal or j <= i]
        w = np.array([math.exp(scale * c) if j == perm[i] else 1.0 for j in kept])
        ref = (w[:, None] * V[0, 0, kept]).sum(0) / w.sum()
        np.testing.assert_allclose(O[0, 0, i], ref, rtol=1e-13)
        assert abs(L[0, 0, i] - math.log(w.sum())) < 1e-13


def test_rows_of_p_sum_to_one():
    # With V = identity (d = N), O is the probability matrix itself.
    r = _rng(5)
    N = 8
    Q = r.normal(size=(1, 1, N, N))
    K = r.normal(size=(1, 1, N, N))
    V = np.eye(N).reshape(1, 1, N, N)
    for causal in (False, True):
        P, _ = oracle.fwd(Q, K, V, 0.9, causal)
        np.testing.assert_allclose(P.sum(-1), 1.0, rtol=0, atol=1e-14)
        assert (P >= 0).all()
        if causal:
            assert np.all(np.triu(P[0, 0], 1) == 0)


def test_shift_invariance():
    # Adding c to a whole logit row ("02 FlashAttention" §5.1) leaves O unchanged and
    # shifts LSE by c.  Realised with one extra dimension: q' = [q, c/scale], k' = [k, 1].
    r = _rng(6)
    B, H, N, d, scale = 1, 2, 10, 4, 0.6
    Q = r.normal(size=(B, H, N, d))
    K = r.normal(size=(B, H, N, d))
    V = r.normal(size=(B, H, N, d))
    c = r.normal(size=(B, H, N)) * 20
    Q2 = np.concatenate([Q, (c / scale)[..., None]], axis=-1)
    K2 = np.concatenate([K, np.ones((B, H, N, 1))], axis=-1)
    V2 = np.concatenate([V, np.zeros((B, H, N, 1))], axis=-1)
    for causal in (False, True):
        O, L = oracle.fwd(Q, K, V, scale, causal)
        O2, L2 = oracle.fwd(Q2, K2, V2, scale, causal)
        np.testing.assert_allclose(O2[..., :d], O, rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(L2, L + c, rtol=1e-13, atol=1e-12)


def test_large_logits_are_safe():
    # Safe softmax ("从Online-Softmax…" 0x02) must not overflow for huge logits.
    Q, K, V = _d1_problem([1000.0, 999.0, -1000.0], [1.0, 2.0, 3.0])
    O, L = oracle.fwd(Q, K, V, 1.0, False)
    e = math.exp(-1.0)
    assert abs(O[0, 0, 0, 0] - (1 + 2 * e) / (1 + e)) < 1e-14
    assert abs(L[0, 0, 0] - (1000 + math.log(1 + e))) < 1e-12


# --------------------------------------------------------------------------
# Causal alignment and GQA indexing ("从Online-Softmax…", 0x09)
# --------------------------------------------------------------------------

def test_causal_masks_match_page(golden_masks):
    for (nq, nk), mask in golden_masks.items():
        np.testing.assert_array_equal(oracle.causal_mask(nq, nk), np.array(mask))


def test_fully_masked_row_is_zero():
    r = _rng(7)
    Q = r.normal(size=(1, 1, 5, 3))
    K = r.normal(size=(1, 1, 2, 3))
    V = r.normal(size=(1, 1, 2, 3)) + 5
    O, L = oracle.fwd(Q, K, V, 1.0, True)
    assert np.all(O[0, 0, :3] == 0) and np.all(np.isneginf(L[0, 0, :3]))
    np.testing.assert_array_equal(O[0, 0, 3], V[0, 0, 0])
    assert np.all(np.isfinite(L[0, 0, 3:]))


def test_gqa_equals_repeated_mha():
    r = _rng(8)
    B, Hq, Hkv, N, d = 2, 6, 2, 7, 5
    Q = r.normal(size=(B, Hq, N, d))
    K = r.normal(size=(B, Hkv, N, d))
    V = r.normal(size=(B, Hkv, N, d))
    dO = r.normal(size=(B, Hq, N, d))
    G = Hq // Hkv
    Kr, Vr = np.repeat(K, G, axis=1), np.repeat(V, G, axis=1)  # head h -> kv head h // G
    for causal in (False, True):
        O, L = oracle.fwd(Q, K, V, 0.4, causal)
        Or, Lr = oracle.fwd(Q, Kr, Vr, 0.4, causal)
        np.testing.assert_array_equal(O, Or)
        np.testing.assert_array_equal(L, Lr)
        g = oracle.bwd(Q, K, V, dO, 0.4, causal)
        gr = oracle.bwd(Q, Kr, Vr, dO, 0.4, causal)
        np.testing.assert_allclose(g["dQ"], gr["dQ"], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(g["dK"], gr["dK"].reshape(B, Hkv, G, N, d).sum(2),
                                   rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(g["dV"], gr["dV"].reshape(B, Hkv, G, N, d).sum(2),
                                   rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------
# Backward: finite differences and invariants
# --------------------------------------------------------------------------

def _loss(Q, K, V, dO, scale, causal):
    O, _ = oracle.fwd(Q, K, V, scale, causal, threads=1)
    return float((O * dO).sum())


@pytest.mark.parametrize("causal,Nq,Nk", [(False, 5, 5), (True, 5, 5), (True, 4, 6), (False, 6, 3),
                                          (True, 6, 3)])
def test_backward_finite_differences(causal, Nq, Nk):
    r = _rng(10 + Nq * 7 + Nk + causal)
    B, Hq, Hkv, d, scale = 1, 2, 1, 3, 0.7
    Q = r.normal(size=(B, Hq, Nq, d))
    K = r.normal(size=(B, Hkv, Nk, d))
    V = r.normal(size=(B, Hkv, Nk, d))
    dO = r.normal(size=(B, Hq, Nq, d))
    g = oracle.bwd(Q, K, V, dO, scale, causal)
    h = 1e-5
    for name, X in (("dQ", Q), ("dK", K), ("dV", V)):
        fd = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += h
            Xm[idx] -= h
            args_p = {"Q": Q, "K": K, "V": V}
            args_m = dict(args_p)
            key = name[1]
            args_p[key], args_m[key] = Xp, Xm
            fd[idx] = (_loss(args_p["Q"], args_p["K"], args_p["V"], dO, scale, causal)
                       - _loss(args_m["Q"], args_m["K"], args_m["V"], dO, scale, causal)) / (2 * h)
        err = np.abs(g[name] - fd).max() / max(np.abs(fd).max(), 1e-300)
        assert err < 1e-6, (name, err)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_invariants(causal):
    # Rows of P sum to one, so sum_j dS_ij = 0; hence sum_j dK_j = 0 and
    # sum_j dV_j = sum_i dO_i within each kv-head group.
    r = _rng(20 + causal)
    B, Hq, Hkv, N, d = 2, 4, 2, 11, 6
    Q = r.normal(size=(B, Hq, N, d)) * 2
    K = r.normal(size=(B, Hkv, N, d))
    V = r.normal(size=(B, Hkv, N, d))
    dO = r.normal(size=(B, Hq, N, d))
    g = oracle.bwd(Q, K, V, dO, 0.5, causal)
    G = Hq // Hkv
    np.testing.assert_allclose(g["dK"].sum(2), 0.0, atol=1e-12)
    np.testing.assert_allclose(g["dV"].sum(2), dO.reshape(B, Hkv, G, N, d).sum((2, 3)),
                               rtol=1e-12, atol=1e-12)
    # D = rowsum(dO * O) is returned alongside.
    np.testing.assert_allclose(g["D"], (dO * g["O"]).sum(-1), rtol=1e-13, atol=1e-14)
    O, L = oracle.fwd(Q, K, V, 0.5, causal)
    np.testing.assert_array_equal(O, g["O"])
    np.testing.assert_array_equal(L, g["LSE"])


def test_row_variants_match_full():
    r = _rng(30)
    B, Hq, Hkv, N, d = 1, 4, 2, 13, 4
    Q = r.normal(size=(B, Hq, N, d))
    K = r.normal(size=(B, Hkv, N, d))
    V = r.normal(size=(B, Hkv, N, d))
    dO = r.normal(size=(B, Hq, N, d))
    for causal in (False, True):
        g = oracle.bwd(Q, K, V, dO, 0.5, causal)
        rows = np.array([0, 5, 12, 13, 30, 51])
        O, L = oracle.fwd_rows(Q, K, V, 0.5, causal, rows)
        np.testing.assert_array_equal(O, g["O"].reshape(-1, d)[rows])
        np.testing.assert_array_equal(L, g["LSE"].reshape(-1)[rows])
        dq = oracle.bwd_dq_rows(Q, K, V, dO, 0.5, causal, rows)
        np.testing.assert_array_equal(dq, g["dQ"].reshape(-1, d)[rows])
        kv = np.array([0, 3, 12, 14, 25])
        dk, dv = oracle.bwd_dkv_rows(Q, K, V, dO, g["LSE"], g["D"], 0.5, causal, kv)
        np.testing.assert_array_equal(dk, g["dK"].reshape(-1, d)[kv])
        np.testing.assert_array_equal(dv, g["dV"].reshape(-1, d)[kv])


def test_oracle_rejects_bad_shapes():
    Q = np.zeros((1, 3, 4, 2))
    K = np.zeros((1, 2, 4, 2))
    with pytest.raises(ValueError):
        oracle.fwd(Q, K, K, 1.0, False)  # Hq % Hkv != 0
    with pytest.raises(ValueError):
        oracle.fwd_rows(np.zeros((1, 1, 4, 2)), np.zeros((1, 1, 4, 2)), np.zeros((1, 1, 4, 2)),
                        1.0, False, [4])
