"""The FP8 forward's parity bound holds for a model of its rounding (CPU only).

tests/test_fp8_parity.py compares the GPU's FP8 forward with the fp64 oracle
under a per-element bound derived from the e4m3 rounding of the
probabilities.  Here a plain numpy model of that arithmetic -- the block
scales folded into the exponent, a running max that moves only when a tile's
max exceeds it by more than 2^4, the exponent offset by +4, P' = P * r_j
rounded to e4m3 (the reference rounding of oracle/fp8.py), row sums from the
unrounded P, and the divisor corrected by the rounding of each tile's
largest P' -- is checked against the oracle under the same bound, on inputs
whose block magnitudes differ (so that r_j < 1 and small P' reach the
subnormal range).  A bound that the model can break would be no bound.
"""

import numpy as np
import pytest

import oracle
from oracle import fp8 as ofp8

from test_fp8_parity import _o_bound_rows

RNG = np.random.default_rng(0xF8B0)


def _blocky(shape, exps):
    x = RNG.standard_normal(shape)
    N = shape[1]
    mul = np.exp2(RNG.choice(exps, size=(shape[0], -(-N // 128))))
    return x * np.repeat(mul, 128, axis=1)[:, :N, None]


def _model_row(q, K, V, sv, scale, causal, i, threshold=4.0, shift=4.0):
    """The FP8 forward's arithmetic for one query row (fp64 except the e4m3 step)."""
    N = K.shape[0]
    T = -(-N // 128)
    lsvm = np.log2(sv.max())
    m, l, corr = -np.inf, 0.0, 0.0
    o = np.zeros(V.shape[1])
    for j in range(T):
        ks = slice(128 * j, min(128 * (j + 1), N))
        s = (K[ks] @ q) * scale * np.log2(np.e)  # scaled score, log2 units
        keys = np.arange(ks.start, ks.stop)
        s = np.where(keys <= i if causal else np.ones_like(keys, bool), s, -np.inf)
        mx = s.max()
        if mx > m + threshold:
            alpha = 0.0 if m == -np.inf else np.exp2(m - mx)
            l, corr, o = l * alpha, corr * alpha, o * alpha
            m = mx
        m_use = 0.0 if m == -np.inf else m - shift
        lr = np.log2(sv[j]) - lsvm
        p = np.exp2(s + lr - m_use)  # P' = P r_j
        pq = ofp8.round_e4m3(p)
        rinv = 2.0 ** -lr
        l += rinv * p.sum()
        pmax = np.exp2(mx + lr - m_use)
        corr += rinv * (pmax - ofp8.round_e4m3(pmax))
        o += pq @ (V[ks] / sv[j])  # the codes of V: V / sv_j
    lo = l - corr
    return o * sv.max() / lo if lo > 0 else o * 0.0


@pytest.mark.parametrize("N,causal,exps", [(300, True, (-1, 0, 1)), (260, False, (-2, 0, 2)),
                                           (384, True, (2, 3))])
def test_model_of_fp8_rounding_stays_within_the_bound(N, causal, exps):
    d = 32
    Q, K, V = _blocky((1, N, d), exps), _blocky((1, N, d), exps), _blocky((1, N, d), exps)
    qc, sq = ofp8.quantize_blocks(Q)
    kc, sk = ofp8.quantize_blocks(K)
    vc, sv = ofp8.quantize_blocks(V)
    Qd, Kd, Vd = (ofp8.dequantize_blocks(c, s)[0] for c, s in ((qc, sq), (kc, sk), (vc, sv)))
    scale = 1.0 / np.sqrt(d)
    Oref, _ = oracle.fwd(Qd[None, None], Kd[None, None], Vd[None, None], scale, causal)
    Oref = Oref[0, 0]
    rows = np.arange(N)
    Om = np.stack([_model_row(Qd[i], Kd, Vd, sv[0].astype(np.float64), scale, causal, i) for i in rows])
    bound = _o_bound_rows(Qd, Kd, Vd, sv[0].astype(np.float64), scale, causal, rows, Oref)
    err = np.abs(Om - Oref)
    assert np.all(err <= bound), float((err / bound).max())
    # The bound is not vacuous: the model's rounding error is a visible share of it.
    assert (err / bound).max() > 0.05
