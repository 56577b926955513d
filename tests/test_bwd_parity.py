"""Backward parity: CUDA library (through the C ABI) vs the fp64 oracle.

The GPU backward consumes the GPU forward's O and LSE, exactly as a caller
would.  Small and medium shapes, the d=64 workload and the causal d=128
workload are compared over every element of dQ, dK and dV against the
oracle's own full backward.  The two long workloads (N = 16384 and 131072)
are compared at full size on seeded sampled rows: dQ rows are recomputed by
the oracle from scratch; dK/dV rows use the oracle with the GPU's LSE (itself
checked on sampled rows) and D recomputed on the CPU from the GPU's O and dO,
because exact per-key-row references need every query row's statistics.
Whole-tensor invariants back those up: sum_j dK_j = 0 and sum_j dV_j =
sum_i dO_i within each kv-head group.
"""

import numpy as np
import pytest
import torch

import oracle
import exact_attention_95_gb300 as pkg
from exact_attention_95_gb300 import inputs

from parity import GRAD_TOL, LSE_TOL, check_o, f64, make, rel_err, to_dev, workload_reference

pytestmark = pytest.mark.gpu


def _gpu_fwd_bwd(g, scale, causal):
    O, L = pkg.attn_fwd(g["Q"], g["K"], g["V"], scale, causal)
    dQ, dK, dV = pkg.attn_bwd(g["Q"], g["K"], g["V"], O, g["dO"], L, scale, causal)
    torch.cuda.synchronize()
    assert pkg.attn_last_device_status() == pkg.ATTN_OK
    return O, L, dQ, dK, dV


SHAPES = [
    # B, Hq, Hkv, N, d
    (1, 1, 1, 1, 64),
    (1, 2, 1, 65, 128),
    (1, 2, 2, 128, 64),
    (2, 2, 1, 191, 128),
    (1, 4, 2, 300, 64),
    (1, 8, 2, 513, 128),
    (1, 2, 2, 1024, 64),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B%dHq%dHkv%dN%dd%d" % s)
def test_bwd_full_parity(shape, causal):
    B, Hq, Hkv, N, d = shape
    t = make(B, Hq, Hkv, N, d, seed=4000 + N + d)
    g = {k: to_dev(v) for k, v in t.items()}
    scale = 1.0 / np.sqrt(d)
    O, L, dQ, dK, dV = _gpu_fwd_bwd(g, scale, causal)
    f = {k: inputs.to_f64(v) for k, v in t.items()}
    ref = oracle.bwd(f["Q"], f["K"], f["V"], f["dO"], scale, causal)
    for name, x in (("dQ", dQ), ("dK", dK), ("dV", dV)):
        e = rel_err(f64(x), ref[name])
        assert e <= GRAD_TOL, f"{name} rel err {e:.3e}"
    assert np.abs(f64(L) - ref["LSE"]).max() <= LSE_TOL


def test_bwd_large_logits_gqa():
    # Q x8 (logit std ~8) with GQA 4:1, causal, d=128, ragged N.
    t = make(1, 8, 2, 700, 128, seed=99, q_mul=8.0)
    g = {k: to_dev(v) for k, v in t.items()}
    scale = 1.0 / np.sqrt(128)
    O, L, dQ, dK, dV = _gpu_fwd_bwd(g, scale, True)
    f = {k: inputs.to_f64(v) for k, v in t.items()}
    ref = oracle.bwd(f["Q"], f["K"], f["V"], f["dO"], scale, True)
    for name, x in (("dQ", dQ), ("dK", dK), ("dV", dV)):
        e = rel_err(f64(x), ref[name])
        assert e <= GRAD_TOL, f"{name} rel err {e:.3e}"


def test_bwd_repeatable():
    # dQ is accumulated with fp32 atomics (order may vary); dK and dV are not.
    t = make(1, 4, 2, 384, 128, seed=7)
    g = {k: to_dev(v) for k, v in t.items()}
    a = _gpu_fwd_bwd(g, 0.09, True)
    b = _gpu_fwd_bwd(g, 0.09, True)
    assert torch.equal(a[3], b[3]) and torch.equal(a[4], b[4])
    assert rel_err(f64(a[2]), f64(b[2])) < 1e-2


@pytest.mark.parametrize("name", ["c2", "c3"])
def test_bwd_workload_every_element(name):
    """The d=64 workload (B4 H16 N1024, non-causal) and the causal d=128 Q x8
    workload (B2 H32 N4096) in the benchmark's launch configuration, against
    the oracle's own full fp64 forward and backward: every element of O, LSE,
    dQ, dK and dV.  Nothing of the reference comes from the GPU (the oracle
    computes its own LSE and D)."""
    w, t, ref = workload_reference(name)
    g = {k: to_dev(v) for k, v in t.items()}
    O, L, dQ, dK, dV = _gpu_fwd_bwd(g, w.scale, w.causal)
    err, ok = check_o(f64(O), ref["O"], bf16_out=True)
    assert ok, f"O max-abs {err:.3e}"
    assert np.abs(f64(L) - ref["LSE"]).max() <= LSE_TOL
    for nm, x in (("dQ", dQ), ("dK", dK), ("dV", dV)):
        e = rel_err(f64(x), ref[nm])
        assert e <= GRAD_TOL, f"{nm} rel err {e:.3e}"


@pytest.mark.parametrize("name", ["c4", "c5"])
def test_bwd_workload_sampled_rows(name):
    """The long workloads at full size in the benchmark's launch configuration."""
    w = inputs.WORKLOADS[name]
    t = inputs.workload_tensors(w)
    g = {k: to_dev(v) for k, v in t.items()}
    O, L, dQ, dK, dV = _gpu_fwd_bwd(g, w.scale, w.causal)
    f = {k: inputs.to_f64(v) for k, v in t.items()}
    total_q = w.B * w.Hq * w.N
    total_k = w.B * w.Hkv * w.N
    qrows = inputs.sample_rows(0xD0 + w.config_id, total_q, 512, must=[0, 1, 127, 128, w.N - 1])
    krows = inputs.sample_rows(0xE0 + w.config_id, total_k, 512, must=[0, 1, 127, 128, w.N - 1])
    qi = torch.from_numpy(qrows).cuda()
    ki = torch.from_numpy(krows).cuda()
    d = w.d
    # Forward statistics on the sampled query rows.
    Oref, Lref = oracle.fwd_rows(f["Q"], f["K"], f["V"], w.scale, w.causal, qrows)
    err, ok = check_o(f64(O.reshape(-1, d)[qi]), Oref, bf16_out=True)
    assert ok, f"O max-abs {err:.3e}"
    assert np.abs(f64(L.reshape(-1)[qi]) - Lref).max() <= LSE_TOL
    # dQ rows: fully independent oracle rows.
    dq_ref = oracle.bwd_dq_rows(f["Q"], f["K"], f["V"], f["dO"], w.scale, w.causal, qrows)
    e = rel_err(f64(dQ.reshape(-1, d)[qi]), dq_ref)
    assert e <= GRAD_TOL, f"dQ rel err {e:.3e}"
    # dK, dV rows with the GPU LSE and D = rowsum(dO * O_gpu) computed here
    # (an exact reference for a key row needs the statistics of every query
    # row: a full fp64 forward, out of reach on the host at these lengths).
    Lg = f64(L)
    Dg = (f["dO"] * f64(O)).sum(-1)
    dk_ref, dv_ref = oracle.bwd_dkv_rows(f["Q"], f["K"], f["V"], f["dO"], Lg, Dg, w.scale, w.causal,
                                         krows)
    e = rel_err(f64(dK.reshape(-1, d)[ki]), dk_ref)
    assert e <= GRAD_TOL, f"dK rel err {e:.3e}"
    e = rel_err(f64(dV.reshape(-1, d)[ki]), dv_ref)
    assert e <= GRAD_TOL, f"dV rel err {e:.3e}"
    # Whole-tensor invariants (exact in real arithmetic), per (b, kv head).
    G = w.Hq // w.Hkv
    dKs = dK.double().sum(2)
    dVs = dV.double().sum(2)
    dOs = g["dO"].double().sum(2).reshape(w.B, w.Hkv, G, d).sum(2)
    l1k = dK.double().abs().sum(2)
    l1v = dV.double().abs().sum(2)
    assert float((dKs.abs() / l1k.clamp_min(1e-30)).max()) < 1e-2
    assert float(((dVs - dOs).abs() / l1v.clamp_min(1e-30)).max()) < 1e-2
    assert torch.isfinite(dQ).all() and torch.isfinite(dK).all() and torch.isfinite(dV).all()


def test_wait_timeout_is_reported():
    # A bounded wait on a barrier that nothing completes must come back as a
    # status, leaving the context usable.
    assert pkg.attn_last_device_status() == pkg.ATTN_OK
    assert pkg.attn_selftest_wait_timeout(20_000_000) == pkg.ATTN_OK
    assert pkg.attn_last_device_status() == pkg.ATTN_ERR_TIMEOUT
    assert pkg.attn_last_device_status() == pkg.ATTN_OK  # cleared by the read
    x = torch.ones(4, device="cuda")
    assert float(x.sum()) == 4.0
