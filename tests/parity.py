"""Helpers shared by the GPU parity tests: seeded inputs, transfer, metrics.

Tolerances (the stated bars):
  fp32 path:   O and LSE max-abs <= 1e-5
  bf16 path:   O max-abs <= 1e-2 (fp32 O output); bf16 O output is allowed one
               extra half-ulp of bf16 at the reference value (the rounding of
               the output itself); LSE max-abs <= 1e-3;
               dQ, dK, dV: max-abs error / max-abs reference <= 2e-2.
"""

import functools

import numpy as np
import torch

import oracle
from exact_attention_95_gb300 import inputs

O_TOL = 1e-2
LSE_TOL = 1e-3
GRAD_TOL = 2e-2
F32_TOL = 1e-5


def make(B, Hq, Hkv, N, d, seed, dtype="bf16", q_mul=1.0, names=("Q", "K", "V", "dO")):
    """Seeded tensors (numpy bf16 bits / fp32), seeds seed + tensor id."""
    out = {}
    for name in names:
        H = Hkv if name in ("K", "V") else Hq
        mul = q_mul if name == "Q" else 1.0
        out[name] = inputs.make_tensor(seed + inputs.TENSOR_IDS[name], (B, H, N, d), dtype, mul)
    return out


def to_dev(a, device="cuda"):
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(a).to(device)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().double().cpu().numpy()


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    """Half a unit in the last place of bf16 at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    e = np.floor(np.log2(ax))
    return 2.0 ** (e - 8)


def check_o(o_gpu: np.ndarray, o_ref: np.ndarray, bf16_out: bool, tol=O_TOL):
    err = np.abs(o_gpu - o_ref)
    bound = tol + (bf16_half_ulp(o_ref) if bf16_out else 0.0)
    worst = float((err - bound).max()) if err.size else -1.0
    return float(err.max()) if err.size else 0.0, worst <= 0.0


def rel_err(x: np.ndarray, ref: np.ndarray) -> float:
    den = float(np.abs(ref).max())
    return float(np.abs(x - ref).max()) / den if den > 0 else float(np.abs(x).max())


@functools.lru_cache(maxsize=2)
def workload_reference(name):
    """The seeded inputs of a named workload and the oracle's full fp64 forward
    and backward on them: (workload, inputs as stored, oracle result dict with
    O, LSE, D, dQ, dK, dV).  Cached, because the causal d=128 workload costs
    tens of seconds on the host cores and both the forward and the backward
    tests compare against it."""
    w = inputs.WORKLOADS[name]
    t = inputs.workload_tensors(w)
    f = {k: inputs.to_f64(v) for k, v in t.items()}
    ref = oracle.bwd(f["Q"], f["K"], f["V"], f["dO"], w.scale, w.causal)
    return w, t, ref
