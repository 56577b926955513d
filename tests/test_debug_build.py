"""The debug variant of the library (-DATTN_DEBUG: explicit bounds checks on
tensor-copy coordinates and store indices, recorded in the device status word
instead of trapping) builds for sm_103a and exports the same C ABI.  On a GPU
it runs a small forward and backward with every check passing and the
release library's results."""

import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest

import exact_attention_95_gb300 as pkg
from exact_attention_95_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_debug_variant_builds_and_exports_the_abi():
    path = libbuild.build(debug=True)
    assert path.endswith("libattn_sm103_debug.so") and os.path.exists(path)
    lib = ctypes.CDLL(path)
    for name in pkg.EXPORTED:
        assert hasattr(lib, name), name


_GPU_SCRIPT = r"""
import numpy as np, torch
import exact_attention_95_gb300 as pkg
from parity import make, to_dev, f64, rel_err
assert pkg.LIB_PATH.endswith("_debug.so")
res = {}
for (B, Hq, Hkv, N, d, causal) in [(1, 4, 2, 300, 128, True), (2, 2, 2, 257, 64, False),
                                    (1, 2, 1, 640, 128, True)]:
    t = make(B, Hq, Hkv, N, d, seed=7100 + N)
    g = {k: to_dev(v) for k, v in t.items()}
    s = 1.0 / np.sqrt(d)
    O, L = pkg.attn_fwd(g["Q"], g["K"], g["V"], s, causal)
    dQ, dK, dV = pkg.attn_bwd(g["Q"], g["K"], g["V"], O, g["dO"], L, s, causal)
    Os, Ls = pkg.attn_fwd_split(g["Q"], g["K"], g["V"], s, causal, num_splits=3)
    torch.cuda.synchronize()
    st = pkg.attn_last_device_status()
    assert st == pkg.ATTN_OK, pkg.attn_status_string(st)
    np.save(f"{OUT}/dbg_{N}_{d}.npy", np.stack([f64(O).ravel()[:4096], f64(dQ).ravel()[:4096],
                                                f64(dK).ravel()[:4096], f64(Os).ravel()[:4096]]))
print("debug-ok")
"""


@pytest.mark.gpu
def test_debug_variant_runs_clean_and_matches_release(tmp_path):
    libbuild.build(debug=True)
    env = dict(os.environ, ATTN_DEBUG="1", PYTHONPATH=os.pathsep.join([ROOT, os.path.join(ROOT, "tests")]))
    code = _GPU_SCRIPT.replace("{OUT}", str(tmp_path))
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "debug-ok" in r.stdout, r.stdout + r.stderr
    # The same calls on the release library give the same outputs.
    import torch
    from parity import make, to_dev, f64
    for (B, Hq, Hkv, N, d, causal) in [(1, 4, 2, 300, 128, True), (2, 2, 2, 257, 64, False),
                                        (1, 2, 1, 640, 128, True)]:
        t = make(B, Hq, Hkv, N, d, seed=7100 + N)
        g = {k: to_dev(v) for k, v in t.items()}
        s = 1.0 / np.sqrt(d)
        O, L = pkg.attn_fwd(g["Q"], g["K"], g["V"], s, causal)
        dQ, dK, dV = pkg.attn_bwd(g["Q"], g["K"], g["V"], O, g["dO"], L, s, causal)
        Os, Ls = pkg.attn_fwd_split(g["Q"], g["K"], g["V"], s, causal, num_splits=3)
        torch.cuda.synchronize()
        ref = np.load(tmp_path / f"dbg_{N}_{d}.npy")
        got = np.stack([f64(O).ravel()[:4096], f64(dQ).ravel()[:4096], f64(dK).ravel()[:4096],
                        f64(Os).ravel()[:4096]])
        # The forward is deterministic; dQ's accumulation order is not.
        assert np.array_equal(ref[0], got[0]) and np.array_equal(ref[3], got[3])
        assert np.abs(ref[1:3] - got[1:3]).max() <= 2e-2 * max(np.abs(ref[1:3]).max(), 1e-30)
