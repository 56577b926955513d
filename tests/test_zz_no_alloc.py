"""attn_bwd_noalloc: the backward for callers that cannot allocate device memory.

Its scratch lives in a fixed array inside the library instead of a caller
workspace.  These tests call it through the C ABI (ctypes, raw pointers) and
compare it with attn_bwd, which uses a caller-allocated workspace, within the
backward's parity tolerance, on two calls in a row (the second call starts
from whatever the first left in the shared scratch array).  The file sorts
last so that a run stopping at the first failure has run every other test.
"""

import ctypes

import numpy as np
import pytest
import torch

import exact_attention_95_gb300 as pkg

from parity import GRAD_TOL, f64, make, rel_err, to_dev

pytestmark = pytest.mark.gpu


def _c_fn():
    fn = pkg.load_library().attn_bwd_noalloc
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i32, i32, vp]
    fn.restype = i32
    return fn


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("shape,causal", [((1, 4, 2, 700, 128), True), ((2, 4, 4, 300, 64), False)])
def test_noalloc_matches_workspace_backward_twice(shape, causal):
    B, Hq, Hkv, N, d = shape
    assert pkg.attn_bwd_workspace_size(B, Hq, Hkv, N, d) <= pkg.NOALLOC_SCRATCH_BYTES
    t = make(B, Hq, Hkv, N, d, seed=8800 + N)
    g = {k: to_dev(v) for k, v in t.items()}
    scale = 1.0 / np.sqrt(d)
    O, L = pkg.attn_fwd(g["Q"], g["K"], g["V"], scale, causal)
    ref = pkg.attn_bwd(g["Q"], g["K"], g["V"], O, g["dO"], L, scale, causal)
    torch.cuda.synchronize()
    fn = _c_fn()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        out = [torch.full_like(g["Q"], float("nan")), torch.full_like(g["K"], float("nan")),
               torch.full_like(g["V"], float("nan"))]
        rc = fn(_p(g["Q"]), _p(g["K"]), _p(g["V"]), _p(O), _p(g["dO"]), _p(L), _p(out[0]),
                _p(out[1]), _p(out[2]), B, Hq, Hkv, N, d, scale, int(causal), pkg.ATTN_BF16, stream)
        assert rc == pkg.ATTN_OK, pkg.attn_status_string(rc)
        torch.cuda.synchronize()
        assert pkg.attn_last_device_status() == pkg.ATTN_OK
        for name, x, r in zip(("dQ", "dK", "dV"), out, ref):
            e = rel_err(f64(x), f64(r))
            assert e <= GRAD_TOL, f"{name} rel err {e:.3e}"


def test_noalloc_rejects_sizes_beyond_its_scratch():
    fn = _c_fn()
    A = ctypes.c_void_p(0x10000)
    B, Hq, Hkv, N, d = 2, 32, 32, 4096, 128  # needs a 130 MiB workspace
    assert pkg.attn_bwd_workspace_size(B, Hq, Hkv, N, d) > pkg.NOALLOC_SCRATCH_BYTES
    rc = fn(A, A, A, A, A, A, A, A, A, B, Hq, Hkv, N, d, 0.1, 1, pkg.ATTN_BF16, None)
    assert rc == pkg.ATTN_ERR_UNSUPPORTED
    # A null or misaligned argument is reported as attn_bwd reports it, before
    # the size limit.
    assert fn(None, A, A, A, A, A, A, A, A, B, Hq, Hkv, N, d, 0.1, 1, pkg.ATTN_BF16, None) == \
        pkg.ATTN_ERR_INVALID_ARG
    assert fn(A, A, A, A, A, A, ctypes.c_void_p(0x10008), A, A, B, Hq, Hkv, N, d, 0.1, 1, pkg.ATTN_BF16,
              None) == pkg.ATTN_ERR_INVALID_ARG
    assert fn(A, A, A, A, A, A, A, A, A, B, Hq, Hkv, N, d, 0.1, 1, 9, None) == pkg.ATTN_ERR_INVALID_ARG
    # Invalid sizes still get attn_bwd's own error codes.
    assert fn(A, A, A, A, A, A, A, A, A, 1, 3, 2, 64, 128, 0.1, 1, 0, None) == pkg.ATTN_ERR_INVALID_ARG
    assert fn(A, A, A, A, A, A, A, A, A, 1, 2, 2, 64, 96, 0.1, 1, 0, None) == pkg.ATTN_ERR_UNSUPPORTED


def test_noalloc_python_wrapper_matches_workspace_backward():
    # The same comparison through the package's wrapper (argument checks,
    # current stream), twice in a row.
    B, Hq, Hkv, N, d, causal = 1, 2, 1, 257, 128, True
    t = make(B, Hq, Hkv, N, d, seed=8900)
    g = {k: to_dev(v) for k, v in t.items()}
    scale = 1.0 / np.sqrt(d)
    O, L = pkg.attn_fwd(g["Q"], g["K"], g["V"], scale, causal)
    ref = pkg.attn_bwd(g["Q"], g["K"], g["V"], O, g["dO"], L, scale, causal)
    for _ in range(2):
        out = pkg.attn_bwd_noalloc(g["Q"], g["K"], g["V"], O, g["dO"], L, scale, causal)
        torch.cuda.synchronize()
        assert pkg.attn_last_device_status() == pkg.ATTN_OK
        for name, x, r in zip(("dQ", "dK", "dV"), out, ref):
            e = rel_err(f64(x), f64(r))
            assert e <= GRAD_TOL, f"{name} rel err {e:.3e}"
