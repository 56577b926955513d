"""The C-ABI library loads, exports every declared symbol, and rejects bad
arguments on the host before touching the GPU (no GPU needed)."""

import ctypes
import os
import re

import pytest

import exact_attention_95_gb300 as pkg
from exact_attention_95_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn), encoding="utf-8").read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(attn_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return pkg.load_library()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert {"attn_fwd", "attn_bwd", "attn_bwd_workspace_size", "attn_status_string",
            "attn_last_device_status"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
    assert set(pkg.EXPORTED) == set(names)


def test_status_strings(lib):
    for code, name in [(0, "ATTN_OK"), (1, "ATTN_ERR_INVALID_ARG"), (2, "ATTN_ERR_UNSUPPORTED"),
                       (3, "ATTN_ERR_CUDA"), (4, "ATTN_ERR_TIMEOUT"), (5, "ATTN_ERR_DEVICE")]:
        assert pkg.attn_status_string(code) == name


def test_workspace_size(lib):
    # fp32 dQ accumulator over N rounded up to 64, plus two fp32 row vectors.
    n = pkg.attn_bwd_workspace_size(2, 4, 2, 100, 64)
    rows = 2 * 4 * 128
    assert n == rows * 64 * 4 + 2 * rows * 4
    assert pkg.attn_bwd_workspace_size(1, 3, 2, 100, 64) == 0  # Hq % Hkv
    assert pkg.attn_bwd_workspace_size(1, 1, 1, 100, 96) == 0  # unsupported d


A = ctypes.c_void_p(0x10000)  # fake, aligned; never dereferenced on these paths


def _fwd(lib, **kw):
    a = dict(Q=A, K=A, V=A, O=A, LSE=A, B=1, Hq=2, Hkv=1, N=128, d=64, scale=0.125, causal=0,
             ind=0, outd=0)
    a.update(kw)
    return lib.attn_fwd(a["Q"], a["K"], a["V"], a["O"], a["LSE"], a["B"], a["Hq"], a["Hkv"],
                        a["N"], a["d"], a["scale"], a["causal"], a["ind"], a["outd"], None)


def test_fwd_argument_errors(lib):
    assert _fwd(lib, Q=None) == pkg.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, LSE=None) == pkg.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, K=ctypes.c_void_p(0x10008)) == pkg.ATTN_ERR_INVALID_ARG  # misaligned
    assert _fwd(lib, N=0) == pkg.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, B=-1) == pkg.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, Hq=3, Hkv=2) == pkg.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, scale=float("nan")) == pkg.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, causal=2) == pkg.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, ind=7) == pkg.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, d=256) == pkg.ATTN_ERR_UNSUPPORTED
    assert _fwd(lib, d=80) == pkg.ATTN_ERR_UNSUPPORTED
    assert _fwd(lib, ind=pkg.ATTN_F32, outd=pkg.ATTN_BF16) == pkg.ATTN_ERR_UNSUPPORTED
    assert _fwd(lib, N=128 * 65536) == pkg.ATTN_ERR_UNSUPPORTED


def _bwd(lib, **kw):
    a = dict(ws=A, wsb=1 << 30, B=1, Hq=2, Hkv=1, N=128, d=64, dtype=0, causal=1)
    a.update(kw)
    return lib.attn_bwd(A, A, A, A, A, A, A, A, A, a["B"], a["Hq"], a["Hkv"], a["N"], a["d"],
                        0.125, a["causal"], a["dtype"], a["ws"], a["wsb"], None)


def test_bwd_argument_errors(lib):
    assert _bwd(lib, ws=None) == pkg.ATTN_ERR_INVALID_ARG
    assert _bwd(lib, ws=ctypes.c_void_p(0x10010)) == pkg.ATTN_ERR_INVALID_ARG  # not 256-aligned
    assert _bwd(lib, wsb=16) == pkg.ATTN_ERR_INVALID_ARG
    assert _bwd(lib, Hq=4, Hkv=3) == pkg.ATTN_ERR_INVALID_ARG
    assert _bwd(lib, d=32) == pkg.ATTN_ERR_UNSUPPORTED
    assert _bwd(lib, dtype=pkg.ATTN_F32) == pkg.ATTN_ERR_UNSUPPORTED
    assert _bwd(lib, dtype=9) == pkg.ATTN_ERR_INVALID_ARG


def test_missing_library_fails_loudly(tmp_path):
    import importlib
    mod = importlib.import_module("exact_attention_95_gb300")
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        # a fresh load from a path that does not exist
        saved = mod._lib
        try:
            mod._lib = None
            mod.load_library(str(tmp_path / "missing.so"))
        finally:
            mod._lib = saved


def _split_ws(rows, d, splits):
    o = (splits * rows * d * 4 + 255) // 256 * 256
    return o + (splits * rows * 4 + 255) // 256 * 256


def test_fwd_split_workspace_size(lib):
    ws = pkg.attn_fwd_split_workspace_size
    assert ws(1, 4, 2, 1, 4096, 128, 1) == 0  # one split: written directly, no workspace
    # 8 key tiles in 4 splits of 2.
    assert ws(2, 4, 2, 3, 1024, 128, 4) == _split_ws(2 * 4 * 3, 128, 4)
    # More splits than tiles are capped at one split per tile.
    assert ws(1, 2, 1, 5, 200, 64, 5) == _split_ws(1 * 2 * 5, 64, 2)
    # 8 tiles over 7 requested splits: tiles of 2, hence 4 non-empty splits.
    assert ws(1, 1, 1, 1, 1024, 64, 7) == _split_ws(1, 64, 4)
    assert ws(1, 1, 1, 1, 1024, 64, -1) == 0
    assert ws(1, 1, 1, 1, 1024, 64, 257) == 0
    assert ws(1, 1, 1, 0, 1024, 64, 2) == 0
    assert ws(1, 1, 1, 1, 1024, 96, 2) == 0
    assert ws(1, 3, 2, 1, 1024, 64, 2) == 0  # Hq % Hkv


def _fwd_split(lib, **kw):
    a = dict(Q=A, K=A, V=A, O=A, LSE=A, B=1, Hq=2, Hkv=1, Nq=16, Nk=1024, d=64, scale=0.125, causal=1,
             outd=0, splits=4, ws=None, wsb=0)
    a.update(kw)
    return lib.attn_fwd_split(a["Q"], a["K"], a["V"], a["O"], a["LSE"], a["B"], a["Hq"], a["Hkv"],
                              a["Nq"], a["Nk"], a["d"], a["scale"], a["causal"], a["outd"], a["splits"],
                              a["ws"], a["wsb"], None)


def test_fwd_split_argument_errors(lib):
    assert _fwd_split(lib, Q=None) == pkg.ATTN_ERR_INVALID_ARG
    assert _fwd_split(lib, Nk=0) == pkg.ATTN_ERR_INVALID_ARG
    assert _fwd_split(lib, Nq=0) == pkg.ATTN_ERR_INVALID_ARG
    assert _fwd_split(lib, splits=-2) == pkg.ATTN_ERR_INVALID_ARG
    assert _fwd_split(lib, splits=300) == pkg.ATTN_ERR_INVALID_ARG
    assert _fwd_split(lib, outd=7) == pkg.ATTN_ERR_INVALID_ARG
    assert _fwd_split(lib, d=256) == pkg.ATTN_ERR_UNSUPPORTED
    assert _fwd_split(lib, Hq=3, Hkv=2) == pkg.ATTN_ERR_INVALID_ARG
    # A split run needs the workspace: missing, short or misaligned.
    assert _fwd_split(lib) == pkg.ATTN_ERR_INVALID_ARG
    need = pkg.attn_fwd_split_workspace_size(1, 2, 1, 16, 1024, 64, 4)
    assert _fwd_split(lib, ws=A, wsb=need - 1) == pkg.ATTN_ERR_INVALID_ARG
    assert _fwd_split(lib, ws=ctypes.c_void_p(0x10010), wsb=need) == pkg.ATTN_ERR_INVALID_ARG


def test_masked_argument_errors(lib):
    M = ctypes.c_void_p(0x20000)

    def fwd(**kw):
        a = dict(Q=A, K=A, V=A, O=A, LSE=A, B=1, Hq=2, Hkv=1, N=256, d=64, scale=0.125, causal=1, m=M, mh=1,
                 outd=0)
        a.update(kw)
        return lib.attn_fwd_masked(a["Q"], a["K"], a["V"], a["O"], a["LSE"], a["B"], a["Hq"], a["Hkv"], a["N"],
                                   a["d"], a["scale"], a["causal"], a["m"], a["mh"], a["outd"], None)

    assert fwd(m=None) == pkg.ATTN_ERR_INVALID_ARG
    assert fwd(mh=3) == pkg.ATTN_ERR_INVALID_ARG  # 1 or Hq
    assert fwd(Q=None) == pkg.ATTN_ERR_INVALID_ARG
    assert fwd(d=96) == pkg.ATTN_ERR_UNSUPPORTED
    assert fwd(N=128 * 2049) == pkg.ATTN_ERR_UNSUPPORTED  # more key tiles than a CTA may list

    def bwd(**kw):
        a = dict(B=1, Hq=2, Hkv=1, N=256, d=64, m=M, mh=2, ws=A, wsb=1 << 30)
        a.update(kw)
        return lib.attn_bwd_masked(A, A, A, A, A, A, A, A, A, a["B"], a["Hq"], a["Hkv"], a["N"], a["d"], 0.125, 1,
                                   a["m"], a["mh"], a["ws"], a["wsb"], None)

    assert bwd(m=None) == pkg.ATTN_ERR_INVALID_ARG
    assert bwd(mh=5) == pkg.ATTN_ERR_INVALID_ARG
    assert bwd(ws=None) == pkg.ATTN_ERR_INVALID_ARG
    assert bwd(Hq=64, Hkv=1, N=128 * 65, mh=1) == pkg.ATTN_ERR_UNSUPPORTED  # 64 x 65 > 4096 pairs


def test_fp8_argument_errors(lib):
    assert lib.attn_fp8_vt_stride(1) == 16 and lib.attn_fp8_vt_stride(4096) == 4096
    assert lib.attn_fp8_vt_stride(300) == 304 and lib.attn_fp8_vt_stride(0) == 0
    S = ctypes.c_void_p(0x30000)

    def fwd(**kw):
        a = dict(Q=A, sq=S, K=A, sk=S, V=A, sv=S, O=A, LSE=A, B=1, Hq=2, Hkv=1, N=256, d=128, scale=0.125,
                 causal=1, outd=0)
        a.update(kw)
        return lib.attn_fwd_fp8(a["Q"], a["sq"], a["K"], a["sk"], a["V"], a["sv"], a["O"], a["LSE"], a["B"],
                                a["Hq"], a["Hkv"], a["N"], a["d"], a["scale"], a["causal"], a["outd"], None)

    assert fwd(sq=None) == pkg.ATTN_ERR_INVALID_ARG
    assert fwd(sv=None) == pkg.ATTN_ERR_INVALID_ARG
    assert fwd(sk=ctypes.c_void_p(0x30002)) == pkg.ATTN_ERR_INVALID_ARG  # misaligned scales
    assert fwd(V=ctypes.c_void_p(0x10008)) == pkg.ATTN_ERR_INVALID_ARG
    assert fwd(scale=0.0) == pkg.ATTN_ERR_INVALID_ARG
    assert fwd(scale=-0.125) == pkg.ATTN_ERR_INVALID_ARG
    assert fwd(outd=5) == pkg.ATTN_ERR_INVALID_ARG
    assert fwd(Hq=3, Hkv=2) == pkg.ATTN_ERR_INVALID_ARG
    assert fwd(d=64) == pkg.ATTN_ERR_UNSUPPORTED  # the FP8 kernel is d = 128 only

    def quant(**kw):
        a = dict(X=A, c=A, s=S, BH=4, N=300, d=128, tr=1)
        a.update(kw)
        return lib.attn_quantize_fp8(a["X"], a["c"], a["s"], a["BH"], a["N"], a["d"], a["tr"], None)

    assert quant(X=None) == pkg.ATTN_ERR_INVALID_ARG
    assert quant(s=None) == pkg.ATTN_ERR_INVALID_ARG
    assert quant(N=0) == pkg.ATTN_ERR_INVALID_ARG
    assert quant(BH=0) == pkg.ATTN_ERR_INVALID_ARG
    assert quant(tr=2) == pkg.ATTN_ERR_INVALID_ARG
    assert quant(c=ctypes.c_void_p(0x10004)) == pkg.ATTN_ERR_INVALID_ARG
    assert quant(d=96) == pkg.ATTN_ERR_UNSUPPORTED


def test_nonpositive_scale_is_rejected(lib):
    # The kernels take the row max on the unscaled scores: the scale must be > 0.
    assert _fwd(lib, scale=0.0) == pkg.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, scale=-1.0) == pkg.ATTN_ERR_INVALID_ARG


def test_binding_rejects_host_and_mistyped_tensors():
    # The Python layer checks placement, dtype, shape and contiguity before
    # any call reaches the library (no GPU needed for these paths).
    import torch
    x = torch.zeros(1, 2, 8, 128, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        pkg.attn_fwd(x, x, x, 0.1, True)  # host tensors
    with pytest.raises(TypeError):
        pkg.attn_fwd(x.int(), x, x, 0.1, True)  # unsupported dtype
    with pytest.raises(TypeError):
        pkg.attn_quantize_fp8(x)  # host tensor
    codes = torch.zeros(1, 2, 8, 128, dtype=torch.uint8)
    sc = torch.ones(1, 2, 1)
    with pytest.raises(TypeError):
        pkg.attn_fwd_fp8(codes, sc, codes, sc, codes, sc, 0.1, True)
    with pytest.raises(TypeError):
        pkg.attn_fwd_masked(x, x, x, torch.ones(1, 1, 1, dtype=torch.uint8), 0.1, True)


def test_binding_rejects_bad_backward_outputs_and_workspace():
    # Outputs and the workspace become kernel write targets: they are checked
    # like inputs.  On a machine without a GPU the helpers are called directly.
    import torch
    x = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        pkg.attn_bwd(x, x, x, x, x, torch.zeros(1, 2, 8), 0.1, True)  # host inputs
    with pytest.raises(TypeError):
        pkg._check_bwd_outputs(x, x, x, 1, 2, 2, 8, 64, None)  # host dQ
    with pytest.raises(TypeError):
        pkg._check_workspace(torch.zeros(16, dtype=torch.uint8), 16, None)  # host workspace
    with pytest.raises(TypeError):
        pkg.attn_bwd_noalloc(x, x, x, x, x, torch.zeros(1, 2, 8), 0.1, True)
    with pytest.raises(TypeError):
        pkg.attn_bwd_masked(x, x, x, x, x, torch.zeros(1, 2, 8), torch.ones(1, 1, 1, dtype=torch.uint8),
                            0.1, True)


@pytest.mark.gpu
def test_binding_rejects_bad_backward_outputs_on_gpu():
    import torch
    dev = torch.device("cuda")
    q = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16, device=dev)
    lse = torch.zeros(1, 2, 8, device=dev)
    good = dict(dQ=torch.empty_like(q), dK=torch.empty_like(q), dV=torch.empty_like(q))
    bad_cases = [
        (TypeError, dict(dQ=torch.empty(1, 2, 8, 64, dtype=torch.bfloat16))),        # host output
        (TypeError, dict(dK=torch.empty(1, 2, 8, 64, dtype=torch.float32, device=dev))),  # fp32 output
        (ValueError, dict(dV=torch.empty(1, 2, 8, 32, dtype=torch.bfloat16, device=dev))),  # wrong shape
        (TypeError, dict(workspace=torch.empty(1 << 20, dtype=torch.uint8))),       # host workspace
        (TypeError, dict(workspace=torch.empty(1 << 18, dtype=torch.float32, device=dev))),
        (ValueError, dict(workspace=torch.empty(16, dtype=torch.uint8, device=dev))),  # too small
    ]
    for exc, kw in bad_cases:
        args = dict(good, **kw)
        with pytest.raises(exc):
            pkg.attn_bwd(q, q, q, q, q, lse, 0.125, True, **args)
        if "workspace" not in kw:
            with pytest.raises(exc):
                pkg.attn_bwd_noalloc(q, q, q, q, q, lse, 0.125, True, **args)
    with pytest.raises(TypeError):
        pkg.attn_fwd(q, q, q, 0.125, True, O=torch.empty(1, 2, 8, 64, dtype=torch.bfloat16))
