"""Exact softmax attention for NVIDIA GB300 (sm_103a): Python binding.

A thin ctypes layer over the C ABI in ``include/attn.h`` (``libattn_sm103.so``,
built in-tree by ``exact_attention_95_gb300.build``).  It only marshals
arguments: PyTorch supplies device memory and the current stream, and every
step of the computation runs in the library's CUDA kernels.  If the library
is missing, every call raises; there is no fallback implementation.

Functions carry the C names:

* ``attn_fwd(Q, K, V, scale, causal, out_dtype=None) -> (O, LSE)``
* ``attn_fwd_split(Q, K, V, scale, causal, num_splits=0, ...) -> (O, LSE)``: query
  and key lengths may differ (bottom-right causal alignment); the key range may
  be split, with the partial results merged
* ``attn_fwd_split_workspace_size(B, Hq, Hkv, Nq, Nk, d, num_splits)``
* ``attn_fwd_masked(Q, K, V, block_mask, scale, causal, out_dtype=None)`` and
  ``attn_bwd_masked(Q, K, V, O, dO, LSE, block_mask, scale, causal)``: block-sparse
  attention with a uint8 CUDA mask [1 or Hq, ceil(N/128), ceil(N/128)]
* ``attn_quantize_fp8(X, transpose=False) -> (codes, scales)`` and
  ``attn_fwd_fp8(Qc, q_scale, Kc, k_scale, Vtc, v_scale, scale, causal)``: e4m3
  codes with one fp32 scale per 128-row block (V transposed) and the FP8
  forward on them (d = 128); ``attn_fp8_vt_stride(N)``
* ``attn_bwd(Q, K, V, O, dO, LSE, scale, causal) -> (dQ, dK, dV)``
* ``attn_bwd_workspace_size(B, Hq, Hkv, N, d)``
* ``attn_last_device_status(stream=None)``, ``attn_status_string(code)``
* ``attn_selftest_wait_timeout(limit_ns)``

Tensors are ``[B, H, N, d]`` contiguous CUDA tensors (bf16, or fp32 for the
fp32 forward); ``LSE`` is ``[B, Hq, N]`` fp32.
"""

from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# ATTN_DEBUG=1 selects the debug build (python -m exact_attention_95_gb300.build
# --debug): the same kernels with explicit bounds checks on tensor-copy
# coordinates and store indices, reported through attn_last_device_status as
# ATTN_ERR_DEVICE instead of an access out of bounds.
LIB_PATH = os.path.join(_HERE, "libattn_sm103_debug.so" if os.environ.get("ATTN_DEBUG") == "1"
                        else "libattn_sm103.so")

ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED = 0, 1, 2
ATTN_ERR_CUDA, ATTN_ERR_TIMEOUT, ATTN_ERR_DEVICE = 3, 4, 5
ATTN_BF16, ATTN_F32 = 0, 1

EXPORTED = ("attn_fwd", "attn_fwd_split", "attn_fwd_split_workspace_size", "attn_fwd_masked",
            "attn_bwd_masked", "attn_quantize_fp8", "attn_fp8_vt_stride", "attn_fwd_fp8", "attn_bwd",
            "attn_bwd_preprocess", "attn_bwd_main", "attn_bwd_convert", "attn_bwd_workspace_size",
            "attn_status_string", "attn_last_device_status", "attn_selftest_wait_timeout")
_BWD_STAGES = {"all": "attn_bwd", "preprocess": "attn_bwd_preprocess", "main": "attn_bwd_main",
               "convert": "attn_bwd_convert"}

_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {attn_status_string(code)}")


def load_library(path: str = LIB_PATH):
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"CUDA library {path} is missing; build it with "
                "`python -m exact_attention_95_gb300.build` (there is no CPU fallback)")
        lib = ctypes.CDLL(path)
        vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i32, i32, i32, vp]
        lib.attn_fwd.restype = i32
        for fname in _BWD_STAGES.values():
            fn = getattr(lib, fname)
            fn.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32,
                           i32, i32, vp, sz, vp]
            fn.restype = i32
        lib.attn_fwd_split.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, i32, i32, i32,
                                       vp, sz, vp]
        lib.attn_fwd_split.restype = i32
        lib.attn_fwd_split_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32]
        lib.attn_fwd_split_workspace_size.restype = sz
        lib.attn_fwd_masked.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i32, vp, i32, i32, vp]
        lib.attn_fwd_masked.restype = i32
        lib.attn_bwd_masked.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i32,
                                        vp, i32, vp, sz, vp]
        lib.attn_bwd_masked.restype = i32
        lib.attn_fp8_vt_stride.argtypes = [i32]
        lib.attn_fp8_vt_stride.restype = i32
        lib.attn_quantize_fp8.argtypes = [vp, vp, vp, ctypes.c_longlong, i32, i32, i32, vp]
        lib.attn_quantize_fp8.restype = i32
        lib.attn_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i32, i32, vp]
        lib.attn_fwd_fp8.restype = i32
        lib.attn_bwd_workspace_size.argtypes = [i32, i32, i32, i32, i32]
        lib.attn_bwd_workspace_size.restype = sz
        lib.attn_status_string.argtypes = [i32]
        lib.attn_status_string.restype = ctypes.c_char_p
        lib.attn_last_device_status.argtypes = [vp]
        lib.attn_last_device_status.restype = i32
        lib.attn_selftest_wait_timeout.argtypes = [ctypes.c_ulonglong, vp]
        lib.attn_selftest_wait_timeout.restype = i32
        _lib = lib
        return lib


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _check_tensor(name, t, dtype, shape, device=None):
    """Placement, dtype, shape and contiguity of a tensor handed to the library.

    Outputs are checked like inputs: a host tensor, a wrong dtype or shape
    would otherwise become a kernel's write target."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _check_workspace(ws, need, device):
    """A caller-given workspace: contiguous uint8 CUDA memory on `device`, at
    least `need` bytes."""
    if not isinstance(ws, torch.Tensor) or not ws.is_cuda:
        raise TypeError("workspace must be a CUDA tensor")
    if ws.device != device:
        raise ValueError(f"workspace is on {ws.device}, expected {device}")
    if ws.dtype != torch.uint8 or not ws.is_contiguous():
        raise TypeError("workspace must be a contiguous uint8 tensor")
    if ws.numel() < need:
        raise ValueError(f"workspace has {ws.numel()} bytes, needs {need}")


def _check_bwd_outputs(dQ, dK, dV, B, Hq, Hkv, N, d, device):
    bf = torch.bfloat16
    _check_tensor("dQ", dQ, bf, (B, Hq, N, d), device)
    _check_tensor("dK", dK, bf, (B, Hkv, N, d), device)
    _check_tensor("dV", dV, bf, (B, Hkv, N, d), device)


def attn_status_string(code: int) -> str:
    return load_library().attn_status_string(int(code)).decode()


def attn_bwd_workspace_size(B: int, Hq: int, Hkv: int, N: int, d: int) -> int:
    return int(load_library().attn_bwd_workspace_size(B, Hq, Hkv, N, d))


def attn_last_device_status(stream=None) -> int:
    return int(load_library().attn_last_device_status(_stream(stream)))


def attn_selftest_wait_timeout(limit_ns: int, stream=None) -> int:
    return int(load_library().attn_selftest_wait_timeout(int(limit_ns), _stream(stream)))


def attn_fwd(Q, K, V, scale=None, causal=False, out_dtype=None, O=None, LSE=None, stream=None):
    """O, LSE = softmax(scale Q K^T [+causal]) V and its row log-sum-exp."""
    lib = load_library()
    B, Hq, N, d = Q.shape
    Hkv = K.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    in_dt = {torch.bfloat16: ATTN_BF16, torch.float32: ATTN_F32}.get(Q.dtype)
    if in_dt is None:
        raise TypeError("Q must be bf16 or fp32")
    if out_dtype is None:
        out_dtype = Q.dtype
    out_dt = {torch.bfloat16: ATTN_BF16, torch.float32: ATTN_F32}[out_dtype]
    _check_tensor("Q", Q, Q.dtype, (B, Hq, N, d))
    dev = Q.device
    _check_tensor("K", K, Q.dtype, (B, Hkv, N, d), dev)
    _check_tensor("V", V, Q.dtype, (B, Hkv, N, d), dev)
    if O is None:
        O = torch.empty((B, Hq, N, d), dtype=out_dtype, device=dev)
    if LSE is None:
        LSE = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
    _check_tensor("O", O, out_dtype, (B, Hq, N, d), dev)
    _check_tensor("LSE", LSE, torch.float32, (B, Hq, N), dev)
    with torch.cuda.device(dev):
        rc = lib.attn_fwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), B, Hq, Hkv, N, d,
                          float(scale), int(bool(causal)), in_dt, out_dt, _stream(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd")
    return O, LSE


def attn_fwd_split_workspace_size(B: int, Hq: int, Hkv: int, Nq: int, Nk: int, d: int,
                                  num_splits: int = 0) -> int:
    return int(load_library().attn_fwd_split_workspace_size(B, Hq, Hkv, Nq, Nk, d, num_splits))


def attn_fwd_split(Q, K, V, scale=None, causal=False, num_splits=0, out_dtype=None, O=None, LSE=None,
                   workspace=None, stream=None):
    """O, LSE of attention with Nq = Q.shape[2] queries and Nk = K.shape[2] keys
    (bottom-right causal alignment when they differ), the key range cut into
    num_splits parts (0: chosen by the library) whose partial results are
    merged.  bf16 inputs; O bf16 (default) or fp32."""
    lib = load_library()
    B, Hq, Nq, d = Q.shape
    Hkv, Nk = K.shape[1], K.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    bf = torch.bfloat16
    if out_dtype is None:
        out_dtype = bf
    out_dt = {torch.bfloat16: ATTN_BF16, torch.float32: ATTN_F32}[out_dtype]
    _check_tensor("Q", Q, bf, (B, Hq, Nq, d))
    dev = Q.device
    _check_tensor("K", K, bf, (B, Hkv, Nk, d), dev)
    _check_tensor("V", V, bf, (B, Hkv, Nk, d), dev)
    if O is None:
        O = torch.empty((B, Hq, Nq, d), dtype=out_dtype, device=dev)
    if LSE is None:
        LSE = torch.empty((B, Hq, Nq), dtype=torch.float32, device=dev)
    _check_tensor("O", O, out_dtype, (B, Hq, Nq, d), dev)
    _check_tensor("LSE", LSE, torch.float32, (B, Hq, Nq), dev)
    ws_bytes = attn_fwd_split_workspace_size(B, Hq, Hkv, Nq, Nk, d, num_splits)
    if workspace is None and ws_bytes > 0:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    if workspace is not None:
        _check_workspace(workspace, ws_bytes, dev)
    wptr = _ptr(workspace) if workspace is not None else ctypes.c_void_p(0)
    wbytes = workspace.numel() if workspace is not None else 0
    with torch.cuda.device(dev):
        rc = lib.attn_fwd_split(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), B, Hq, Hkv, Nq, Nk, d,
                                float(scale), int(bool(causal)), out_dt, int(num_splits), wptr, wbytes,
                                _stream(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_split")
    return O, LSE


def _check_mask(block_mask, Hq, N, device):
    T = (N + 127) // 128
    if not isinstance(block_mask, torch.Tensor) or not block_mask.is_cuda or block_mask.dtype != torch.uint8:
        raise TypeError("block_mask must be a uint8 CUDA tensor")
    if block_mask.device != device:
        raise ValueError(f"block_mask is on {block_mask.device}, expected {device}")
    m = block_mask if block_mask.dim() == 3 else block_mask.reshape(1, T, T)
    if tuple(m.shape[1:]) != (T, T) or m.shape[0] not in (1, Hq) or not m.is_contiguous():
        raise ValueError(f"block_mask must be contiguous [1 or {Hq}, {T}, {T}], got {tuple(block_mask.shape)}")
    return m, m.shape[0]


def attn_fwd_masked(Q, K, V, block_mask, scale=None, causal=False, out_dtype=None, O=None, LSE=None,
                    stream=None):
    """Block-sparse forward: block_mask[h, i, j] == 0 removes the 128 x 128 block
    (query tile i, key tile j) of head h (h = 0 for a mask shared by all heads)."""
    lib = load_library()
    B, Hq, N, d = Q.shape
    Hkv = K.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    bf = torch.bfloat16
    out_dtype = bf if out_dtype is None else out_dtype
    out_dt = {torch.bfloat16: ATTN_BF16, torch.float32: ATTN_F32}[out_dtype]
    _check_tensor("Q", Q, bf, (B, Hq, N, d))
    dev = Q.device
    for name, t, H in (("K", K, Hkv), ("V", V, Hkv)):
        _check_tensor(name, t, bf, (B, H, N, d), dev)
    m, mh = _check_mask(block_mask, Hq, N, dev)
    O = torch.empty((B, Hq, N, d), dtype=out_dtype, device=dev) if O is None else O
    LSE = torch.empty((B, Hq, N), dtype=torch.float32, device=dev) if LSE is None else LSE
    _check_tensor("O", O, out_dtype, (B, Hq, N, d), dev)
    _check_tensor("LSE", LSE, torch.float32, (B, Hq, N), dev)
    with torch.cuda.device(dev):
        rc = lib.attn_fwd_masked(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), B, Hq, Hkv, N, d, float(scale),
                                 int(bool(causal)), _ptr(m), mh, out_dt, _stream(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_masked")
    return O, LSE


def attn_fp8_vt_stride(N: int) -> int:
    """Row length of transposed FP8 codes: N rounded up to 16."""
    return int(load_library().attn_fp8_vt_stride(int(N)))


def attn_quantize_fp8(X, transpose=False, codes=None, scales=None, stream=None):
    """Per-128-row-block e4m3 quantization of X [B, H, N, d] (bf16).

    Returns (codes, scales): codes uint8 [B, H, N, d], or with transpose
    [B, H, d, attn_fp8_vt_stride(N)]; scales fp32 [B, H, ceil(N / 128)]."""
    lib = load_library()
    B, H, N, d = X.shape
    _check_tensor("X", X, torch.bfloat16, (B, H, N, d))
    dev = X.device
    T = (N + 127) // 128
    cshape = (B, H, d, attn_fp8_vt_stride(N)) if transpose else (B, H, N, d)
    codes = torch.empty(cshape, dtype=torch.uint8, device=dev) if codes is None else codes
    scales = torch.empty((B, H, T), dtype=torch.float32, device=dev) if scales is None else scales
    _check_tensor("codes", codes, torch.uint8, cshape, dev)
    _check_tensor("scales", scales, torch.float32, (B, H, T), dev)
    with torch.cuda.device(dev):
        rc = lib.attn_quantize_fp8(_ptr(X), _ptr(codes), _ptr(scales), B * H, N, d, int(bool(transpose)),
                                   _stream(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_quantize_fp8")
    return codes, scales


def attn_fwd_fp8(Qc, q_scale, Kc, k_scale, Vtc, v_scale, scale=None, causal=False, out_dtype=None, O=None,
                 LSE=None, stream=None):
    """FP8 forward on block-quantized Q, K and transposed V (see attn_quantize_fp8)."""
    lib = load_library()
    B, Hq, N, d = Qc.shape
    Hkv = Kc.shape[1]
    T = (N + 127) // 128
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out_dtype = torch.bfloat16 if out_dtype is None else out_dtype
    out_dt = {torch.bfloat16: ATTN_BF16, torch.float32: ATTN_F32}[out_dtype]
    u8, f32 = torch.uint8, torch.float32
    _check_tensor("Qc", Qc, u8, (B, Hq, N, d))
    dev = Qc.device
    _check_tensor("Kc", Kc, u8, (B, Hkv, N, d), dev)
    _check_tensor("Vtc", Vtc, u8, (B, Hkv, d, attn_fp8_vt_stride(N)), dev)
    _check_tensor("q_scale", q_scale, f32, (B, Hq, T), dev)
    _check_tensor("k_scale", k_scale, f32, (B, Hkv, T), dev)
    _check_tensor("v_scale", v_scale, f32, (B, Hkv, T), dev)
    O = torch.empty((B, Hq, N, d), dtype=out_dtype, device=dev) if O is None else O
    LSE = torch.empty((B, Hq, N), dtype=f32, device=dev) if LSE is None else LSE
    _check_tensor("O", O, out_dtype, (B, Hq, N, d), dev)
    _check_tensor("LSE", LSE, f32, (B, Hq, N), dev)
    with torch.cuda.device(dev):
        rc = lib.attn_fwd_fp8(_ptr(Qc), _ptr(q_scale), _ptr(Kc), _ptr(k_scale), _ptr(Vtc), _ptr(v_scale),
                              _ptr(O), _ptr(LSE), B, Hq, Hkv, N, d, float(scale), int(bool(causal)), out_dt,
                              _stream(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_fp8")
    return O, LSE


def _bwd_inputs(Q, K, V, O, dO, LSE):
    """Checks the backward's inputs; returns (B, Hq, Hkv, N, d, device)."""
    B, Hq, N, d = Q.shape
    Hkv = K.shape[1]
    bf = torch.bfloat16
    _check_tensor("Q", Q, bf, (B, Hq, N, d))
    dev = Q.device
    for name, t, H in (("K", K, Hkv), ("V", V, Hkv), ("O", O, Hq), ("dO", dO, Hq)):
        _check_tensor(name, t, bf, (B, H, N, d), dev)
    _check_tensor("LSE", LSE, torch.float32, (B, Hq, N), dev)
    return B, Hq, Hkv, N, d, dev


def attn_bwd_masked(Q, K, V, O, dO, LSE, block_mask, scale=None, causal=False, dQ=None, dK=None, dV=None,
                    workspace=None, stream=None):
    """Block-sparse backward with the mask of attn_fwd_masked."""
    lib = load_library()
    B, Hq, Hkv, N, d, dev = _bwd_inputs(Q, K, V, O, dO, LSE)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    m, mh = _check_mask(block_mask, Hq, N, dev)
    dQ = torch.empty_like(Q) if dQ is None else dQ
    dK = torch.empty_like(K) if dK is None else dK
    dV = torch.empty_like(V) if dV is None else dV
    _check_bwd_outputs(dQ, dK, dV, B, Hq, Hkv, N, d, dev)
    ws_bytes = attn_bwd_workspace_size(B, Hq, Hkv, N, d)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    _check_workspace(workspace, ws_bytes, dev)
    with torch.cuda.device(dev):
        rc = lib.attn_bwd_masked(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(LSE), _ptr(dQ), _ptr(dK),
                                 _ptr(dV), B, Hq, Hkv, N, d, float(scale), int(bool(causal)), _ptr(m), mh,
                                 _ptr(workspace), workspace.numel(), _stream(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_bwd_masked")
    return dQ, dK, dV


def attn_bwd(Q, K, V, O, dO, LSE, scale=None, causal=False, dQ=None, dK=None, dV=None,
             workspace=None, stream=None, stage="all"):
    """dQ, dK, dV of O = attention(Q, K, V) given dO and the forward's LSE.

    ``stage`` selects one of the C entry points: "all" (attn_bwd) or one of
    "preprocess", "main", "convert" (run in that order with the same
    workspace to obtain the same result)."""
    lib = load_library()
    B, Hq, Hkv, N, d, dev = _bwd_inputs(Q, K, V, O, dO, LSE)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dQ = torch.empty_like(Q) if dQ is None else dQ
    dK = torch.empty_like(K) if dK is None else dK
    dV = torch.empty_like(V) if dV is None else dV
    _check_bwd_outputs(dQ, dK, dV, B, Hq, Hkv, N, d, dev)
    ws_bytes = attn_bwd_workspace_size(B, Hq, Hkv, N, d)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    _check_workspace(workspace, ws_bytes, dev)
    fname = _BWD_STAGES[stage]
    with torch.cuda.device(dev):
        rc = getattr(lib, fname)(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(LSE), _ptr(dQ),
                                 _ptr(dK), _ptr(dV), B, Hq, Hkv, N, d, float(scale),
                                 int(bool(causal)), ATTN_BF16, _ptr(workspace), workspace.numel(),
                                 _stream(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, fname)
    return dQ, dK, dV


# ---------------------------------------------------------------- no-alloc backward
EXPORTED = EXPORTED + ("attn_bwd_noalloc",)
NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024


def attn_bwd_noalloc(Q, K, V, O, dO, LSE, scale=None, causal=False, dQ=None, dK=None, dV=None,
                     stream=None):
    """attn_bwd with the library's fixed scratch array instead of a workspace.

    For callers that cannot allocate device memory where they run the
    backward.  The C call allocates nothing; problems whose workspace would
    exceed NOALLOC_SCRATCH_BYTES are rejected (ATTN_ERR_UNSUPPORTED).  Calls on
    one device share the scratch array: do not let them overlap on the GPU.
    (Here the outputs are allocated by PyTorch unless given.)"""
    lib = load_library()
    fn = lib.attn_bwd_noalloc
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i32, i32, vp]
    fn.restype = i32
    B, Hq, Hkv, N, d, dev = _bwd_inputs(Q, K, V, O, dO, LSE)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dQ = torch.empty_like(Q) if dQ is None else dQ
    dK = torch.empty_like(K) if dK is None else dK
    dV = torch.empty_like(V) if dV is None else dV
    _check_bwd_outputs(dQ, dK, dV, B, Hq, Hkv, N, d, dev)
    with torch.cuda.device(dev):
        rc = fn(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(LSE), _ptr(dQ), _ptr(dK), _ptr(dV),
                B, Hq, Hkv, N, d, float(scale), int(bool(causal)), ATTN_BF16, _stream(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_bwd_noalloc")
    return dQ, dK, dV
