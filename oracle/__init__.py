"""fp64 CPU oracle for exact softmax attention -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline may import this package.  The CUDA library never imports it, and it
never imports the CUDA library.  The arithmetic lives in ``attn_oracle.cpp``
(plain C++17, fp64); this module compiles it with the host compiler and wraps
it with ctypes over numpy arrays.

Every wrapper takes fp64 numpy arrays in the row-major [B, H, N, d] layout
(d contiguous) and returns fp64 numpy arrays.  See ``attn_oracle.h`` for the
conventions (grouping of query heads, causal alignment, LSE units).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.cpp")
_HDR = os.path.join(_HERE, "attn_oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so next to its source (host compiler, no GPU)."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread",
               "-o", tmp, _SRC]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            dp = ctypes.POINTER(ctypes.c_double)
            fp = ctypes.POINTER(ctypes.c_float)
            lp = ctypes.POINTER(ctypes.c_int64)
            i64, i32, f64 = ctypes.c_int64, ctypes.c_int, ctypes.c_double
            lib.oracle_causal_keep.argtypes = [i64, i64, i64, i64]
            lib.oracle_softmax3.argtypes = [dp, i64, dp]
            lib.oracle_softmax3_f32.argtypes = [fp, i64, fp]
            lib.oracle_online_row.argtypes = [dp, dp, i64, i64, lp, i64, dp, dp, dp, dp]
            lib.oracle_online_softmax_f32.argtypes = [fp, i64, i64, fp]
            shape = [i32, i32, i32, i64, i64, i32, f64, i32]
            lib.oracle_fwd.argtypes = [dp, dp, dp] + shape + [dp, dp, i32]
            lib.oracle_fwd_rows.argtypes = [dp, dp, dp] + shape + [lp, i64, dp, dp, i32]
            lib.oracle_bwd.argtypes = [dp, dp, dp, dp] + shape + [dp, dp, dp, dp, dp, dp, i32]
            lib.oracle_bwd_dq_rows.argtypes = [dp, dp, dp, dp] + shape + [lp, i64, dp, i32]
            lib.oracle_bwd_dkv_rows.argtypes = [dp, dp, dp, dp, dp, dp] + shape + [lp, i64, dp, dp, i32]
            u8p = ctypes.POINTER(ctypes.c_uint8)
            lib.oracle_fwd_masked.argtypes = [dp, dp, dp] + shape + [u8p, i32, i64, dp, dp, i32]
            lib.oracle_bwd_masked.argtypes = [dp, dp, dp, dp] + shape + [u8p, i32, i64, dp, dp, dp, dp, dp, i32]
            _lib = lib
    return _lib


def _d(a):
    a = np.ascontiguousarray(a, dtype=np.float64)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f(a):
    a = np.ascontiguousarray(a, dtype=np.float32)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def _l(a):
    a = np.ascontiguousarray(a, dtype=np.int64)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))


def _check(rc, name):
    if rc != 0:
        raise ValueError(f"{name} rejected its arguments (code {rc})")


def _shapes(Q, K, V=None):
    B, Hq, Nq, d = Q.shape
    B2, Hkv, Nk, d2 = K.shape
    if B2 != B or d2 != d:
        raise ValueError("Q and K disagree on batch or head dim")
    if V is not None and tuple(V.shape) != tuple(K.shape):
        raise ValueError("V must have the shape of K")
    return B, Hq, Hkv, Nq, Nk, d


def causal_keep(i: int, j: int, Nq: int, Nk: int) -> bool:
    return bool(_load().oracle_causal_keep(i, j, Nq, Nk))


def causal_mask(Nq: int, Nk: int) -> np.ndarray:
    """The oracle's keep-mask as an [Nq, Nk] 0/1 array."""
    return np.array([[causal_keep(i, j, Nq, Nk) for j in range(Nk)] for i in range(Nq)],
                    dtype=np.int64)


def softmax3(x) -> np.ndarray:
    x, px = _d(x)
    out, po = _d(np.empty_like(x))
    _check(_load().oracle_softmax3(px, x.size, po), "softmax3")
    return out


def softmax3_f32(x) -> np.ndarray:
    x, px = _f(x)
    out, po = _f(np.empty_like(x))
    _check(_load().oracle_softmax3_f32(px, x.size, po), "softmax3_f32")
    return out


def online_softmax_f32(x, block: int) -> np.ndarray:
    x, px = _f(x)
    out, po = _f(np.empty_like(x))
    _check(_load().oracle_online_softmax_f32(px, x.size, block, po), "online_softmax_f32")
    return out


def online_row(s, v, block_sizes):
    """Online (m, l, O) merge over one score row; returns (O, m_trace, l_trace, O_trace)."""
    s, ps = _d(s)
    v = np.asarray(v, dtype=np.float64)
    if v.ndim == 1:
        v = v[:, None]
    v, pv = _d(v)
    n, dv = v.shape
    bs, pb = _l(block_sizes)
    O, pO = _d(np.zeros(dv))
    mt, pm = _d(np.zeros(len(bs)))
    lt, pl = _d(np.zeros(len(bs)))
    Ot, pOt = _d(np.zeros((len(bs), dv)))
    _check(_load().oracle_online_row(ps, pv, n, dv, pb, len(bs), pO, pm, pl, pOt), "online_row")
    return O, mt, lt, Ot


def fwd(Q, K, V, scale: float, causal: bool, threads: int = 0):
    """Full forward.  Returns (O [B,Hq,Nq,d], LSE [B,Hq,Nq])."""
    B, Hq, Hkv, Nq, Nk, d = _shapes(Q, K, V)
    Q, pq = _d(Q)
    K, pk = _d(K)
    V, pv = _d(V)
    O, po = _d(np.empty((B, Hq, Nq, d)))
    L, pl = _d(np.empty((B, Hq, Nq)))
    _check(_load().oracle_fwd(pq, pk, pv, B, Hq, Hkv, Nq, Nk, d, scale, int(causal),
                              po, pl, threads), "fwd")
    return O, L


def fwd_rows(Q, K, V, scale: float, causal: bool, rows, threads: int = 0):
    """Forward on query rows rows[r] = (b*Hq + h)*Nq + i.  Returns (O [n,d], LSE [n])."""
    B, Hq, Hkv, Nq, Nk, d = _shapes(Q, K, V)
    Q, pq = _d(Q)
    K, pk = _d(K)
    V, pv = _d(V)
    rows, pr = _l(rows)
    O, po = _d(np.empty((len(rows), d)))
    L, pl = _d(np.empty(len(rows)))
    _check(_load().oracle_fwd_rows(pq, pk, pv, B, Hq, Hkv, Nq, Nk, d, scale, int(causal),
                                   pr, len(rows), po, pl, threads), "fwd_rows")
    return O, L


def bwd(Q, K, V, dO, scale: float, causal: bool, threads: int = 0):
    """Full backward.  Returns dict with dQ, dK, dV, O, LSE, D."""
    B, Hq, Hkv, Nq, Nk, d = _shapes(Q, K, V)
    Q, pq = _d(Q)
    K, pk = _d(K)
    V, pv = _d(V)
    dO, pdo = _d(dO)
    dQ, pdq = _d(np.empty((B, Hq, Nq, d)))
    dK, pdk = _d(np.empty((B, Hkv, Nk, d)))
    dV, pdv = _d(np.empty((B, Hkv, Nk, d)))
    O, po = _d(np.empty((B, Hq, Nq, d)))
    L, pl = _d(np.empty((B, Hq, Nq)))
    D, pD = _d(np.empty((B, Hq, Nq)))
    _check(_load().oracle_bwd(pq, pk, pv, pdo, B, Hq, Hkv, Nq, Nk, d, scale, int(causal),
                              pdq, pdk, pdv, po, pl, pD, threads), "bwd")
    return {"dQ": dQ, "dK": dK, "dV": dV, "O": O, "LSE": L, "D": D}


def bwd_dq_rows(Q, K, V, dO, scale: float, causal: bool, rows, threads: int = 0):
    B, Hq, Hkv, Nq, Nk, d = _shapes(Q, K, V)
    Q, pq = _d(Q)
    K, pk = _d(K)
    V, pv = _d(V)
    dO, pdo = _d(dO)
    rows, pr = _l(rows)
    dQ, pdq = _d(np.empty((len(rows), d)))
    _check(_load().oracle_bwd_dq_rows(pq, pk, pv, pdo, B, Hq, Hkv, Nq, Nk, d, scale,
                                      int(causal), pr, len(rows), pdq, threads), "bwd_dq_rows")
    return dQ


def bwd_dkv_rows(Q, K, V, dO, LSE, D, scale: float, causal: bool, kv_rows, threads: int = 0):
    """dK, dV on key rows kv_rows[r] = (b*Hkv + hk)*Nk + j given per-query LSE and D."""
    B, Hq, Hkv, Nq, Nk, d = _shapes(Q, K, V)
    Q, pq = _d(Q)
    K, pk = _d(K)
    V, pv = _d(V)
    dO, pdo = _d(dO)
    LSE, pl = _d(LSE)
    D, pD = _d(D)
    rows, pr = _l(kv_rows)
    dK, pdk = _d(np.empty((len(rows), d)))
    dV, pdv = _d(np.empty((len(rows), d)))
    _check(_load().oracle_bwd_dkv_rows(pq, pk, pv, pdo, pl, pD, B, Hq, Hkv, Nq, Nk, d, scale,
                                       int(causal), pr, len(rows), pdk, pdv, threads),
           "bwd_dkv_rows")
    return dK, dV


def _mask(bmask, Hq, Nq, Nk, bsize):
    m = np.ascontiguousarray(np.asarray(bmask) != 0, dtype=np.uint8)
    nqb, nkb = -(-Nq // bsize), -(-Nk // bsize)
    if m.ndim == 2:
        m = m[None]
    if m.shape[1:] != (nqb, nkb) or m.shape[0] not in (1, Hq):
        raise ValueError(f"block mask must be [1 or Hq, {nqb}, {nkb}], got {m.shape}")
    return m, m.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)), m.shape[0]


def fwd_masked(Q, K, V, scale: float, causal: bool, bmask, bsize: int = 128, threads: int = 0):
    """Block-sparse forward: bmask [Hq or 1, ceil(Nq/bsize), ceil(Nk/bsize)], zero
    entries remove the block's keys.  Returns (O, LSE)."""
    B, Hq, Hkv, Nq, Nk, d = _shapes(Q, K, V)
    m, pm, mh = _mask(bmask, Hq, Nq, Nk, bsize)
    Q, pq = _d(Q)
    K, pk = _d(K)
    V, pv = _d(V)
    O, po = _d(np.empty((B, Hq, Nq, d)))
    L, pl = _d(np.empty((B, Hq, Nq)))
    _check(_load().oracle_fwd_masked(pq, pk, pv, B, Hq, Hkv, Nq, Nk, d, scale, int(causal), pm, mh,
                                     bsize, po, pl, threads), "fwd_masked")
    return O, L


def bwd_masked(Q, K, V, dO, scale: float, causal: bool, bmask, bsize: int = 128, threads: int = 0):
    """Block-sparse backward.  Returns dict with dQ, dK, dV, O, LSE."""
    B, Hq, Hkv, Nq, Nk, d = _shapes(Q, K, V)
    m, pm, mh = _mask(bmask, Hq, Nq, Nk, bsize)
    Q, pq = _d(Q)
    K, pk = _d(K)
    V, pv = _d(V)
    dO, pdo = _d(dO)
    dQ, pdq = _d(np.empty((B, Hq, Nq, d)))
    dK, pdk = _d(np.empty((B, Hkv, Nk, d)))
    dV, pdv = _d(np.empty((B, Hkv, Nk, d)))
    O, po = _d(np.empty((B, Hq, Nq, d)))
    L, pl = _d(np.empty((B, Hq, Nq)))
    _check(_load().oracle_bwd_masked(pq, pk, pv, pdo, B, Hq, Hkv, Nq, Nk, d, scale, int(causal), pm, mh,
                                     bsize, pdq, pdk, pdv, po, pl, threads), "bwd_masked")
    return {"dQ": dQ, "dK": dK, "dV": dV, "O": O, "LSE": L}
