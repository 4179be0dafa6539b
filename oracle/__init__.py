"""FP64 CPU oracle for exact attention (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  It computes the plain
definition of attention and its gradient (see ``fa_oracle.c``) and shares no
code with the CUDA path.

``build()`` compiles ``fa_oracle.c`` with gcc (OpenMP) into
``liboracle.so`` next to this file; every function here converts its inputs
to float64 exactly (bf16 and fp32 values are all representable) and returns
float64 numpy arrays.
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int64)
_i64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile the oracle if the shared library is missing or older than its source."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-Wall",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        lib.oracle_fwd.argtypes = [_dp, _dp, _dp, _i64, _i64, _i64, _i64, _i64, ctypes.c_int,
                                   ctypes.c_double, _dp, _dp]
        lib.oracle_fwd_rows.argtypes = [_dp, _dp, _dp, _i64, _i64, _i64, _i64, ctypes.c_int,
                                        ctypes.c_double, _ip, _ip, _i64, _dp, _dp]
        lib.oracle_probs.argtypes = [_dp, _dp, _i64, _i64, ctypes.c_int, ctypes.c_double, _dp]
        lib.oracle_bwd.argtypes = [_dp, _dp, _dp, _dp, _i64, _i64, _i64, _i64, ctypes.c_int,
                                   ctypes.c_double, ctypes.c_int, _ip, _i64, _dp, _dp, _dp, _dp]
        lib.oracle_round_bf16.argtypes = [ctypes.c_double]
        lib.oracle_round_bf16.restype = ctypes.c_double
        for f in (lib.oracle_fwd, lib.oracle_fwd_rows, lib.oracle_probs, lib.oracle_bwd,
                  lib.oracle_num_threads):
            f.restype = ctypes.c_int
        _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_dp)


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise RuntimeError(f"{what} failed with status {rc}")


def num_threads() -> int:
    """OpenMP threads the oracle uses (honours OMP_NUM_THREADS)."""
    return int(_load().oracle_num_threads())


def attention_fwd(q, k, v, causal: bool, scale: float):
    """O [B,H,N,d] and LSE [B,H,N] (natural log) for every head.

    k and v may hold a different number of keys than q holds queries (tests
    attend to one block of keys at a time); causal keeps key j for query i
    iff j <= i.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, d = q.shape
    Nk = k.shape[2]
    if k.shape != (B, H, Nk, d) or v.shape != k.shape:
        raise ValueError("q [B,H,N,d], k and v [B,H,Nk,d] expected")
    o = np.empty_like(q)
    lse = np.empty((B, H, N), dtype=np.float64)
    _check(_load().oracle_fwd(_ptr(q), _ptr(k), _ptr(v), B, H, N, Nk, d, int(causal),
                              float(scale), _ptr(o), _ptr(lse)), "oracle_fwd")
    return o, lse


def attention_fwd_rows(q, k, v, causal: bool, scale: float, heads, rows):
    """O rows [n, d] and LSE [n] for samples (heads[s], rows[s]); head = b*H + h."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, d = q.shape
    heads = np.ascontiguousarray(heads, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    n = heads.size
    if rows.size != n:
        raise ValueError("heads and rows must have the same length")
    o = np.empty((n, d), dtype=np.float64)
    lse = np.empty(n, dtype=np.float64)
    _check(_load().oracle_fwd_rows(_ptr(q), _ptr(k), _ptr(v), B, H, N, d, int(causal),
                                   float(scale), heads.ctypes.data_as(_ip),
                                   rows.ctypes.data_as(_ip), n, _ptr(o), _ptr(lse)),
           "oracle_fwd_rows")
    return o, lse


def attention_probs(q, k, causal: bool, scale: float) -> np.ndarray:
    """P [N, N] for one head (q, k of shape [N, d])."""
    q, k = _f64(q), _f64(k)
    N, d = q.shape
    p = np.empty((N, N), dtype=np.float64)
    _check(_load().oracle_probs(_ptr(q), _ptr(k), N, d, int(causal), float(scale), _ptr(p)),
           "oracle_probs")
    return p


_O_STORAGE = {"exact": 0, "bf16": 1, "f32": 2}


def round_bf16(x: float) -> float:
    """x rounded to the nearest bfloat16 value, ties to even (normal range)."""
    return float(_load().oracle_round_bf16(float(x)))


def attention_bwd(q, k, v, do, causal: bool, scale: float, heads=None, o_storage="exact"):
    """dQ, dK, dV [n, N, d] and D [n, N] for the listed heads (all when None).

    o_storage names the precision the output O is stored in before the
    backward forms D = rowsum(dO o O): "exact" (FP64, the true gradient of the
    exact function), "bf16" or "f32" (O rounded to the storage type the
    backward is handed).
    """
    if o_storage not in _O_STORAGE:
        raise ValueError(f"o_storage must be one of {sorted(_O_STORAGE)}")
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, H, N, d = q.shape
    if heads is None:
        n = B * H
        hp = None
    else:
        heads = np.ascontiguousarray(heads, dtype=np.int64)
        n = heads.size
        hp = heads.ctypes.data_as(_ip)
    dq = np.empty((n, N, d), dtype=np.float64)
    dk = np.empty_like(dq)
    dv = np.empty_like(dq)
    dvec = np.empty((n, N), dtype=np.float64)
    _check(_load().oracle_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(do), B, H, N, d, int(causal),
                              float(scale), _O_STORAGE[o_storage], hp, n, _ptr(dq), _ptr(dk),
                              _ptr(dv), _ptr(dvec)),
           "oracle_bwd")
    return dq, dk, dv, dvec


def _group_size(hq: int, hkv: int) -> int:
    if hkv < 1 or hq % hkv:
        raise ValueError("the number of query heads must be a multiple of the K/V heads")
    return hq // hkv


def attention_fwd_gqa(q, k, v, causal: bool, scale: float):
    """Grouped-query attention: O [B,Hq,N,d] and LSE [B,Hq,N].

    q is [B,Hq,N,d]; k and v are [B,Hkv,N,d] with Hq = g*Hkv, and query head
    h attends with K/V head h // g (the multi-query and grouped-query variants
    of "FlashAttention-2"; Hkv = 1 is multi-query).  By definition this is
    standard attention per query head, i.e. the MHA definition applied to K
    and V repeated g times along the head axis.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    g = _group_size(q.shape[1], k.shape[1])
    return attention_fwd(q, np.repeat(k, g, axis=1), np.repeat(v, g, axis=1), causal, scale)


def attention_bwd_gqa(q, k, v, do, causal: bool, scale: float, o_storage="exact"):
    """dQ [B,Hq,N,d], dK and dV [B,Hkv,N,d], D [B,Hq,N]: the gradient of
    attention_fwd_gqa.  Repeating K/V along the head axis is linear and its
    transpose sums over the group, so dK (dV) of K/V head j is the sum of the
    MHA dK (dV) of the g query heads that read it.
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    g = _group_size(Hq, Hkv)
    dq, dk, dv, dvec = attention_bwd(q, np.repeat(k, g, axis=1), np.repeat(v, g, axis=1), do,
                                     causal, scale, o_storage=o_storage)
    dk = dk.reshape(B, Hkv, g, N, d).sum(axis=2)
    dv = dv.reshape(B, Hkv, g, N, d).sum(axis=2)
    return dq.reshape(B, Hq, N, d), dk, dv, dvec.reshape(B, Hq, N)
