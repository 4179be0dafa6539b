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
        lib.oracle_round_bf16_array.argtypes = [_dp, _i64, _dp]
        lib.oracle_round_bf16.argtypes = [ctypes.c_double]
        lib.oracle_round_bf16.restype = ctypes.c_double
        for f in (lib.oracle_fwd, lib.oracle_fwd_rows, lib.oracle_probs, lib.oracle_bwd,
                  lib.oracle_num_threads, lib.oracle_round_bf16_array):
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


def stored_output(o, o_storage: str = "bf16") -> np.ndarray:
    """O as a backward is handed it when the forward stores it in o_storage:
    "bf16" (each value rounded as round_bf16 rounds it), "f32" or "exact".
    attention_bwd forms D from exactly these values, so a backward given
    them as its O input is compared with attention_bwd on equal inputs."""
    if o_storage not in _O_STORAGE:
        raise ValueError(f"o_storage must be one of {sorted(_O_STORAGE)}")
    o = _f64(o)
    if o_storage == "exact":
        return o.copy()
    if o_storage == "f32":
        return o.astype(np.float32).astype(np.float64)
    out = np.empty_like(o)
    _check(_load().oracle_round_bf16_array(_ptr(o), o.size, _ptr(out)),
           "oracle_round_bf16_array")
    return out


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


# ---------------------------------------------------------------- FP8 (E4M3) with incoherent processing
#
# "FlashAttention scaling, multi-GPU training and weight quantization"
# (section 1, FlashAttention-3, FP8 low-precision support) names two devices
# that keep FP8 attention accurate: block quantisation, where each small tile
# gets a scale of its own, and incoherent processing, where Q and K are
# multiplied by a random orthogonal matrix before quantisation so that outlier
# channels are spread over all channels.  The pages fix neither the matrix,
# the tile, the scale rule nor which operands go to FP8; the readings taken
# here: the matrix is a Hadamard transform with random signs (orthogonal, and
# applied in O(d log d)); a tile is 128 rows of one head, mapped onto the
# E4M3 range by the factor 448 / amax (448 the largest finite E4M3 value) and
# dequantised by amax / 448; only Q and K are quantised, and P V stays BF16.
# The kernels must decide every E4M3 code exactly as done here, so the
# rotation and the scaling are carried out in float32 in the order stated
# below; everything after the codes is FP64.

E4M3_MAX = 448.0


def round_e4m3(x) -> np.ndarray:
    """Nearest E4M3 value (1 sign, 4 exponent bits with bias 7, 3 mantissa
    bits, no infinities; largest finite 448, subnormals k * 2^-9), ties to
    even, magnitudes beyond the largest finite value saturated to it."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, fe = np.frexp(a)                 # a = f 2^fe with f in [0.5, 1): exponent fe - 1
    e = np.maximum(fe.astype(np.float64) - 1.0, -6.0)  # below 2^-6 the spacing stays 2^-9
    step = np.exp2(e - 3.0)             # 3 mantissa bits
    q = np.round(a / step) * step       # exact: step is a power of two; round() is half-even
    q = np.minimum(q, E4M3_MAX)
    return np.copysign(q, x)


def fwht_f32(x) -> np.ndarray:
    """Unnormalised Walsh-Hadamard transform along the last axis (a power of
    two), in float32, butterfly stages h = 1, 2, 4, ...: at stage h the pair
    (y[i], y[i + h]) of each block of 2h becomes (y[i] + y[i + h], y[i] - y[i + h]).
    Each output is formed by the same float32 additions in the same order on
    every platform, so a quantised code decided from it is reproducible."""
    y = np.array(x, dtype=np.float32, copy=True)
    d = y.shape[-1]
    lead = y.shape[:-1]
    h = 1
    while h < d:
        y = y.reshape(lead + (d // (2 * h), 2, h))
        a = y[..., 0, :]
        b = y[..., 1, :]
        y = np.stack([a + b, a - b], axis=-2).reshape(lead + (d,))
        h *= 2
    return y


def rotate_f32(x, signs) -> np.ndarray:
    """x R with R = diag(signs) H / sqrt(d) (H the Sylvester Hadamard matrix,
    signs +-1), evaluated as the kernels evaluate it: the signs first, then the
    transform, then one multiplication by the float32 value of 1/sqrt(d).
    R is orthogonal, so (Q R)(K R)^T = Q K^T."""
    x = np.asarray(x, dtype=np.float32)
    s = np.asarray(signs, dtype=np.float32)
    inv = np.float32(1.0 / np.sqrt(x.shape[-1]))
    return fwht_f32(x * s) * inv


def quantize_e4m3_tiles(x, tile: int = 128):
    """Per-tile E4M3 quantisation of x [B,H,N,d] (float32).  For every head and
    block of `tile` rows with largest magnitude amax > 0: the code of x is
    round_e4m3(float32(x * m)) with the float32 factor m = 448 / amax, and the
    tile's dequantisation scale is the float32 value amax / 448 (an all-zero
    tile has codes 0 and scale 1).  Returns the code values (float64, exactly
    representable) and the scales [B,H,ceil(N/tile)]."""
    x = np.asarray(x, dtype=np.float32)
    B, H, N, d = x.shape
    nt = (N + tile - 1) // tile
    scales = np.empty((B, H, nt), dtype=np.float32)
    codes = np.empty(x.shape, dtype=np.float64)
    top = np.float32(E4M3_MAX)
    for t in range(nt):
        blk = x[:, :, t * tile:(t + 1) * tile, :]
        amax = np.abs(blk).max(axis=(2, 3)).astype(np.float32)
        nz = amax > 0
        safe = np.where(nz, amax, np.float32(1.0)).astype(np.float32)
        scales[:, :, t] = np.where(nz, safe / top, np.float32(1.0))
        m = np.where(nz, top / safe, np.float32(0.0)).astype(np.float32)
        q = (blk * m[:, :, None, None]).astype(np.float32)
        codes[:, :, t * tile:(t + 1) * tile, :] = round_e4m3(q)
    return codes, scales


def attention_fwd_fp8(q, k, v, signs, causal: bool, scale: float, Hkv=None):
    """The FP8 forward's definition: Q and K rotated by R (incoherent
    processing) and quantised to E4M3 with per-tile scales; O and LSE are
    exact attention (FP64) on the dequantised rotated Q, K and on V as given.
    Returns (O, LSE, (q codes, q scales), (k codes, k scales))."""
    qr = rotate_f32(q, signs)
    kr = rotate_f32(k, signs)
    qc, qs = quantize_e4m3_tiles(qr)
    kc, ks = quantize_e4m3_tiles(kr)
    qd = qc * np.repeat(qs.astype(np.float64), 128, axis=2)[:, :, :qc.shape[2], None]
    kd = kc * np.repeat(ks.astype(np.float64), 128, axis=2)[:, :, :kc.shape[2], None]
    if Hkv is not None and Hkv != np.asarray(q).shape[1]:
        o, lse = attention_fwd_gqa(qd, kd, v, causal, scale)
    else:
        o, lse = attention_fwd(qd, kd, v, causal, scale)
    return o, lse, (qc, qs), (kc, ks)
