"""ctypes binding of libfa.so: the C-ABI calls of include/fa.h under the same names.

Argument marshalling only: each function checks that it was handed CUDA
tensors of the right dtype and layout, reads their pointers and sizes, and
calls the library on the current (or given) stream.  Every numeric step runs
in the library's kernels; there is no fallback of any kind, and importing the
binding fails loudly when libfa.so has not been built.
"""

from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

_lib = None

FA_OK = 0
FA_ERR_INVALID_ARG = -1
FA_ERR_UNSUPPORTED = -2
FA_ERR_MISALIGNED = -3
FA_ERR_CUDA = -4
FA_ERR_DEVICE_TIMEOUT = -5
FA_ERR_NO_MEMORY = -6

_vp = ctypes.c_void_p
_i = ctypes.c_int
_f = ctypes.c_float
_sz = ctypes.c_size_t

_SIGNATURES = {
    "fa_fwd": ([_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp], _i),
    "fa_bwd_workspace_bytes": ([_i, _i, _i, _i], _sz),
    "fa_bwd": ([_vp] * 9 + [_i, _i, _i, _i, _i, _f, _vp, _sz, _vp], _i),
    "fa_bwd_preprocess": ([_vp] * 5 + [_i, _i, _i, _i, _vp], _i),
    "fa_bwd_dkdv": ([_vp] * 8 + [_i, _i, _i, _i, _i, _f, _vp], _i),
    "fa_bwd_dq": ([_vp] * 7 + [_i, _i, _i, _i, _i, _f, _vp], _i),
    "fa_bwd_dq_preprocess": ([_vp] * 9 + [_i, _i, _i, _i, _i, _f, _vp], _i),
    "fa_fwd_f32": ([_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp], _i),
    "fa_bwd_f32": ([_vp] * 9 + [_i, _i, _i, _i, _i, _f, _vp, _sz, _vp], _i),
    "fa_error_string": ([_i], ctypes.c_char_p),
    "fa_device_status": ([_i], _i),
    "fa_last_device_status": ([], _i),
    "fa_set_wait_timeout_ns": ([ctypes.c_ulonglong], None),
    "fa_selftest_wait_timeout": ([ctypes.c_ulonglong, _vp], _i),
    "fa_bwd_noalloc": ([_vp] * 9 + [_i, _i, _i, _i, _i, _f, _vp], _i),
    "fa_fwd_gqa": ([_vp] * 5 + [_i] * 6 + [_f, _vp], _i),
    "fa_bwd_gqa": ([_vp] * 9 + [_i] * 6 + [_f, _vp, _sz, _vp], _i),
    "fa_fwd_splitkv_workspace_bytes": ([_i] * 7, _sz),
    "fa_fwd_splitkv": ([_vp] * 5 + [_i] * 6 + [_f, _i, _vp, _sz, _vp], _i),
    "fa_fp8_quantize": ([_vp] * 4 + [_i] * 3 + [_vp], _i),
    "fa_fwd_fp8": ([_vp] * 7 + [_i] * 6 + [_f, _vp], _i),
}

NOALLOC_SCRATCH_BYTES = 8 << 20  # FA_NOALLOC_SCRATCH_BYTES in include/fa.h


class FaError(RuntimeError):
    """A non-zero fa_status returned by the library."""

    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {error_string(status)} (status {status})")


def lib_path() -> str:
    return _build.LIB_PATH


def load() -> ctypes.CDLL:
    """The loaded libfa.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        path = _build.LIB_PATH
        if not os.path.exists(path):
            raise ImportError(f"{path} is missing: build it first "
                              "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(path)
        for name, (args, res) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
    return _lib


def error_string(status: int) -> str:
    return load().fa_error_string(int(status)).decode()


def _check(rc: int, what: str) -> None:
    if rc != FA_OK:
        raise FaError(rc, what)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


def _bhnd(q: torch.Tensor):
    if q.dim() != 4:
        raise ValueError("tensors must be [B, H, N, d]")
    return tuple(int(x) for x in q.shape)


def _expect(t: torch.Tensor, name: str, dtype, shape) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


# ----------------------------------------------------------------- BF16 path

def fa_fwd(q, k, v, o, lse, causal: bool, scale: float, stream=None) -> None:
    """O, LSE of exact attention (bf16 q/k/v/o, fp32 lse) into o and lse."""
    B, H, N, d = _bhnd(q)
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o)):
        _expect(t, name, torch.bfloat16, (B, H, N, d))
    _expect(lse, "lse", torch.float32, (B, H, N))
    _check(load().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d,
                         int(bool(causal)), float(scale), _stream(stream)), "fa_fwd")


def _gqa_heads(q, k):
    B, Hq, N, d = _bhnd(q)
    if k.dim() != 4:
        raise ValueError("k must be [B, Hkv, N, d]")
    return B, Hq, int(k.shape[1]), N, d


def fa_fwd_gqa(q, k, v, o, lse, causal: bool, scale: float, stream=None) -> None:
    """Grouped-query attention forward: q, o [B,Hq,N,d]; k, v [B,Hkv,N,d]; Hkv divides Hq."""
    B, Hq, Hkv, N, d = _gqa_heads(q, k)
    for name, t, h in (("q", q, Hq), ("k", k, Hkv), ("v", v, Hkv), ("o", o, Hq)):
        _expect(t, name, torch.bfloat16, (B, h, N, d))
    _expect(lse, "lse", torch.float32, (B, Hq, N))
    _check(load().fa_fwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, N, d,
                             int(bool(causal)), float(scale), _stream(stream)), "fa_fwd_gqa")


# ----------------------------------------------------------------- FP8 forward

def _host_signs(signs, d: int):
    """d signs (+1 / -1) as a C float array (returned as is if it already is
    one of length d); the library validates the values."""
    if isinstance(signs, ctypes.Array) and len(signs) == d:
        return signs
    if isinstance(signs, torch.Tensor):
        vals = signs.detach().to("cpu", torch.float64).reshape(-1).tolist()
    else:
        vals = [float(x) for x in signs]
    if len(vals) != d:
        raise ValueError(f"signs must hold d = {d} entries, got {len(vals)}")
    return (ctypes.c_float * d)(*vals)


def fa_fp8_quantize(x, signs, codes, scales, stream=None) -> None:
    """Rotation by diag(signs) H / sqrt(d) and per-128-row-tile E4M3 codes:
    x bf16 [B,H,N,d] -> codes uint8 [B,H,N,d], scales float32 [B,H,ceil(N/128)]."""
    B, H, N, d = _bhnd(x)
    _expect(x, "x", torch.bfloat16, (B, H, N, d))
    _expect(codes, "codes", torch.uint8, (B, H, N, d))
    _expect(scales, "scales", torch.float32, (B, H, (N + 127) // 128))
    arr = _host_signs(signs, d)
    _check(load().fa_fp8_quantize(_ptr(x), ctypes.cast(arr, _vp), _ptr(codes), _ptr(scales),
                                  B * H, N, d, _stream(stream)), "fa_fp8_quantize")


def fa_fwd_fp8(q8, q_scale, k8, k_scale, v, o, lse, causal: bool, scale: float,
               stream=None) -> None:
    """Forward from E4M3 codes of the rotated Q [B,Hq,N,d] and K [B,Hkv,N,d] and
    their tile scales; v bf16 [B,Hkv,N,d]; o bf16 [B,Hq,N,d]; lse float32."""
    B, Hq, Hkv, N, d = _gqa_heads(q8, k8)
    nt = (N + 127) // 128
    _expect(q8, "q8", torch.uint8, (B, Hq, N, d))
    _expect(k8, "k8", torch.uint8, (B, Hkv, N, d))
    _expect(q_scale, "q_scale", torch.float32, (B, Hq, nt))
    _expect(k_scale, "k_scale", torch.float32, (B, Hkv, nt))
    _expect(v, "v", torch.bfloat16, (B, Hkv, N, d))
    _expect(o, "o", torch.bfloat16, (B, Hq, N, d))
    _expect(lse, "lse", torch.float32, (B, Hq, N))
    _check(load().fa_fwd_fp8(_ptr(q8), _ptr(q_scale), _ptr(k8), _ptr(k_scale), _ptr(v), _ptr(o),
                             _ptr(lse), B, Hq, Hkv, N, d, int(bool(causal)), float(scale),
                             _stream(stream)), "fa_fwd_fp8")


def fa_bwd_gqa(q, k, v, o, do, lse, dq, dk, dv, causal: bool, scale: float, workspace=None,
               stream=None) -> None:
    """Grouped-query attention backward: dq [B,Hq,N,d], dk and dv [B,Hkv,N,d] (fp32)."""
    B, Hq, Hkv, N, d = _gqa_heads(q, k)
    for name, t, h in (("q", q, Hq), ("k", k, Hkv), ("v", v, Hkv), ("o", o, Hq), ("do", do, Hq)):
        _expect(t, name, torch.bfloat16, (B, h, N, d))
    _expect(lse, "lse", torch.float32, (B, Hq, N))
    for name, t, h in (("dq", dq, Hq), ("dk", dk, Hkv), ("dv", dv, Hkv)):
        _expect(t, name, torch.float32, (B, h, N, d))
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().fa_bwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq),
                             _ptr(dk), _ptr(dv), B, Hq, Hkv, N, d, int(bool(causal)),
                             float(scale), _ptr(workspace), ws_bytes, _stream(stream)),
           "fa_bwd_gqa")


def fa_fwd_splitkv_workspace_bytes(B: int, Hq: int, Hkv: int, Nq: int, Nk: int, d: int,
                                   n_splits: int = 0) -> int:
    return int(load().fa_fwd_splitkv_workspace_bytes(int(B), int(Hq), int(Hkv), int(Nq), int(Nk),
                                                     int(d), int(n_splits)))


def fa_fwd_splitkv(q, k, v, o, lse, scale: float, n_splits: int = 0, workspace=None,
                   stream=None) -> None:
    """Decode forward: q, o [B,Hq,Nq,d]; k, v [B,Hkv,Nk,d] (bf16); no mask; the keys
    are cut into n_splits chunks (<= 0: the library's choice) merged at the end."""
    B, Hq, Nq, d = _bhnd(q)
    if k.dim() != 4:
        raise ValueError("k must be [B, Hkv, Nk, d]")
    Hkv, Nk = int(k.shape[1]), int(k.shape[2])
    for name, t, shape in (("q", q, (B, Hq, Nq, d)), ("k", k, (B, Hkv, Nk, d)),
                           ("v", v, (B, Hkv, Nk, d)), ("o", o, (B, Hq, Nq, d))):
        _expect(t, name, torch.bfloat16, shape)
    _expect(lse, "lse", torch.float32, (B, Hq, Nq))
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().fa_fwd_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Nq,
                                 Nk, d, float(scale), int(n_splits), _ptr(workspace), ws_bytes,
                                 _stream(stream)), "fa_fwd_splitkv")


def fa_bwd_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(load().fa_bwd_workspace_bytes(int(B), int(H), int(N), int(d)))


def fa_bwd(q, k, v, o, do, lse, dq, dk, dv, causal: bool, scale: float, workspace=None,
           stream=None) -> None:
    """dQ, dK, dV (fp32) of exact attention; workspace None lets the library allocate."""
    B, H, N, d = _bhnd(q)
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("do", do)):
        _expect(t, name, torch.bfloat16, (B, H, N, d))
    _expect(lse, "lse", torch.float32, (B, H, N))
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _expect(t, name, torch.float32, (B, H, N, d))
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq),
                         _ptr(dk), _ptr(dv), B, H, N, d, int(bool(causal)), float(scale),
                         _ptr(workspace), ws_bytes, _stream(stream)), "fa_bwd")


def fa_bwd_preprocess(o, do, lse, delta_ws, lse2_ws, stream=None) -> None:
    """D = rowsum(dO o O) and LSE*log2(e) into padded [B*H, roundup(N,128)] vectors."""
    B, H, N, d = _bhnd(o)
    n_pad = (N + 127) // 128 * 128
    _expect(o, "o", torch.bfloat16, (B, H, N, d))
    _expect(do, "do", torch.bfloat16, (B, H, N, d))
    _expect(lse, "lse", torch.float32, (B, H, N))
    _expect(delta_ws, "delta_ws", torch.float32, (B * H, n_pad))
    _expect(lse2_ws, "lse2_ws", torch.float32, (B * H, n_pad))
    _check(load().fa_bwd_preprocess(_ptr(o), _ptr(do), _ptr(lse), _ptr(delta_ws), _ptr(lse2_ws),
                                    B, H, N, d, _stream(stream)), "fa_bwd_preprocess")


def _bwd_step_inputs(q, k, v, do, delta_ws, lse2_ws):
    B, H, N, d = _bhnd(q)
    n_pad = (N + 127) // 128 * 128
    for name, t in (("q", q), ("k", k), ("v", v), ("do", do)):
        _expect(t, name, torch.bfloat16, (B, H, N, d))
    _expect(delta_ws, "delta_ws", torch.float32, (B * H, n_pad))
    _expect(lse2_ws, "lse2_ws", torch.float32, (B * H, n_pad))
    return B, H, N, d


def fa_bwd_dkdv(q, k, v, do, delta_ws, lse2_ws, dk, dv, causal: bool, scale: float,
                stream=None) -> None:
    """dK and dV, after fa_bwd_preprocess or fa_bwd_dq_preprocess."""
    B, H, N, d = _bwd_step_inputs(q, k, v, do, delta_ws, lse2_ws)
    for name, t in (("dk", dk), ("dv", dv)):
        _expect(t, name, torch.float32, (B, H, N, d))
    _check(load().fa_bwd_dkdv(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(delta_ws), _ptr(lse2_ws),
                              _ptr(dk), _ptr(dv), B, H, N, d, int(bool(causal)), float(scale),
                              _stream(stream)), "fa_bwd_dkdv")


def fa_bwd_dq(q, k, v, do, delta_ws, lse2_ws, dq, causal: bool, scale: float,
              stream=None) -> None:
    """dQ, after fa_bwd_preprocess."""
    B, H, N, d = _bwd_step_inputs(q, k, v, do, delta_ws, lse2_ws)
    _expect(dq, "dq", torch.float32, (B, H, N, d))
    _check(load().fa_bwd_dq(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(delta_ws), _ptr(lse2_ws),
                            _ptr(dq), B, H, N, d, int(bool(causal)), float(scale),
                            _stream(stream)), "fa_bwd_dq")


def fa_bwd_dq_preprocess(q, k, v, o, do, lse, delta_ws, lse2_ws, dq, causal: bool,
                         scale: float, stream=None) -> None:
    """dQ with the first backward step fused: also writes delta_ws and lse2_ws
    (as fa_bwd_preprocess does) for fa_bwd_dkdv, which runs after it."""
    B, H, N, d = _bwd_step_inputs(q, k, v, do, delta_ws, lse2_ws)
    _expect(o, "o", torch.bfloat16, (B, H, N, d))
    _expect(lse, "lse", torch.float32, (B, H, N))
    _expect(dq, "dq", torch.float32, (B, H, N, d))
    _check(load().fa_bwd_dq_preprocess(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse),
                                       _ptr(delta_ws), _ptr(lse2_ws), _ptr(dq), B, H, N, d,
                                       int(bool(causal)), float(scale), _stream(stream)),
           "fa_bwd_dq_preprocess")


def fa_bwd_noalloc(q, k, v, o, do, lse, dq, dk, dv, causal: bool, scale: float,
                   stream=None) -> None:
    """fa_bwd without a workspace and without any device allocation.

    For callers that may not allocate device memory at call time: the D / LSE2
    scratch is an array of NOALLOC_SCRATCH_BYTES built into the library (one
    per GPU, kept until the process exits).  Raises FaError (FA_ERR_NO_MEMORY)
    when the workload needs more.  The first call on a device should come
    before any stream capture; calls that overlap on the GPU race on the
    shared array.
    """
    B, H, N, d = _bhnd(q)
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("do", do)):
        _expect(t, name, torch.bfloat16, (B, H, N, d))
    _expect(lse, "lse", torch.float32, (B, H, N))
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _expect(t, name, torch.float32, (B, H, N, d))
    _check(load().fa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse),
                                 _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, d, int(bool(causal)),
                                 float(scale), _stream(stream)), "fa_bwd_noalloc")


# ----------------------------------------------------------------- FP32 path

def fa_fwd_f32(q, k, v, o, lse, causal: bool, scale: float, stream=None) -> None:
    B, H, N, d = _bhnd(q)
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o)):
        _expect(t, name, torch.float32, (B, H, N, d))
    _expect(lse, "lse", torch.float32, (B, H, N))
    _check(load().fa_fwd_f32(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d,
                             int(bool(causal)), float(scale), _stream(stream)), "fa_fwd_f32")


def fa_bwd_f32(q, k, v, o, do, lse, dq, dk, dv, causal: bool, scale: float, workspace=None,
               stream=None) -> None:
    B, H, N, d = _bhnd(q)
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("do", do), ("dq", dq), ("dk", dk),
                    ("dv", dv)):
        _expect(t, name, torch.float32, (B, H, N, d))
    _expect(lse, "lse", torch.float32, (B, H, N))
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().fa_bwd_f32(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq),
                             _ptr(dk), _ptr(dv), B, H, N, d, int(bool(causal)), float(scale),
                             _ptr(workspace), ws_bytes, _stream(stream)), "fa_bwd_f32")


# ----------------------------------------------------------------- status

def fa_device_status(clear: bool = False) -> int:
    return int(load().fa_device_status(int(bool(clear))))


def fa_last_device_status() -> int:
    return int(load().fa_last_device_status())


def fa_set_wait_timeout_ns(ns: int) -> None:
    load().fa_set_wait_timeout_ns(int(ns))


def fa_selftest_wait_timeout(timeout_ns: int, stream=None) -> int:
    return int(load().fa_selftest_wait_timeout(int(timeout_ns), _stream(stream)))
