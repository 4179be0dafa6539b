"""The C-ABI library builds, loads and exports what include/fa.h declares;
host-side argument checks reject bad calls before anything is launched.
None of these calls reaches a kernel, so no GPU is needed."""

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def fa():
    from exact_io_aware_18_gb300 import build
    build.build()
    import exact_io_aware_18_gb300 as pkg
    pkg.load()
    return pkg


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(fa_[a-z0-9_]+)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("fa_fwd", "fa_bwd", "fa_fwd_f32", "fa_bwd_f32", "fa_bwd_workspace_bytes",
                 "fa_error_string", "fa_device_status", "fa_bwd_preprocess", "fa_bwd_dkdv",
                 "fa_bwd_dq", "fa_fwd_gqa", "fa_bwd_gqa", "fa_fp8_quantize", "fa_fwd_fp8",
                 "fa_last_device_status", "fa_bwd_dq_preprocess"):
        assert must in names


def test_library_exports_every_declared_symbol(fa):
    lib = ctypes.CDLL(fa.lib_path())
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", fa.lib_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\s[TW]\s+(fa_[a-z0-9_]+)$", out, flags=re.M))
    assert set(declared_functions()) <= exported


def test_error_strings(fa):
    for status in range(-6, 1):
        assert fa.error_string(status)
    assert fa.error_string(-99) == "unknown status"


def test_workspace_is_linear_in_n(fa):
    # The page on GPU SRAM and tiling notes that at N = 32000 the N x N score
    # matrix alone is about 2 GB per head in 16-bit; the backward's workspace
    # must stay O(N) (two FP32 vectors per head).
    n = 32000
    ws = fa.fa_bwd_workspace_bytes(1, 1, n, 128)
    assert ws == 2 * 4 * ((n + 127) // 128 * 128)
    assert ws < n * n * 2 / 1000
    assert fa.fa_bwd_workspace_bytes(8, 16, 2048, 128) == 2 * 4 * 8 * 16 * 2048
    assert fa.fa_bwd_workspace_bytes(0, 1, 1, 64) == 0


def _call_fwd(lib, ptrs, B=1, H=1, N=128, d=64, causal=0, scale=0.125):
    return lib.fa_fwd(*ptrs, B, H, N, d, causal, scale, None)


def test_argument_checks_before_launch(fa):
    lib = fa.load()
    good = [0x10000 * (i + 1) for i in range(5)]  # aligned fake pointers: never dereferenced
    assert _call_fwd(lib, [0] + good[1:]) == fa.FA_ERR_INVALID_ARG
    assert _call_fwd(lib, [good[0] + 8] + good[1:]) == fa.FA_ERR_MISALIGNED
    assert _call_fwd(lib, good, d=96) == fa.FA_ERR_UNSUPPORTED
    assert _call_fwd(lib, good, d=256) == fa.FA_ERR_UNSUPPORTED
    assert _call_fwd(lib, good, N=0) == fa.FA_ERR_INVALID_ARG
    assert _call_fwd(lib, good, B=-1) == fa.FA_ERR_INVALID_ARG
    assert _call_fwd(lib, good, scale=0.0) == fa.FA_ERR_INVALID_ARG
    assert _call_fwd(lib, good, scale=float("nan")) == fa.FA_ERR_INVALID_ARG
    assert _call_fwd(lib, good, scale=-1.0) == fa.FA_ERR_INVALID_ARG
    assert _call_fwd(lib, good, B=70000) == fa.FA_ERR_UNSUPPORTED
    f32 = lib.fa_fwd_f32(0, *good[1:], 1, 1, 16, 64, 0, 0.125, None)
    assert f32 == fa.FA_ERR_INVALID_ARG
    bwd = lib.fa_bwd(*([0x10000] * 9), 1, 1, 16, 80, 0, 0.125, None, 0, None)
    assert bwd == fa.FA_ERR_UNSUPPORTED
    bwd = lib.fa_bwd(*([0x10000] * 8 + [0x10004]), 1, 1, 16, 64, 0, 0.125, None, 0, None)
    assert bwd == fa.FA_ERR_MISALIGNED
    bwd = lib.fa_bwd(*([0x10000] * 9), 1, 1, 16, 64, 0, 0.125, 0x20000, 16, None)
    assert bwd == fa.FA_ERR_NO_MEMORY
    pre = lib.fa_bwd_preprocess(*([0x10000] * 4 + [0]), 1, 1, 16, 64, None)
    assert pre == fa.FA_ERR_INVALID_ARG
    dq = lib.fa_bwd_dq(*([0x10000] * 7), 1, 1, 16, 64, 1, 0.0, None)
    assert dq == fa.FA_ERR_INVALID_ARG
    dq = lib.fa_bwd_dq(*([0x10000] * 6 + [0x10008]), 1, 1, 16, 64, 1, 0.125, None)
    assert dq == fa.FA_ERR_MISALIGNED
    # the fused dQ step needs O and LSE: a null one is an argument error
    for null_at in (3, 5):
        ptrs = [0x10000] * 9
        ptrs[null_at] = 0
        fused = lib.fa_bwd_dq_preprocess(*ptrs, 1, 1, 16, 64, 1, 0.125, None)
        assert fused == fa.FA_ERR_INVALID_ARG
    fused = lib.fa_bwd_dq_preprocess(*([0x10000] * 3 + [0x10004] + [0x10000] * 5), 1, 1, 16, 64,
                                     1, 0.125, None)
    assert fused == fa.FA_ERR_MISALIGNED


def test_binding_rejects_cpu_tensors(fa):
    import torch
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    lse = torch.zeros(1, 1, 8)
    with pytest.raises(ValueError):
        fa.fa_fwd(q, q, q, q, lse, False, 0.125)


def test_gqa_head_counts_are_checked_before_launch(fa):
    lib = fa.load()
    p = [0x10000] * 5
    # Hkv must divide Hq and lie in [1, Hq]
    for hq, hkv in ((4, 3), (2, 4), (4, 0), (4, -1)):
        assert lib.fa_fwd_gqa(*p, 1, hq, hkv, 16, 64, 1, 0.125, None) == fa.FA_ERR_INVALID_ARG
        assert lib.fa_bwd_gqa(*([0x10000] * 9), 1, hq, hkv, 16, 64, 1, 0.125, None, 0,
                              None) == fa.FA_ERR_INVALID_ARG
    # the other checks still come first: misaligned pointer, bad head dimension
    assert lib.fa_fwd_gqa(*p[:4], 0x10004, 1, 4, 2, 16, 64, 1, 0.125,
                          None) == fa.FA_ERR_MISALIGNED
    assert lib.fa_fwd_gqa(*p, 1, 4, 2, 16, 96, 1, 0.125, None) == fa.FA_ERR_UNSUPPORTED


def test_splitkv_argument_checks_before_launch(fa):
    lib = fa.load()
    p = [0x10000] * 5
    ok = [1, 4, 2, 1, 4096, 128, 0.125, 2]      # B, Hq, Hkv, Nq, Nk, d, scale, n_splits
    def call(args, ws=None, nbytes=0):
        return lib.fa_fwd_splitkv(*p, *args, ws, nbytes, None)
    assert call([1, 4, 3, 1, 4096, 128, 0.125, 2]) == fa.FA_ERR_INVALID_ARG   # 3 does not divide 4
    assert call([1, 4, 2, 0, 4096, 128, 0.125, 2]) == fa.FA_ERR_INVALID_ARG   # Nq = 0
    assert call([1, 4, 2, 1, 0, 128, 0.125, 2]) == fa.FA_ERR_INVALID_ARG      # Nk = 0
    assert call([1, 4, 2, 1, 4096, 96, 0.125, 2]) == fa.FA_ERR_UNSUPPORTED    # d = 96
    assert call(ok, ws=0x10004, nbytes=1 << 30) == fa.FA_ERR_MISALIGNED
    need = lib.fa_fwd_splitkv_workspace_bytes(1, 4, 2, 1, 4096, 128, 2)
    assert call(ok, ws=0x10000, nbytes=need - 16) == fa.FA_ERR_NO_MEMORY


def test_splitkv_workspace_follows_the_split_plan(fa):
    lib = fa.load()
    # 4096 keys = 32 key tiles; 5 requested -> chunks of 7 tiles -> 5 splits;
    # 40 requested -> one tile per split, 32 splits; per split and query row:
    # d FP32 outputs + 1 FP32 LSE
    per = 1 * 4 * 3 * (128 + 1) * 4
    assert lib.fa_fwd_splitkv_workspace_bytes(1, 4, 2, 3, 4096, 128, 5) == 5 * per
    assert lib.fa_fwd_splitkv_workspace_bytes(1, 4, 2, 3, 4096, 128, 40) == 32 * per
    assert lib.fa_fwd_splitkv_workspace_bytes(1, 4, 4, 3, 4096, 128, 1) == per
    assert lib.fa_fwd_splitkv_workspace_bytes(1, 4, 2, 3, 4096, 96, 1) == 0
    assert lib.fa_fwd_splitkv_workspace_bytes(1, 4, 3, 3, 4096, 128, 1) == 0   # 3 does not divide 4


def test_fp8_argument_checks_before_launch(fa):
    lib = fa.load()
    P = 0x10000
    signs = (ctypes.c_float * 128)(*([1.0, -1.0] * 64))
    bad = (ctypes.c_float * 128)(*([1.0] * 127 + [0.5]))
    sp = ctypes.cast(signs, ctypes.c_void_p)
    def quant(s=sp, x=P, BH=4, N=300, d=128):
        return lib.fa_fp8_quantize(x, s, P, P, BH, N, d, None)
    assert quant(s=None) == fa.FA_ERR_INVALID_ARG
    assert quant(s=ctypes.cast(bad, ctypes.c_void_p)) == fa.FA_ERR_INVALID_ARG   # not +-1
    assert quant(x=0) == fa.FA_ERR_INVALID_ARG
    assert quant(x=P + 8) == fa.FA_ERR_MISALIGNED
    assert quant(N=0) == fa.FA_ERR_INVALID_ARG
    assert quant(d=96) == fa.FA_ERR_UNSUPPORTED

    def fwd(B=1, Hq=4, Hkv=2, N=256, d=128, scale=0.125, ptrs=None):
        ptrs = ptrs or [P] * 7
        return lib.fa_fwd_fp8(*ptrs, B, Hq, Hkv, N, d, 1, scale, None)
    assert fwd(d=96) == fa.FA_ERR_UNSUPPORTED            # head dimension 64 or 128
    assert fwd(Hkv=3) == fa.FA_ERR_INVALID_ARG           # 3 does not divide 4
    assert fwd(scale=-1.0) == fa.FA_ERR_INVALID_ARG
    assert fwd(ptrs=[P, 0, P, P, P, P, P]) == fa.FA_ERR_INVALID_ARG   # no Q scales
    assert fwd(ptrs=[P, P, P, P + 4, P, P, P]) == fa.FA_ERR_MISALIGNED


def test_fp8_binding_checks_signs(fa):
    torch = pytest.importorskip("torch")
    with pytest.raises(ValueError):
        fa._lib._host_signs([1.0, -1.0], 128)
    arr = fa._lib._host_signs(torch.tensor([1.0, -1.0] * 32), 64)
    assert list(arr)[:4] == [1.0, -1.0, 1.0, -1.0]
