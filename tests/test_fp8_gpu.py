"""GPU parity for the FP8 forward with incoherent processing against the
oracle's definition (block-quantised E4M3 codes of Q R and K R, R =
diag(signs) H / sqrt(d), then FP64 attention on the dequantised values).

The quantisation is integer work decided in float32, so the GPU's codes and
scales must equal the oracle's bit for bit.  O and LSE then carry the BF16
forward's error bounds: the scores' codes are exact on both sides, and what
differs is the FP32 accumulation of the code products and BF16 P V.  Calls go
through the C ABI (fa_fp8_quantize, fa_fwd_fp8).
"""

import numpy as np
import pytest

import fa_inputs
import oracle
from helpers import (BF16_LSE_MAX_ABS, BF16_O_MAX_ABS, BF16_O_REL_RMS, inputs, max_abs, rel_rms,
                     scale_for, to_device_bf16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import exact_io_aware_18_gb300 as pkg
    pkg.fa_set_wait_timeout_ns(1_000_000_000)
    pkg.fa_device_status(clear=True)
    yield pkg
    assert pkg.fa_device_status(clear=True) == pkg.FA_OK


def _e4m3_values():
    """Value of every E4M3 byte from the format's bit fields (NaN for S.1111.111)."""
    out = np.empty(256, dtype=np.float64)
    for code in range(256):
        s, e, m = code >> 7, (code >> 3) & 15, code & 7
        if e == 15 and m == 7:
            out[code] = np.nan
            continue
        v = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
        out[code] = -v if s else v
    return out


E4M3 = _e4m3_values()


@pytest.mark.parametrize("B,H,N,d,seed", [(1, 3, 300, 128, 1), (2, 2, 129, 64, 2),
                                          (1, 2, 1024, 128, 3)])
def test_quantize_codes_and_scales_are_exact(fa, B, H, N, d, seed):
    import torch
    x = inputs(seed, B, H, N, d, names=("q",))
    bits = x["q_bits"].copy()
    bits[0, 0, 128:256] = 0                        # an all-zero tile (scale 1)
    bits[-1, -1, :5, 7] = 0x4400                   # a few large entries (bf16 512)
    xf = fa_inputs.bf16_to_f32(bits)
    signs = fa_inputs.random_signs(seed + 10, d)
    codes, scales = fa.fp8_quantize(to_device_bf16(bits, torch.device("cuda:0")), signs)
    torch.cuda.synchronize()
    got = E4M3[codes.cpu().numpy()]
    want_c, want_s = oracle.quantize_e4m3_tiles(oracle.rotate_f32(xf, signs))
    assert not np.any(np.isnan(got))
    assert np.array_equal(got, want_c)
    assert np.array_equal(scales.cpu().numpy(), want_s)
    assert want_s[0, 0, 1] == 1.0


def _fp8_case(fa, seed, B, Hq, Hkv, N, d, causal):
    import torch
    dev = torch.device("cuda:0")
    x = inputs(seed, B, Hq, N, d, names=("q", "k", "v"))
    for n in ("k", "v"):
        x[n] = np.ascontiguousarray(x[n][:, :Hkv])
        x[n + "_bits"] = np.ascontiguousarray(x[n + "_bits"][:, :Hkv])
    signs = fa_inputs.random_signs(seed + 100, d)
    s = scale_for(d)
    q, k, v = (to_device_bf16(x[n + "_bits"], dev) for n in ("q", "k", "v"))
    o, lse = fa.attention_fwd_fp8(q, k, v, signs, causal=causal, scale=s)
    torch.cuda.synchronize()
    o_ref, lse_ref, _, _ = oracle.attention_fwd_fp8(x["q"], x["k"], x["v"], signs, causal, s,
                                                    Hkv=Hkv)
    return o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref


CASES = [  # B, Hq, Hkv, N, d, causal
    (1, 2, 2, 300, 128, True),
    (2, 2, 2, 512, 128, False),
    (1, 4, 2, 257, 128, True),     # grouped-query, ragged last tile
    (1, 2, 1, 1000, 128, False),   # multi-query, several key tiles
    (1, 1, 1, 1, 128, True),       # one query, one key
    (1, 2, 2, 300, 64, True),      # d = 64: 64-byte rows of codes
    (2, 4, 2, 513, 64, False),     # d = 64, grouped-query, ragged last tile
]


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal", CASES)
def test_fp8_forward_matches_oracle(fa, B, Hq, Hkv, N, d, causal):
    o, lse, o_ref, lse_ref = _fp8_case(fa, 7 + N, B, Hq, Hkv, N, d, causal)
    assert max_abs(o, o_ref) <= BF16_O_MAX_ABS
    assert rel_rms(o, o_ref) <= BF16_O_REL_RMS
    assert max_abs(lse, lse_ref) <= BF16_LSE_MAX_ABS


def test_fp8_forward_is_deterministic(fa):
    import torch
    dev = torch.device("cuda:0")
    x = inputs(5, 2, 4, 700, 128, names=("q", "k", "v"))
    q, k, v = (to_device_bf16(x[n + "_bits"], dev) for n in ("q", "k", "v"))
    signs = fa_inputs.random_signs(5, 128)
    o1, l1 = fa.attention_fwd_fp8(q, k, v, signs, causal=True)
    o2, l2 = fa.attention_fwd_fp8(q, k, v, signs, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_fp8_forward_full_size_sampled_heads(fa):
    """The bench's shape (B=8, H=16, N=2048, d=128, causal): codes and scales of
    the whole Q and K exactly, O and LSE of four whole heads."""
    import torch
    B, H, N, d = 8, 16, 2048, 128
    dev = torch.device("cuda:0")
    x = inputs(4, B, H, N, d, names=("q", "k", "v"))
    signs = fa_inputs.random_signs(4, d)
    s = scale_for(d)
    q, k, v = (to_device_bf16(x[n + "_bits"], dev) for n in ("q", "k", "v"))
    q8, qs = fa.fp8_quantize(q, signs)
    k8, ks = fa.fp8_quantize(k, signs)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    fa.fa_fwd_fp8(q8, qs, k8, ks, v, o, lse, True, s)
    torch.cuda.synchronize()
    qc, qsc = oracle.quantize_e4m3_tiles(oracle.rotate_f32(x["q"], signs))
    kc, ksc = oracle.quantize_e4m3_tiles(oracle.rotate_f32(x["k"], signs))
    assert np.array_equal(E4M3[q8.cpu().numpy()], qc)
    assert np.array_equal(E4M3[k8.cpu().numpy()], kc)
    assert np.array_equal(qs.cpu().numpy(), qsc) and np.array_equal(ks.cpu().numpy(), ksc)
    o_h = o.float().cpu().numpy()
    lse_h = lse.cpu().numpy()
    for b, h in ((0, 0), (3, 7), (5, 12), (7, 15)):
        qd = (qc[b, h] * np.repeat(qsc[b, h].astype(np.float64), 128)[:N, None])[None, None]
        kd = (kc[b, h] * np.repeat(ksc[b, h].astype(np.float64), 128)[:N, None])[None, None]
        o_ref, lse_ref = oracle.attention_fwd(qd, kd, x["v"][b:b + 1, h:h + 1], True, s)
        assert max_abs(o_h[b, h], o_ref[0, 0]) <= BF16_O_MAX_ABS
        assert rel_rms(o_h[b, h], o_ref[0, 0]) <= BF16_O_REL_RMS
        assert max_abs(lse_h[b, h], lse_ref[0, 0]) <= BF16_LSE_MAX_ABS
