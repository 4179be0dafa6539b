"""Tensors past 2^31 elements: every global offset on the path is 64-bit.

B = 4, H = 32768, N = 129, d = 128 gives 2.16e9 elements per tensor (4.3 GB
in BF16, 8.7 GB per FP32 gradient), with a ragged last tile of one row.  The
forward and the backward run on the whole batch; the first head and the last
one (which lies past the 2^31-element mark in every tensor) are checked
against the oracle with the BF16 bounds.  Inputs are drawn on the device from
a seeded generator; the oracle receives the exact BF16 values of the checked
heads.
"""

import numpy as np
import pytest

import oracle
from helpers import (BF16_GRAD_MAX_ABS, BF16_GRAD_REL_RMS, BF16_LSE_MAX_ABS, BF16_O_MAX_ABS,
                     BF16_O_REL_RMS, max_abs, rel_rms, scale_for)

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


def test_tensors_beyond_2_31_elements(fa):
    import torch
    dev = torch.device("cuda:0")
    B, H, N, d = 4, 32768, 129, 128
    assert B * H * N * d > 2 ** 31
    s = scale_for(d)
    gen = torch.Generator(device=dev)
    gen.manual_seed(11)

    def draw():
        return torch.randn(B, H, N, d, generator=gen, device=dev).to(torch.bfloat16)

    q, k, v, do = draw(), draw(), draw(), draw()
    o, lse = fa.attention_fwd(q, k, v, causal=True, scale=s)
    dq, dk, dv = fa.attention_bwd(q, k, v, o, do, lse, causal=True, scale=s)
    torch.cuda.synchronize()
    last = B * H - 1
    assert last * N * d > 2 ** 31

    def heads(t):  # heads 0 and B*H-1 as exact float64 values, [1, 2, N, d]
        flat = t.reshape(B * H, N, -1)
        return torch.stack([flat[0], flat[last]]).unsqueeze(0).double().cpu().numpy()

    xq, xk, xv, xdo = heads(q), heads(k), heads(v), heads(do)
    ro, rl = oracle.attention_fwd(xq, xk, xv, True, s)
    got_o = heads(o)
    got_lse = torch.stack([lse.reshape(B * H, N)[0],
                           lse.reshape(B * H, N)[last]]).unsqueeze(0).cpu().numpy()
    assert max_abs(got_o, ro) <= BF16_O_MAX_ABS
    assert rel_rms(got_o, ro) <= BF16_O_REL_RMS
    assert max_abs(got_lse, rl) <= BF16_LSE_MAX_ABS
    refs = oracle.attention_bwd(xq, xk, xv, xdo, True, s, o_storage="bf16")[:3]
    for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
        g = heads(got).reshape(2, N, d)
        assert max_abs(g, ref) <= BF16_GRAD_MAX_ABS, name
        assert rel_rms(g, ref) <= BF16_GRAD_REL_RMS, name
    assert np.isfinite(got_o).all()
