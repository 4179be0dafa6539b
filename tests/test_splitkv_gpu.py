"""GPU parity for the split-KV decode forward against the FP64 oracle's
definition: every query attends to all Nk keys (no mask), query head h with
K/V head h // (Hq / Hkv).  The chunks' partial results are merged on the GPU;
the result must equal the plain definition over all keys.  Calls go through
the C ABI (fa_fwd_splitkv)."""

import numpy as np
import pytest

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


def _decode_inputs(seed, B, Hq, Hkv, Nq, Nk, d):
    """Q: the first Nq rows of a draw of Nk rows; K, V: the first Hkv heads."""
    x = inputs(seed, B, Hq, Nk, d, names=("q", "k", "v"))
    out = {}
    for n, heads, rows in (("q", Hq, Nq), ("k", Hkv, Nk), ("v", Hkv, Nk)):
        out[n] = np.ascontiguousarray(x[n][:, :heads, :rows])
        out[n + "_bits"] = np.ascontiguousarray(x[n + "_bits"][:, :heads, :rows])
    return out


def _run(fa, x, s, n_splits):
    import torch
    dev = torch.device("cuda:0")
    q, k, v = (to_device_bf16(x[n + "_bits"], dev) for n in ("q", "k", "v"))
    o, lse = fa.attention_decode(q, k, v, scale=s, n_splits=n_splits)
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), lse.cpu().numpy()


CASES = [  # B, Hq, Hkv, Nq, Nk, d, n_splits (0: the library's choice)
    (2, 8, 2, 1, 4096, 128, 0),
    (1, 4, 4, 16, 3000, 64, 7),
    (1, 4, 1, 130, 1000, 128, 3),
    (1, 2, 2, 5, 129, 64, 50),     # more splits asked for than key tiles
    (4, 8, 8, 1, 257, 128, 0),
]


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,n_splits", CASES)
def test_splitkv_matches_oracle(fa, B, Hq, Hkv, Nq, Nk, d, n_splits):
    x = _decode_inputs(700 + Nk + Nq, B, Hq, Hkv, Nq, Nk, d)
    s = scale_for(d)
    o, lse = _run(fa, x, s, n_splits)
    ro, rl = oracle.attention_fwd_gqa(x["q"], x["k"], x["v"], False, s)
    assert max_abs(o, ro) <= BF16_O_MAX_ABS
    assert rel_rms(o, ro) <= BF16_O_REL_RMS
    assert max_abs(lse, rl) <= BF16_LSE_MAX_ABS


def test_one_split_is_the_forward(fa):
    """With one chunk the merge is the identity: the bits of fa_fwd_gqa."""
    import torch
    B, Hq, Hkv, N, d = 1, 4, 2, 300, 128
    x = _decode_inputs(31, B, Hq, Hkv, N, N, d)
    s = scale_for(d)
    dev = torch.device("cuda:0")
    q, k, v = (to_device_bf16(x[n + "_bits"], dev) for n in ("q", "k", "v"))
    o1, l1 = fa.attention_decode(q, k, v, scale=s, n_splits=1)
    o2, l2 = fa.attention_fwd(q, k, v, causal=False, scale=s)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_split_count_changes_only_rounding(fa):
    """Different chunkings agree with each other within the output bounds."""
    x = _decode_inputs(32, 2, 8, 2, 1, 8192, 128)
    s = scale_for(128)
    o_a, l_a = _run(fa, x, s, 1)
    o_b, l_b = _run(fa, x, s, 64)
    assert max_abs(o_a, o_b) <= BF16_O_MAX_ABS
    assert max_abs(l_a, l_b) <= BF16_LSE_MAX_ABS


def test_splitkv_at_the_benched_decode_shape(fa):
    """B=4 Hq=32 Hkv=8 Nq=1 Nk=16384 d=128 with the library's own split
    count, the configuration the bench times: every query row against the
    oracle."""
    B, Hq, Hkv, Nq, Nk, d = 4, 32, 8, 1, 16384, 128
    # K, V for the K/V heads only (the first two tensors of one seeded draw),
    # Q at its own size from another seed.
    kv = inputs(4, B, Hkv, Nk, d, names=("q", "k"))
    qx = inputs(5, B, Hq, Nq, d, names=("q",))
    x = {"q": qx["q"], "q_bits": qx["q_bits"], "k": kv["q"], "k_bits": kv["q_bits"],
         "v": kv["k"], "v_bits": kv["k_bits"]}
    s = scale_for(d)
    o, lse = _run(fa, x, s, 0)
    ro, rl = oracle.attention_fwd_gqa(x["q"], x["k"], x["v"], False, s)
    assert max_abs(o, ro) <= BF16_O_MAX_ABS
    assert rel_rms(o, ro) <= BF16_O_REL_RMS
    assert max_abs(lse, rl) <= BF16_LSE_MAX_ABS
