"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory
at call time (runtimes that reserve all device memory at start-up, or code
whose memory belongs to an allocator it must not bypass).  Its scratch is an
array built into the library; this file checks it against fa_bwd.

Kept in a file that pytest collects last, so that a run stopping at the first
failure has run every other test first; it also passes on its own.
"""

import pytest

from helpers import inputs, scale_for, to_device_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import exact_io_aware_18_gb300 as pkg
    return pkg


@pytest.mark.parametrize("B,H,N,d,causal", [(8, 16, 2048, 128, True), (1, 3, 300, 64, False)])
def test_noalloc_matches_fa_bwd_twice(fa, B, H, N, d, causal):
    import torch
    dev = torch.device("cuda:0")
    x = inputs(60 + N, B, H, N, d)
    s = scale_for(d)
    q, k, v, do = (to_device_bf16(x[n + "_bits"], dev) for n in ("q", "k", "v", "do"))
    o, lse = fa.attention_fwd(q, k, v, causal=causal, scale=s)
    ref = fa.attention_bwd(q, k, v, o, do, lse, causal=causal, scale=s)
    for _ in range(2):  # the second call runs on the scratch the first one left behind
        got = [torch.full(q.shape, float("nan"), dtype=torch.float32, device=dev)
               for _ in range(3)]
        fa.fa_bwd_noalloc(q, k, v, o, do, lse, *got, causal, s)
        torch.cuda.synchronize()
        # The same kernels on the same inputs, each gradient entry one sum in
        # a fixed order: the results agree bit for bit.
        for g, r in zip(got, ref):
            assert torch.equal(g, r)
    assert fa.fa_device_status(clear=True) == fa.FA_OK


def test_noalloc_rejects_workloads_beyond_its_scratch(fa):
    lib = fa.load()
    # 2 * 4 * B*H*roundup(N,128) bytes: 1 x 1 x 2^20 + 128 rows is one tile past the limit.
    n_rows = fa._lib.NOALLOC_SCRATCH_BYTES // 8
    rc = lib.fa_bwd_noalloc(*([0x10000] * 9), 1, 1, n_rows + 1, 128, 1, 0.088, None)
    assert rc == fa.FA_ERR_NO_MEMORY
    rc = lib.fa_bwd_noalloc(*([0x10000] * 9), 1, 1, 16, 96, 1, 0.088, None)
    assert rc == fa.FA_ERR_UNSUPPORTED


@pytest.mark.parametrize("B,H,N,d,scale", [(70000, 1, 1, 128, 0.088), (1, 1, 16, 96, 0.088),
                                           (1, 1, 0, 64, 0.125), (1, 1, 16, 64, -1.0)])
def test_noalloc_rejects_what_fa_bwd_rejects_with_the_same_status(fa, B, H, N, d, scale):
    """Argument errors come back before anything is launched, with the code
    fa_bwd gives for the same arguments (its checks run first)."""
    lib = fa.load()
    ptrs = [0x10000] * 9
    want = lib.fa_bwd(*ptrs, B, H, N, d, 1, scale, None, 0, None)
    assert want != fa.FA_OK
    assert lib.fa_bwd_noalloc(*ptrs, B, H, N, d, 1, scale, None) == want
