"""Device memory of the attention calls stays O(N d) at the long-sequence
workload (bf16, B=1 H=16 N=32768 d=128, causal).

Standard attention writes the N x N score matrix to device memory; at
N = 32000 that is about 2 GB per head in half precision ("LLM part 06:
FlashAttention - GPU SRAM, tiling and online softmax", section 1).  The tiled
path keeps scores on chip, so a forward plus a backward here allocates only
its outputs and the backward's O(N) workspace (D and the base-2 LSE per row).

What is counted: everything the binding allocates through PyTorch (the
outputs), measured as PyTorch's peak, plus everything the library allocates
itself (the workspace, taken on the stream from the device's default memory
pool when the caller passes none), measured as that pool's high-water mark.
The calls go through the C ABI.
"""

import ctypes

import pytest

from helpers import scale_for

pytestmark = pytest.mark.gpu

CU_MEMPOOL_ATTR_USED_MEM_HIGH = 8  # cuda.h, CUmemPool_attribute


def _default_pool_high_water(ordinal: int, reset: bool) -> int:
    """High-water mark in bytes of the device's default memory pool (the pool
    cudaMallocAsync draws from); optionally reset it first."""
    cu = ctypes.CDLL("libcuda.so.1")
    dev = ctypes.c_int()
    assert cu.cuDeviceGet(ctypes.byref(dev), ordinal) == 0
    pool = ctypes.c_void_p()
    assert cu.cuDeviceGetDefaultMemPool(ctypes.byref(pool), dev) == 0
    val = ctypes.c_uint64(0)
    if reset:
        assert cu.cuMemPoolSetAttribute(pool, CU_MEMPOOL_ATTR_USED_MEM_HIGH,
                                        ctypes.byref(val)) == 0
    assert cu.cuMemPoolGetAttribute(pool, CU_MEMPOOL_ATTR_USED_MEM_HIGH, ctypes.byref(val)) == 0
    return int(val.value)


def test_long_sequence_call_memory_is_linear_in_n():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import exact_io_aware_18_gb300 as fa

    B, H, N, d = 1, 16, 32768, 128
    dev = torch.device("cuda:0")
    gen = torch.Generator(device=dev)
    gen.manual_seed(3)
    q, k, v, do = (torch.randn(B, H, N, d, generator=gen, device=dev).to(torch.bfloat16)
                   for _ in range(4))
    s = scale_for(d)
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats(dev)
    base = torch.cuda.memory_allocated(dev)
    _default_pool_high_water(0, reset=True)

    o, lse = fa.attention_fwd(q, k, v, causal=True, scale=s)
    dq, dk, dv = fa.attention_bwd(q, k, v, o, do, lse, causal=True, scale=s)  # workspace: library
    torch.cuda.synchronize()
    torch_peak = torch.cuda.max_memory_allocated(dev) - base
    lib_peak = _default_pool_high_water(0, reset=False)
    assert fa.fa_device_status(clear=True) == fa.FA_OK

    elems = B * H * N * d
    outputs = elems * 2 + B * H * N * 4 + 3 * elems * 4  # O bf16, LSE, dQ dK dV fp32
    workspace = fa.fa_bwd_workspace_bytes(B, H, N, d)
    assert workspace == 2 * B * H * N * 4                 # N is a multiple of 128 here
    scores_one_head = N * N * 2                           # one bf16 N x N matrix: 2 GiB
    # PyTorch holds the outputs and nothing else the call asked for (its
    # allocator rounds each block up to 2 MiB at most).
    assert torch_peak <= outputs + 5 * (2 << 20)
    # The library's own allocation is the O(N) workspace (pool granularity 2 MiB).
    assert 0 < lib_peak <= workspace + (2 << 20)
    # Together: a few bytes per (row, column) of the inputs, far from N^2.
    total = torch_peak + lib_peak
    assert total <= 16 * elems
    assert total * 2 < scores_one_head
    for t in (o, lse, dq, dk, dv):
        assert bool(torch.isfinite(t).all())
