"""Seeded synthetic inputs for exact attention, shared by every consumer.

The oracle tests, the CUDA parity tests and ``bench.py`` all draw their
inputs from here, so that both sides of a comparison see the same numbers.
This module holds no attention arithmetic at all: it only turns a seed and a
list of shapes into i.i.d. standard-normal samples and, for bfloat16
workloads, rounds them to bfloat16.

Generator (the same on x86-64 and aarch64):

* splitmix64 counter stream: the k-th 64-bit word of seed ``s`` is
  ``mix64(s + (k + 1) * 0x9E3779B97F4A7C15)``, with ``mix64`` the published
  splitmix64 finaliser (shift/xor/multiply by 0xBF58476D1CE4E5B9 and
  0x94D049BB133111EB);
* Box-Muller in double precision on consecutive word pairs (2p, 2p+1):
  ``u1 = ((w0 >> 11) + 1) * 2**-53`` in (0, 1], ``u2 = (w1 >> 11) * 2**-53``,
  ``z0 = sqrt(-2 ln u1) cos(2 pi u2)``, ``z1 = sqrt(-2 ln u1) sin(2 pi u2)``;
* cast to float32, then (bf16 workloads) round to nearest even on the top 16
  bits of the float32 pattern.

Tensors are drawn in the order Q, K, V, dO from one stream per seed, each of
shape [B, H, N, d] in row-major order, one after the other.
"""

from __future__ import annotations

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK_PAIRS = 1 << 21


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def splitmix64_words(seed: int, start: int, count: int) -> np.ndarray:
    """Words ``start .. start+count-1`` of the splitmix64 stream of ``seed``."""
    k = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + k * _GOLDEN)


def normal_stream(seed: int, start: int, count: int) -> np.ndarray:
    """float32 samples ``start .. start+count-1`` of the normal stream of ``seed``.

    ``start`` and ``count`` must be even (samples come in Box-Muller pairs).
    """
    if start % 2 or count % 2:
        raise ValueError("normal_stream works on whole Box-Muller pairs")
    out = np.empty(count, dtype=np.float32)
    two_pi = 2.0 * np.pi
    scale = 2.0 ** -53
    done = 0
    while done < count:
        n = min(count - done, 2 * _CHUNK_PAIRS)
        w = splitmix64_words(seed, start + done, n)
        w0 = w[0::2] >> np.uint64(11)
        w1 = w[1::2] >> np.uint64(11)
        u1 = (w0.astype(np.float64) + 1.0) * scale
        u2 = w1.astype(np.float64) * scale
        r = np.sqrt(-2.0 * np.log(u1))
        t = two_pi * u2
        chunk = out[done:done + n]
        chunk[0::2] = (r * np.cos(t)).astype(np.float32)
        chunk[1::2] = (r * np.sin(t)).astype(np.float32)
        done += n
    return out


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); uint16 patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    with np.errstate(over="ignore"):
        return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact float32 values of bfloat16 bit patterns."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def attention_inputs(seed: int, B: int, H: int, N: int, d: int, dtype: str = "bf16",
                     names=("q", "k", "v", "do")) -> dict:
    """Q, K, V, dO for one workload, drawn in that order from ``seed``.

    Returns a dict of float32 arrays of shape [B, H, N, d] whose values are
    exactly representable in ``dtype``; for ``dtype == "bf16"`` the dict also
    holds the uint16 patterns under ``"<name>_bits"``.  ``names`` selects a
    prefix of (q, k, v, do): asking for fewer tensors never changes the ones
    returned.
    """
    if dtype not in ("bf16", "f32"):
        raise ValueError(f"dtype must be bf16 or f32, got {dtype!r}")
    order = ("q", "k", "v", "do")
    if tuple(names) != order[:len(names)]:
        raise ValueError("names must be a prefix of (q, k, v, do)")
    size = B * H * N * d
    pad = size + (size % 2)
    out = {}
    for t, name in enumerate(names):
        z = normal_stream(seed, t * pad, pad)[:size].reshape(B, H, N, d)
        if dtype == "bf16":
            bits = bf16_bits(z)
            out[name + "_bits"] = bits
            out[name] = bf16_to_f32(bits)
        else:
            out[name] = z
    return out


def random_signs(seed: int, d: int) -> np.ndarray:
    """d random signs (+1.0 / -1.0, float32): entry i is -1 when bit 63 of word
    i of the splitmix64 stream of ``seed`` is set."""
    w = splitmix64_words(seed, 0, d)
    return np.where((w >> np.uint64(63)) == 1, np.float32(-1.0), np.float32(1.0)).astype(np.float32)
