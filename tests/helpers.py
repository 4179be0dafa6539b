"""Shared test utilities: input upload, error metrics, row sampling."""

import json
import math
import os

import numpy as np

import fa_inputs

# Error bounds for the attention path (outputs vs the FP64 oracle).
BF16_O_MAX_ABS = 1e-2
BF16_O_REL_RMS = 5e-3
BF16_LSE_MAX_ABS = 1e-3
BF16_GRAD_MAX_ABS = 1e-2
BF16_GRAD_REL_RMS = 5e-3
F32_MAX_ABS = 1e-4


def scale_for(d):
    """1/sqrt(d) as the C float the library receives."""
    return float(np.float32(1.0 / math.sqrt(d)))


def to_device_bf16(bits, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def to_device_f32(x, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(device)


def max_abs(got, ref):
    return float(np.max(np.abs(np.asarray(got, dtype=np.float64) - ref))) if np.size(ref) else 0.0


def rel_rms(got, ref):
    ref = np.asarray(ref, dtype=np.float64)
    den = float(np.sqrt(np.sum(ref * ref)))
    num = float(np.sqrt(np.sum((np.asarray(got, dtype=np.float64) - ref) ** 2)))
    return num / den if den > 0 else num


def sample_rows(seed, BH, N, n_random, heads=None):
    """(heads, rows): every head listed gets the tile-edge rows plus random ones."""
    rng = np.random.default_rng(seed)
    heads = list(range(BH)) if heads is None else list(heads)
    fixed = {0, 1, N - 1, N - 2}
    for t in range(0, N, 128):
        fixed.update({t - 1, t, t + 1})
    fixed = sorted(r for r in fixed if 0 <= r < N)
    hs, rs = [], []
    for h in heads:
        rows = set(fixed)
        rows.update(int(r) for r in rng.integers(0, N, size=n_random))
        for r in sorted(rows):
            hs.append(h)
            rs.append(r)
    return np.array(hs, dtype=np.int64), np.array(rs, dtype=np.int64)


def inputs(seed, B, H, N, d, dtype="bf16", names=("q", "k", "v", "do")):
    return fa_inputs.attention_inputs(seed, B, H, N, d, dtype, names)


def oracle_o_lse_on_device(x, causal, scale, device):
    """The oracle's O rounded to bf16 (as the oracle rounds the O its
    backward forms D from) and its LSE rounded to float32, on the device:
    the inputs a backward gets when compared with the oracle on equal inputs."""
    import torch
    import oracle
    ro, rl = oracle.attention_fwd(x["q"], x["k"], x["v"], causal, scale)
    ob = oracle.stored_output(ro, "bf16").astype(np.float32)
    bits = fa_inputs.bf16_bits(ob)  # exact: ob already holds bf16 values
    o = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    lse = torch.from_numpy(np.ascontiguousarray(rl, dtype=np.float32))
    return o.to(device), lse.to(device)


def diagnostic(what, **values):
    """A measured figure that is reported, not asserted: printed (visible
    with pytest -s or -rP) and, when FA_DIAGNOSTICS names a file, appended
    to it as one JSON line."""
    line = {"what": what, **{k: float(v) for k, v in values.items()}}
    print("DIAGNOSTIC", json.dumps(line))
    path = os.environ.get("FA_DIAGNOSTICS")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(line) + "\n")
