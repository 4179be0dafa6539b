"""Pins of the FP64 CPU oracle to facts the pages and the mathematics fix.

None of these re-types the oracle's own formula: each checks a property that
a correct attention must have and that a plausible slip in the oracle (a
dropped term, a wrong sign or index, a transposed operand, a wrong mask or
scale) would break.  All run on the CPU in well under a minute.
"""

import math
import os

import numpy as np
import pytest

import fa_inputs


def _scale(d):
    # the API takes scale as a C float; the oracle promotes that float to double
    return float(np.float32(1.0 / math.sqrt(d)))


def _rand(seed, B, H, N, d):
    x = fa_inputs.attention_inputs(seed, B, H, N, d, "f32")
    return x["q"], x["k"], x["v"], x["do"]


# ---------------------------------------------------------------- softmax rows

@pytest.mark.parametrize("causal", [False, True])
def test_probability_rows_sum_to_one(oracle_lib, causal):
    q, k, _, _ = _rand(11, 1, 1, 37, 8)
    p = oracle_lib.attention_probs(q[0, 0], k[0, 0], causal, _scale(8))
    assert np.all(p >= 0.0)
    assert np.max(np.abs(p.sum(axis=1) - 1.0)) <= 1e-12
    if causal:  # key j visible to query i iff j <= i
        assert np.all(np.triu(p, 1) == 0.0)
        assert np.all(np.diag(p) > 0.0)
    else:
        assert np.all(p > 0.0)


# ------------------------------------------------- online-softmax merge (page 3)

def _block_stats(oracle_lib, q, k, v, scale):
    """Normalised O, block max m and l = sum exp(s - m) of one key block."""
    o, lse = oracle_lib.attention_fwd(q, k, v, False, scale)
    s = scale * np.einsum("bhid,bhjd->bhij", q.astype(np.float64), k.astype(np.float64))
    m = s.max(axis=-1)
    l = np.exp(lse - m)
    return o, m, l


def _merge(o1, m1, l1, o2_unnorm, m2, l2):
    """The two-block merge of the online-softmax page (section 2): O1 is the
    normalised running output, O2 the unnormalised block product."""
    m = np.maximum(m1, m2)
    l = l1 * np.exp(m1 - m) + l2 * np.exp(m2 - m)
    o = (o1 * (l1 * np.exp(m1 - m) / l)[..., None]
         + o2_unnorm * (np.exp(m2 - m) / l)[..., None])
    return o, m, l


def test_two_block_merge_equals_full_softmax_at_every_cut(oracle_lib):
    B, H, N, d = 1, 2, 12, 6
    q, k, v, _ = _rand(12, B, H, N, d)
    s = _scale(d)
    o_full, lse_full = oracle_lib.attention_fwd(q, k, v, False, s)
    for cut in range(1, N):
        o1, m1, l1 = _block_stats(oracle_lib, q, k[:, :, :cut], v[:, :, :cut], s)
        o2, m2, l2 = _block_stats(oracle_lib, q, k[:, :, cut:], v[:, :, cut:], s)
        o, m, l = _merge(o1, m1, l1, o2 * l2[..., None], m2, l2)
        assert np.max(np.abs(o - o_full)) <= 1e-12, cut
        assert np.max(np.abs(m + np.log(l) - lse_full)) <= 1e-12, cut


def test_three_way_fold_equals_full_softmax(oracle_lib):
    B, H, N, d = 2, 1, 15, 4
    q, k, v, _ = _rand(13, B, H, N, d)
    s = _scale(d)
    o_full, lse_full = oracle_lib.attention_fwd(q, k, v, False, s)
    cuts = [(0, 4), (4, 11), (11, 15)]
    o, m, l = _block_stats(oracle_lib, q, k[:, :, 0:4], v[:, :, 0:4], s)
    for a, b in cuts[1:]:
        o2, m2, l2 = _block_stats(oracle_lib, q, k[:, :, a:b], v[:, :, a:b], s)
        o, m, l = _merge(o, m, l, o2 * l2[..., None], m2, l2)
    assert np.max(np.abs(o - o_full)) <= 1e-12
    assert np.max(np.abs(m + np.log(l) - lse_full)) <= 1e-12


def _buggy_blocked_snippet(q, k, v, block, scale):
    """Restatement of the blocked PyTorch example on the Hindi page
    ("implementation details"): it keeps O already divided by L, yet rescales
    it by exp(M - M_new) alone before dividing by L_new, dropping the old L."""
    q, k, v = (np.asarray(t, dtype=np.float64) for t in (q, k, v))
    n = q.shape[0]
    o = np.zeros_like(q)
    lsum = np.zeros(n)
    mx = np.full(n, -np.inf)
    for i in range(0, n, block):
        rows = slice(i, i + block)
        for j in range(0, n, block):
            sblk = scale * q[rows] @ k[j:j + block].T
            m_new = np.maximum(mx[rows], sblk.max(axis=1))
            e = np.exp(sblk - m_new[:, None])
            a = np.exp(mx[rows] - m_new)
            l_new = a * lsum[rows] + e.sum(axis=1)
            o[rows] = (a[:, None] * o[rows] + e @ v[j:j + block]) / l_new[:, None]
            lsum[rows] = l_new
            mx[rows] = m_new
    return o


def test_oracle_differs_from_the_buggy_blocked_example(oracle_lib):
    N, d, block = 40, 8, 16
    q, k, v, _ = _rand(14, 1, 1, N, d)
    s = _scale(d)
    o, _ = oracle_lib.attention_fwd(q, k, v, False, s)
    # one block: the missing factor is L_old = 0, so the example is right
    one = _buggy_blocked_snippet(q[0, 0], k[0, 0], v[0, 0], N, s)
    assert np.max(np.abs(one - o[0, 0])) <= 1e-12
    # several blocks: the example is wrong and the oracle must not follow it
    many = _buggy_blocked_snippet(q[0, 0], k[0, 0], v[0, 0], block, s)
    assert np.max(np.abs(many - o[0, 0])) > 1e-2


# ------------------------------------------------------------- closed forms

def test_single_key_returns_v_and_its_score(oracle_lib):
    q, k, v, _ = _rand(15, 2, 3, 1, 16)
    s = _scale(16)
    for causal in (False, True):
        o, lse = oracle_lib.attention_fwd(q, k, v, causal, s)
        assert np.array_equal(o, v.astype(np.float64))
        for b in range(2):
            for h in range(3):
                want = s * math.fsum(float(x) * float(y) for x, y in zip(q[b, h, 0], k[b, h, 0]))
                assert abs(lse[b, h, 0] - want) <= 1e-12


def test_constant_value_rows(oracle_lib):
    B, H, N, d = 1, 2, 9, 5
    q, k, _, _ = _rand(16, B, H, N, d)
    row = np.array([0.5, -1.25, 3.0, 0.0, 2.0])
    v = np.broadcast_to(row, (B, H, N, d)).copy()
    for causal in (False, True):
        o, _ = oracle_lib.attention_fwd(q, k, v, causal, _scale(d))
        assert np.max(np.abs(o - row)) <= 1e-14


def test_first_causal_query(oracle_lib):
    B, H, N, d = 2, 2, 7, 8
    q, k, v, _ = _rand(17, B, H, N, d)
    s = _scale(d)
    o, lse = oracle_lib.attention_fwd(q, k, v, True, s)
    assert np.array_equal(o[:, :, 0], v[:, :, 0].astype(np.float64))
    want = s * np.einsum("bhd,bhd->bh", q[:, :, 0].astype(np.float64), k[:, :, 0].astype(np.float64))
    assert np.max(np.abs(lse[:, :, 0] - want)) <= 1e-12


def test_uniform_scores_forward(oracle_lib):
    B, H, N, d = 1, 1, 10, 4
    q, _, v, _ = _rand(18, B, H, N, d)
    k = np.zeros_like(q)
    o, lse = oracle_lib.attention_fwd(q, k, v, False, 0.3)
    assert np.max(np.abs(o - v.astype(np.float64).mean(axis=2, keepdims=True))) <= 1e-14
    assert np.max(np.abs(lse - math.log(N))) <= 1e-14
    o, lse = oracle_lib.attention_fwd(q, k, v, True, 0.3)
    prefix = np.cumsum(v.astype(np.float64), axis=2) / np.arange(1, N + 1)[:, None]
    assert np.max(np.abs(o - prefix)) <= 1e-14
    assert np.max(np.abs(lse[0, 0] - np.log(np.arange(1, N + 1)))) <= 1e-14


def test_uniform_scores_causal_dv(oracle_lib):
    B, H, N, d = 1, 1, 8, 3
    q, _, v, do = _rand(19, B, H, N, d)
    k = np.zeros_like(q)
    _, _, dv, _ = oracle_lib.attention_bwd(q, k, v, do, True, 0.7)
    do64 = do[0, 0].astype(np.float64)
    for j in range(N):
        want = sum(do64[i] / (i + 1) for i in range(j, N))
        assert np.max(np.abs(dv[0, j] - want)) <= 1e-14


# ------------------------------------------------------------- invariances

@pytest.mark.parametrize("causal", [False, True])
def test_key_shift_invariance(oracle_lib, causal):
    B, H, N, d = 1, 2, 11, 4
    q, k, v, _ = _rand(20, B, H, N, d)
    u = np.array([0.25, -0.5, 1.0, 0.125])
    s = _scale(d)
    o, lse = oracle_lib.attention_fwd(q, k, v, causal, s)
    o2, lse2 = oracle_lib.attention_fwd(q, k + u, v, causal, s)
    assert np.max(np.abs(o2 - o)) <= 1e-12
    assert np.max(np.abs(lse2 - (lse + s * q.astype(np.float64) @ u))) <= 1e-12


def test_permutation_invariance(oracle_lib):
    B, H, N, d = 1, 1, 13, 6
    q, k, v, _ = _rand(21, B, H, N, d)
    s = _scale(d)
    o, lse = oracle_lib.attention_fwd(q, k, v, False, s)
    perm = np.random.default_rng(0).permutation(N)
    o_kv, lse_kv = oracle_lib.attention_fwd(q, k[:, :, perm], v[:, :, perm], False, s)
    assert np.max(np.abs(o_kv - o)) <= 1e-12
    assert np.max(np.abs(lse_kv - lse)) <= 1e-12
    o_q, lse_q = oracle_lib.attention_fwd(q[:, :, perm], k, v, False, s)
    assert np.max(np.abs(o_q - o[:, :, perm])) <= 1e-14
    assert np.max(np.abs(lse_q - lse[:, :, perm])) <= 1e-14


def test_rows_entry_matches_full_forward(oracle_lib):
    B, H, N, d = 2, 3, 20, 8
    q, k, v, _ = _rand(22, B, H, N, d)
    s = _scale(d)
    for causal in (False, True):
        o, lse = oracle_lib.attention_fwd(q, k, v, causal, s)
        heads = np.array([0, 5, 3, 1, 2])
        rows = np.array([0, 19, 7, 1, 13])
        orow, lrow = oracle_lib.attention_fwd_rows(q, k, v, causal, s, heads, rows)
        assert np.array_equal(orow, o.reshape(B * H, N, d)[heads, rows])
        assert np.array_equal(lrow, lse.reshape(B * H, N)[heads, rows])


# ------------------------------------------------------------- gradients

@pytest.mark.parametrize("causal", [False, True])
def test_gradient_identities(oracle_lib, causal):
    B, H, N, d = 2, 1, 9, 5
    q, k, v, do = _rand(23, B, H, N, d)
    s = _scale(d)
    dq, dk, dv, dvec = oracle_lib.attention_bwd(q, k, v, do, causal, s)
    dk = dk.reshape(B, H, N, d)
    dv = dv.reshape(B, H, N, d)
    # rows of dS sum to zero, so the keys' gradients sum to zero
    assert np.max(np.abs(dk.sum(axis=2))) <= 1e-12
    # each query's probabilities sum to one, so sum_j dV_j = sum_i dO_i
    assert np.max(np.abs(dv.sum(axis=2) - do.astype(np.float64).sum(axis=2))) <= 1e-12
    # D_i = dO_i . O_i = sum_j P_ij dP_ij
    for b in range(B):
        p = oracle_lib.attention_probs(q[b, 0], k[b, 0], causal, s)
        dp = do[b, 0].astype(np.float64) @ v[b, 0].astype(np.float64).T
        assert np.max(np.abs((p * dp).sum(axis=1) - dvec[b])) <= 1e-12


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d", [(1, 2), (5, 3), (8, 4)])
def test_backward_matches_finite_differences(oracle_lib, causal, N, d):
    q, k, v, do = (t.astype(np.float64) for t in _rand(24 + N, 1, 1, N, d))
    s = 0.6

    def loss(qq, kk, vv):
        o, _ = oracle_lib.attention_fwd(qq, kk, vv, causal, s)
        return float((do * o).sum())

    dq, dk, dv, _ = oracle_lib.attention_bwd(q, k, v, do, causal, s)
    h = 1e-6
    for grad, which in ((dq, 0), (dk, 1), (dv, 2)):
        num = np.zeros((N, d))
        for i in range(N):
            for c in range(d):
                args_p = [q.copy(), k.copy(), v.copy()]
                args_m = [q.copy(), k.copy(), v.copy()]
                args_p[which][0, 0, i, c] += h
                args_m[which][0, 0, i, c] -= h
                num[i, c] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        scale_ref = max(1.0, np.max(np.abs(num)))
        assert np.max(np.abs(grad[0] - num)) <= 1e-6 * scale_ref, which


def test_backward_head_selection(oracle_lib):
    B, H, N, d = 2, 2, 6, 4
    q, k, v, do = _rand(30, B, H, N, d)
    full = oracle_lib.attention_bwd(q, k, v, do, True, 0.5)
    heads = np.array([3, 0])
    part = oracle_lib.attention_bwd(q, k, v, do, True, 0.5, heads=heads)
    for a, b in zip(full, part):
        assert np.array_equal(a[heads], b)


def test_backward_d_uses_exact_forward_output(oracle_lib):
    B, H, N, d = 1, 1, 7, 3
    q, k, v, do = _rand(31, B, H, N, d)
    o, _ = oracle_lib.attention_fwd(q, k, v, True, 0.5)
    _, _, _, dvec = oracle_lib.attention_bwd(q, k, v, do, True, 0.5)
    assert np.max(np.abs(dvec[0] - (do[0, 0].astype(np.float64) * o[0, 0]).sum(axis=1))) <= 1e-14


def test_oracle_rejects_bad_arguments(oracle_lib):
    q = np.zeros((1, 1, 4, 2))
    with pytest.raises(RuntimeError):
        oracle_lib.attention_fwd_rows(q, q, q, False, 1.0, np.array([1]), np.array([0]))
    with pytest.raises(RuntimeError):
        oracle_lib.attention_fwd_rows(q, q, q, False, 1.0, np.array([0]), np.array([4]))


# ------------------------------------------------- D from the stored output

def test_round_bf16_fixed_values(oracle_lib):
    r = oracle_lib.round_bf16
    for exact in (1.0, -2.5, 0.15625, 3.140625, 2.0 ** -100, -(2.0 ** 100), 0.0):
        assert r(exact) == exact
    assert r(1.0 + 2.0 ** -8) == 1.0                       # tie, even neighbour below
    assert r(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6       # tie, even neighbour above
    assert r(1.0 + 0.7 * 2.0 ** -7) == 1.0 + 2.0 ** -7     # nearest
    assert r(300.5) == 300.0                               # spacing 2 between 256 and 512
    assert r(-(1.0 + 3 * 2.0 ** -8)) == -(1.0 + 2.0 ** -6)


def test_round_bf16_matches_float32_bit_rounding(oracle_lib):
    # float32 inputs: a single rounding either way, so the two independent
    # implementations (frexp/nearbyint in the oracle, integer bit arithmetic in
    # the input generator) must agree exactly.
    x = np.random.default_rng(5).standard_normal(20000).astype(np.float32) * 7
    want = fa_inputs.bf16_to_f32(fa_inputs.bf16_bits(x)).astype(np.float64)
    got = np.array([oracle_lib.round_bf16(float(t)) for t in x])
    assert np.array_equal(got, want)


def test_stored_output_rounds_like_the_generator(oracle_lib):
    # stored_output is the O a backward is handed: each value rounded by the
    # oracle's own bf16 rounding, which agrees with the input generator's
    # independent bit arithmetic on float32 values (one rounding either way).
    x = np.random.default_rng(6).standard_normal((3, 41)).astype(np.float32) * 5
    got = oracle_lib.stored_output(x, "bf16")
    want = fa_inputs.bf16_to_f32(fa_inputs.bf16_bits(x)).astype(np.float64)
    assert got.shape == x.shape and np.array_equal(got, want)
    assert np.array_equal(oracle_lib.stored_output(x, "f32"), x.astype(np.float64))
    y = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 300.5, 0.0, -2.5])
    assert np.array_equal(oracle_lib.stored_output(y, "bf16"),
                          [1.0, 1.0 + 2.0 ** -6, 300.0, 0.0, -2.5])
    assert np.array_equal(oracle_lib.stored_output(y, "exact"), y)


def test_stored_output_is_what_the_backward_forms_d_from(oracle_lib):
    B, H, N, d = 1, 2, 9, 8
    q, k, v, do = _rand(34, B, H, N, d)
    o, _ = oracle_lib.attention_fwd(q, k, v, True, 0.5)
    *_, dvec = oracle_lib.attention_bwd(q, k, v, do, True, 0.5, o_storage="bf16")
    ob = oracle_lib.stored_output(o, "bf16")
    want = (do.astype(np.float64) * ob).sum(axis=3).reshape(B * H, N)
    assert np.max(np.abs(dvec - want)) <= 1e-12


def test_stored_output_d(oracle_lib):
    B, H, N, d = 1, 1, 7, 6
    q, k, v, do = _rand(32, B, H, N, d)
    o, _ = oracle_lib.attention_fwd(q, k, v, True, 0.5)
    *_, d_exact = oracle_lib.attention_bwd(q, k, v, do, True, 0.5)
    *_, d_bf16 = oracle_lib.attention_bwd(q, k, v, do, True, 0.5, o_storage="bf16")
    *_, d_f32 = oracle_lib.attention_bwd(q, k, v, do, True, 0.5, o_storage="f32")
    do64 = do[0, 0].astype(np.float64)
    o_b = fa_inputs.bf16_to_f32(fa_inputs.bf16_bits(o[0, 0].astype(np.float32))).astype(np.float64)
    assert np.max(np.abs(d_bf16[0] - (do64 * o_b).sum(axis=1))) <= 1e-12
    o_f = o[0, 0].astype(np.float32).astype(np.float64)
    assert np.max(np.abs(d_f32[0] - (do64 * o_f).sum(axis=1))) <= 1e-12
    assert np.max(np.abs(d_bf16 - d_exact)) > 1e-6  # the rounding is really applied


def test_stored_output_is_exact_when_o_is_representable(oracle_lib):
    # One key: O = V, which is already a bf16 value, so rounding O changes nothing.
    q, k, v, do = _rand(33, 1, 2, 1, 8)
    v = fa_inputs.bf16_to_f32(fa_inputs.bf16_bits(v))
    a = oracle_lib.attention_bwd(q, k, v, do, False, 0.5)
    b = oracle_lib.attention_bwd(q, k, v, do, False, 0.5, o_storage="bf16")
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


# ---------------------------------------------------------------- grouped-query attention

def _gqa_inputs(seed, B, Hq, Hkv, N, d):
    q, k, v, do = _rand(seed, B, Hq, N, d)
    return q, np.ascontiguousarray(k[:, :Hkv]), np.ascontiguousarray(v[:, :Hkv]), do


def test_gqa_with_one_query_head_per_group_is_mha(oracle_lib):
    q, k, v, do = _rand(40, 2, 3, 9, 4)
    for causal in (False, True):
        a = oracle_lib.attention_fwd(q, k, v, causal, 0.5)
        b = oracle_lib.attention_fwd_gqa(q, k, v, causal, 0.5)
        assert all(np.array_equal(x, y) for x, y in zip(a, b))
        ga = oracle_lib.attention_bwd(q, k, v, do, causal, 0.5)
        gb = oracle_lib.attention_bwd_gqa(q, k, v, do, causal, 0.5)
        for x, y in zip(ga, gb):
            assert np.array_equal(x.reshape(y.shape), y)


@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (6, 3), (4, 1)])
def test_gqa_query_head_reads_its_group(oracle_lib, Hq, Hkv):
    # query head h attends with K/V head h // (Hq / Hkv), one head at a time
    B, N, d = 2, 7, 4
    q, k, v, _ = _gqa_inputs(41, B, Hq, Hkv, N, d)
    g = Hq // Hkv
    o, lse = oracle_lib.attention_fwd_gqa(q, k, v, True, 0.5)
    for b in range(B):
        for h in range(Hq):
            j = h // g
            o1, l1 = oracle_lib.attention_fwd(q[b:b + 1, h:h + 1], k[b:b + 1, j:j + 1],
                                              v[b:b + 1, j:j + 1], True, 0.5)
            assert np.array_equal(o[b, h], o1[0, 0]) and np.array_equal(lse[b, h], l1[0, 0])


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (3, 1)])
def test_gqa_backward_matches_finite_differences(oracle_lib, causal, Hq, Hkv):
    # perturbing one K/V entry moves every query head of its group, so this
    # pins the group sums of dK and dV as well as dQ
    N, d, s = 5, 3, 0.6
    q, k, v, do = (t.astype(np.float64) for t in _gqa_inputs(42 + Hq, 1, Hq, Hkv, N, d))

    def loss(qq, kk, vv):
        o, _ = oracle_lib.attention_fwd_gqa(qq, kk, vv, causal, s)
        return float((do * o).sum())

    dq, dk, dv, _ = oracle_lib.attention_bwd_gqa(q, k, v, do, causal, s)
    h = 1e-6
    for grad, which in ((dq, 0), (dk, 1), (dv, 2)):
        base = (q, k, v)[which]
        num = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            args_p = [q.copy(), k.copy(), v.copy()]
            args_m = [q.copy(), k.copy(), v.copy()]
            args_p[which][idx] += h
            args_m[which][idx] -= h
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        scale_ref = max(1.0, np.max(np.abs(num)))
        assert np.max(np.abs(grad - num)) <= 1e-6 * scale_ref, which


def test_gqa_rejects_heads_that_do_not_divide(oracle_lib):
    q = np.zeros((1, 3, 4, 2))
    k = np.zeros((1, 2, 4, 2))
    with pytest.raises(ValueError):
        oracle_lib.attention_fwd_gqa(q, k, k, False, 1.0)


# ---------------------------------------------------------------- FP8 (E4M3) and incoherent processing

def _e4m3_table():
    """Every finite E4M3 value, decoded from the bit fields of the format
    (sign, 4-bit exponent with bias 7, 3-bit mantissa; exponent field 0 is
    subnormal; the all-ones pattern S.1111.111 is NaN)."""
    vals = []
    for code in range(256):
        s, e, m = code >> 7, (code >> 3) & 15, code & 7
        if e == 15 and m == 7:
            continue
        v = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
        vals.append((-v if s else v, code))
    return vals


def test_e4m3_codes_are_fixed_points(oracle_lib):
    table = _e4m3_table()
    v = np.array([t[0] for t in table])
    assert np.array_equal(oracle_lib.round_e4m3(v), v)
    pos = np.unique(v[v >= 0])
    assert pos.max() == 448.0 and pos[1] == 2.0 ** -9 and len(pos) == 127


def test_e4m3_ties_to_even_and_saturates(oracle_lib):
    # the midpoint of two neighbours goes to the one whose mantissa is even
    by_val = {}
    for v, code in _e4m3_table():
        if v >= 0:
            by_val[v] = code
    pos = sorted(by_val)
    lo, hi = np.array(pos[:-1]), np.array(pos[1:])
    mid = (lo + hi) / 2
    got = oracle_lib.round_e4m3(np.concatenate([mid, -mid]))
    want = np.where([by_val[a] % 2 == 0 for a in lo], lo, hi)
    assert np.array_equal(got, np.concatenate([want, -want]))
    # just off the midpoint the nearer neighbour wins
    eps = (hi - lo) * 1e-3
    assert np.array_equal(oracle_lib.round_e4m3(mid - eps), lo)
    assert np.array_equal(oracle_lib.round_e4m3(mid + eps), hi)
    # beyond the largest finite value: saturation, not infinity or NaN
    assert np.array_equal(oracle_lib.round_e4m3([449.0, 1e6, -3e38]), [448.0, 448.0, -448.0])
    assert oracle_lib.round_e4m3([0.0])[0] == 0.0


def test_e4m3_matches_torch_float8(oracle_lib):
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    x = fa_inputs.normal_stream(5, 0, 20000).astype(np.float32) * np.float32(60.0)
    x = np.clip(x, -448.0, 448.0)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(oracle_lib.round_e4m3(x), ref)


@pytest.mark.parametrize("d", [64, 128])
def test_fwht_is_the_sylvester_hadamard_product(oracle_lib, d):
    scipy_linalg = pytest.importorskip("scipy.linalg")
    x = fa_inputs.normal_stream(7, 0, 6 * d).reshape(6, d)
    H = scipy_linalg.hadamard(d).astype(np.float64)
    got = oracle_lib.fwht_f32(x).astype(np.float64)
    want = x.astype(np.float64) @ H  # H is symmetric
    assert np.max(np.abs(got - want)) <= 1e-5 * np.max(np.abs(want))
    # applied twice it is d times the identity
    twice = oracle_lib.fwht_f32(oracle_lib.fwht_f32(x)).astype(np.float64)
    assert np.max(np.abs(twice - d * x)) <= 1e-4 * d


def test_fwht_butterfly_order_is_fixed(oracle_lib):
    # exact small case: the first stage pairs neighbours, the last pairs halves
    x = np.array([1.0, 2.0, 4.0, 8.0], dtype=np.float32)
    assert np.array_equal(oracle_lib.fwht_f32(x), np.array([15.0, -5.0, -9.0, 3.0], np.float32))


def test_rotation_is_orthogonal_and_keeps_scores(oracle_lib):
    d = 128
    signs = fa_inputs.random_signs(3, d)
    assert set(np.unique(signs)) == {-1.0, 1.0}
    q, k, _, _ = _rand(21, 1, 2, 40, d)
    qr = oracle_lib.rotate_f32(q, signs).astype(np.float64)
    kr = oracle_lib.rotate_f32(k, signs).astype(np.float64)
    s0 = q.astype(np.float64) @ np.swapaxes(k.astype(np.float64), -1, -2)
    s1 = qr @ np.swapaxes(kr, -1, -2)
    assert np.max(np.abs(s1 - s0)) <= 1e-4
    assert np.allclose(np.linalg.norm(qr, axis=-1), np.linalg.norm(q, axis=-1), rtol=1e-5)
    # the rotation is not the identity, and the signs matter
    assert np.max(np.abs(qr - q)) > 0.5
    other = oracle_lib.rotate_f32(q, np.ones(d, np.float32)).astype(np.float64)
    assert np.max(np.abs(other - qr)) > 0.5


def test_tile_quantisation_bounds_and_independence(oracle_lib):
    x = fa_inputs.normal_stream(9, 0, 2 * 300 * 64).reshape(1, 2, 300, 64)
    x[0, 1, 128:256] *= np.float32(37.0)      # one tile far larger than the others
    x[0, 0, 256:] = 0.0                       # an all-zero ragged tail tile
    codes, scales = oracle_lib.quantize_e4m3_tiles(x)
    assert scales.shape == (1, 2, 3)
    assert np.all(np.abs(codes) <= 448.0)
    assert scales[0, 0, 2] == 1.0 and np.all(codes[0, 0, 256:] == 0.0)
    for h in range(2):
        for t in range(3):
            blk = x[0, h, t * 128:(t + 1) * 128].astype(np.float64)
            c = codes[0, h, t * 128:(t + 1) * 128]
            if not np.any(blk):
                continue
            amax = np.abs(blk).max()
            assert np.isclose(scales[0, h, t], amax / 448.0, rtol=1e-6)
            assert np.abs(c).max() == 448.0           # the tile's largest entry hits the top code
            err = np.abs(c * scales[0, h, t] - blk)
            # E4M3 keeps 3 mantissa bits: half a spacing is at most 2^-4 of the
            # value, and at most 2^-10 * scale among subnormals
            assert np.all(err <= np.maximum(np.abs(blk) * 2.0 ** -4, 2.0 ** -10 * scales[0, h, t]) * 1.0001)
    # scaling one tile by a power of two moves only that tile's scale
    y = x.copy()
    y[0, 1, :128] *= np.float32(8.0)
    c2, s2 = oracle_lib.quantize_e4m3_tiles(y)
    assert np.array_equal(c2, codes)
    assert s2[0, 1, 0] == 8.0 * scales[0, 1, 0] and np.array_equal(s2[0, :, 1:], scales[0, :, 1:])


def _golden(name):
    vals = {}
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", name)) as f:
        for line in f:
            line = line.split("#", 1)[0].split()
            if len(line) == 2:
                vals[line[0]] = int(line[1], 0)
    return vals


def test_tile_scale_rule_on_a_hand_worked_tile(oracle_lib):
    # tests/golden/fp8_scale_rule.txt: a tile whose code differs between
    # x * (448 / amax) and x / (amax / 448); the fixture's float32 steps are
    # re-derived here with IEEE float32 arithmetic before the oracle is asked.
    g = _golden("fp8_scale_rule.txt")
    f32 = lambda bits: np.uint32(bits).view(np.float32)  # noqa: E731
    amax, xv = f32(g["amax_bits"]), f32(g["x_bits"])
    m = np.float32(np.float32(448.0) / amax)
    assert m.view(np.uint32) == g["m_bits"]
    assert np.float32(xv * m).view(np.uint32) == g["product_bits"]
    assert np.float32(xv / np.float32(amax / np.float32(448.0))) == 92.0
    tile = np.zeros((1, 1, 128, 64), np.float32)
    tile[0, 0, 0, 0] = amax
    tile[0, 0, 5, 7] = xv
    codes, scales = oracle_lib.quantize_e4m3_tiles(tile)
    assert codes[0, 0, 0, 0] == 448.0
    assert codes[0, 0, 5, 7] == g["code_rule_multiply"]
    assert codes[0, 0, 5, 7] != g["code_rule_divide"]
    assert scales[0, 0, 0] == np.float32(amax / np.float32(448.0))


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_forward_is_close_to_exact_attention(oracle_lib, causal):
    d = 64
    q, k, v, _ = _rand(31, 1, 2, 200, d)
    signs = fa_inputs.random_signs(4, d)
    o8, lse8, (qc, qs), (kc, ks) = oracle_lib.attention_fwd_fp8(q, k, v, signs, causal, _scale(d))
    o, lse = oracle_lib.attention_fwd(q, k, v, causal, _scale(d))
    # E4M3 keeps 3 mantissa bits, so each score moves by a few hundredths
    # (rows with few keys, early causal rows, show it most); rotating only one
    # of Q and K, or a wrong scale, moves O by about one (RMS > 0.1)
    assert np.max(np.abs(o8 - o)) < 0.25 and np.max(np.abs(lse8 - lse)) < 0.1
    assert np.sqrt(np.mean((o8 - o) ** 2)) < 0.02
    # and it is FP64 attention on exactly the dequantised rotated Q and K
    qd = qc * np.repeat(qs.astype(np.float64), 128, axis=2)[:, :, :200, None]
    kd = kc * np.repeat(ks.astype(np.float64), 128, axis=2)[:, :, :200, None]
    o2, lse2 = oracle_lib.attention_fwd(qd, kd, v, causal, _scale(d))
    assert np.array_equal(o2, o8) and np.array_equal(lse2, lse8)



# ---------------------------------------------------------------- a second implementation

@pytest.mark.parametrize("causal", [False, True])
def test_c_oracle_agrees_with_numpy_library_routines(oracle_lib, causal):
    """The C oracle against the definition evaluated with numpy's matmul, exp
    and max on whole matrices (a separate implementation: an indexing slip in
    the C loops shows up here)."""
    q, k, v, do = _rand(13, 2, 3, 70, 16)
    s = _scale(16)
    o, lse = oracle_lib.attention_fwd(q, k, v, causal, s)
    S = s * np.einsum("bhid,bhjd->bhij", q.astype(np.float64), k.astype(np.float64))
    if causal:
        S = np.where(np.tril(np.ones((70, 70), dtype=bool)), S, -np.inf)
    m = S.max(axis=-1, keepdims=True)
    E = np.exp(S - m)
    l = E.sum(axis=-1, keepdims=True)
    o_np = (E / l) @ v.astype(np.float64)
    lse_np = (m + np.log(l))[..., 0]
    assert np.max(np.abs(o - o_np)) <= 1e-12
    assert np.max(np.abs(lse - lse_np)) <= 1e-12
