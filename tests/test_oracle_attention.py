"""Pins of the decode-attention oracle (oracle/attention.cpp) against closed forms and
invariants that hold whatever order it sums in: a one-position softmax, uniform scores,
two-position softmaxes written out, the causal and tree visibility rules, the grouping of
query heads onto kv heads, the bf16 rounding of q, and invariance under permuting the cached
positions. No GPU."""
import math

import numpy as np
import pytest

import oracle as orc


def bf16(a):
    """fp32 -> bf16 bits by truncation (the test inputs below are chosen bf16-exact)."""
    return (np.asarray(a, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def f32(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def rand_bf16(rng, shape, scale=1.0):
    return bf16(rng.standard_normal(shape).astype(np.float32) * np.float32(scale))


def test_single_visible_position_returns_its_value():
    rng = np.random.default_rng(0)
    hd, nq, nkv = 16, 4, 2
    q = rng.standard_normal((1, nq * hd)).astype(np.float32)
    k = rand_bf16(rng, (1, nkv * hd))
    v = rand_bf16(rng, (1, nkv * hd))
    o, base = orc.attention(q, k, v, 0, nq, nkv, hd, 0.125)
    vv = f32(v)[0]
    for hq in range(nq):
        kvh = hq // 2
        assert np.array_equal(o[0, hq * hd:(hq + 1) * hd], vv[kvh * hd:(kvh + 1) * hd])
        assert np.array_equal(base[0, hq * hd:(hq + 1) * hd], np.abs(vv[kvh * hd:(kvh + 1) * hd]))


def test_uniform_scores_give_the_mean_of_the_visible_values():
    rng = np.random.default_rng(1)
    hd, nq, nkv, L, M = 8, 2, 1, 5, 4
    q = np.zeros((M, nq * hd), np.float32)
    k = rand_bf16(rng, (L + M, nkv * hd))
    v = rand_bf16(rng, (L + M, nkv * hd))
    o, _ = orc.attention(q, k, v, L, nq, nkv, hd, 1.0)
    vv = f32(v)
    for i in range(M):  # causal: cached 0..L-1 and window 0..i
        want = vv[:L + i + 1].mean(axis=0)
        for hq in range(nq):
            np.testing.assert_allclose(o[i, hq * hd:(hq + 1) * hd], want, rtol=1e-14, atol=1e-15)


def two_point(sa, v0, v1):
    """softmax over scores (sa, 0) applied to (v0, v1)."""
    e = math.exp(sa)
    return (e * v0 + v1) / (e + 1.0)


def test_two_positions_closed_form():
    hd, scale = 2, 0.75
    a = 1.5  # bf16-exact
    q = np.array([[a, 0.0]], np.float32)
    k = bf16([[1.0, 0.0], [0.0, 0.0]])  # cached position 0, window position 0
    v = bf16([[2.0, -1.0], [-3.0, 0.5]])
    o, base = orc.attention(q, k, v, 1, 1, 1, hd, scale)
    for d, (v0, v1) in enumerate([(2.0, -3.0), (-1.0, 0.5)]):
        assert o[0, d] == pytest.approx(two_point(scale * a, v0, v1), rel=1e-15, abs=1e-15)
        assert base[0, d] == pytest.approx(two_point(scale * a, abs(v0), abs(v1)), rel=1e-15)


def test_q_is_rounded_to_bf16_nearest_even():
    hd, scale = 2, 1.0
    k = bf16([[1.0, 0.0], [0.0, 0.0]])
    v = bf16([[1.0, 0.0], [0.0, 0.0]])
    # 1 + 2^-8 is a tie between bf16 1.0 and 1 + 2^-7: rounds to the even 1.0;
    # 1 + 3 * 2^-9 rounds up to 1 + 2^-7
    for qv, eff in ((1.0 + 2.0 ** -8, 1.0), (1.0 + 3 * 2.0 ** -9, 1.0 + 2.0 ** -7)):
        o, _ = orc.attention(np.array([[qv, 0.0]], np.float32), k, v, 1, 1, 1, hd, scale)
        assert o[0, 0] == pytest.approx(two_point(scale * eff, 1.0, 0.0), rel=1e-15)


def test_causal_window_ignores_later_guesses():
    rng = np.random.default_rng(2)
    hd, nq, nkv, L, M = 16, 4, 2, 7, 6
    q = rng.standard_normal((M, nq * hd)).astype(np.float32)
    k = rand_bf16(rng, (L + M, nkv * hd))
    v = rand_bf16(rng, (L + M, nkv * hd))
    o, _ = orc.attention(q, k, v, L, nq, nkv, hd, 0.25)
    for j in range(M):  # perturb window position j: tokens i < j unchanged, i >= j change
        v2 = v.copy()
        v2[L + j] = rand_bf16(rng, (nkv * hd,))
        o2, _ = orc.attention(q, k, v2, L, nq, nkv, hd, 0.25)
        for i in range(M):
            same = np.array_equal(o2[i], o[i])
            assert same == (i < j), (i, j)


def test_tree_mask_two_point_closed_form_and_empty_rows():
    hd, M = 2, 4
    a, scale = 2.0, 0.5
    q = np.tile(np.array([[a, 0.0]], np.float32), (M, 1))
    # window position 0 has key (1, 0); the others key 0: token i sees {0, i}
    k = bf16([[1.0, 0.0]] + [[0.0, 0.0]] * (M - 1))
    vals = [4.0, -2.0, 0.5, 8.0]
    v = bf16([[x, 0.0] for x in vals])
    mask = np.array([1 | (1 << i) for i in range(M)], np.uint32)
    o, _ = orc.attention(q, k, v, 0, 1, 1, hd, scale, mask=mask)
    assert o[0, 0] == vals[0]
    for i in range(1, M):
        assert o[i, 0] == pytest.approx(two_point(scale * a, vals[0], vals[i]), rel=1e-15)
    # a token that sees nothing outputs zeros
    o, base = orc.attention(q, k, v, 0, 1, 1, hd, scale, mask=np.array([0, 1, 3, 0], np.uint32))
    assert np.all(o[0] == 0) and np.all(o[3] == 0) and np.all(base[0] == 0)
    assert o[1, 0] == vals[0]


def test_grouped_heads_read_their_kv_head():
    rng = np.random.default_rng(3)
    hd, nq, nkv, L, M = 8, 4, 2, 6, 2
    q1 = rng.standard_normal((M, hd)).astype(np.float32)
    q = np.tile(q1, (1, nq))  # every query head asks the same question
    k1 = rand_bf16(rng, (L + M, hd))
    v1 = rand_bf16(rng, (L + M, hd), 0.5)
    k = np.concatenate([k1, k1], axis=1)  # kv heads 0 and 1: same keys
    v = np.concatenate([v1, bf16(f32(v1) * 2.0)], axis=1)  # kv head 1: values doubled (exact)
    o, _ = orc.attention(q, k, v, L, nq, nkv, hd, 0.3)
    for i in range(M):
        h0 = o[i, 0:hd]
        assert np.array_equal(o[i, hd:2 * hd], h0)  # heads 0, 1: kv head 0
        np.testing.assert_allclose(o[i, 2 * hd:3 * hd], 2.0 * h0, rtol=1e-14, atol=1e-15)
        assert np.array_equal(o[i, 3 * hd:4 * hd], o[i, 2 * hd:3 * hd])


def test_permuting_cached_positions_changes_nothing():
    rng = np.random.default_rng(4)
    hd, nq, nkv, L, M = 16, 2, 1, 33, 3
    q = rng.standard_normal((M, nq * hd)).astype(np.float32)
    k = rand_bf16(rng, (L + M, nkv * hd))
    v = rand_bf16(rng, (L + M, nkv * hd))
    o, _ = orc.attention(q, k, v, L, nq, nkv, hd, 0.2)
    perm = np.concatenate([rng.permutation(L), np.arange(L, L + M)])
    o2, _ = orc.attention(q, k[perm], v[perm], L, nq, nkv, hd, 0.2)
    np.testing.assert_allclose(o2, o, rtol=1e-13, atol=1e-14)


def test_rejects_bad_arguments():
    q = np.zeros((1, 8), np.float32)
    kv = np.zeros((1, 8), np.uint16)
    with pytest.raises(ValueError):
        orc.attention(q, kv, kv, 0, 3, 2, 4, 1.0)  # 3 query heads over 2 kv heads
    with pytest.raises(ValueError):
        orc.attention(np.zeros((33, 8), np.float32), np.zeros((33, 8), np.uint16),
                      np.zeros((33, 8), np.uint16), 0, 1, 1, 8, 1.0)  # window longer than 32


def test_window_token_equals_the_token_decoded_alone():
    """Token i of a causal window over L cached positions sees the same positions, in the same
    order, as the token alone over L + i cached positions (the window's earlier rows cached):
    the same fp64 result (the pages' rule that checking guesses gives plain decoding's output)."""
    rng = np.random.default_rng(6)
    hd, nq, nkv, L, M = 16, 4, 2, 9, 5
    q = rng.standard_normal((M, nq * hd)).astype(np.float32)
    k = rand_bf16(rng, (L + M, nkv * hd))
    v = rand_bf16(rng, (L + M, nkv * hd))
    o, base = orc.attention(q, k, v, L, nq, nkv, hd, 0.3)
    for i in range(M):
        oi, bi = orc.attention(q[i:i + 1], k[:L + i + 1], v[:L + i + 1], L + i, nq, nkv, hd, 0.3)
        assert np.array_equal(oi[0], o[i]) and np.array_equal(bi[0], base[i]), i
