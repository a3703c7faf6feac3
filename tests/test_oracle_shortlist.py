"""Pins of the shortlist oracle (oracle/shortlist.cpp): the small copy and the per-row score
bounds of a Q8_0 output head. Checked against things other than the oracle: Q8_0 and affine4
blocks decoded here with numpy from the byte layouts, the extremal rules that define the
affine4 scale and bias, the Cauchy-Schwarz bound's tightness on the activation that attains
it, a closed form for rows the small copy represents exactly, and the property the method
rests on (the true argmax always survives). No GPU."""
import numpy as np
import pytest

from quantized_decode_gemv_block_gb300 import inputs

Q8_0, AFFINE4 = 1, 3


def np_q8_0(rows: np.ndarray, K: int) -> np.ndarray:
    """Q8_0 bytes (N x K/32*34) -> fp64 weights: fp16 d then 32 int8 codes per block."""
    b = rows.reshape(rows.shape[0], K // 32, 34)
    d = b[:, :, 0:2].copy().view(np.float16)[:, :, 0].astype(np.float64)
    q = b[:, :, 2:].copy().view(np.int8).astype(np.float64)
    return (d[:, :, None] * q).reshape(rows.shape[0], K)


def np_affine4(rows: np.ndarray, K: int):
    """affine4 bytes -> (weights, s, b): fp16 s, fp16 b, 16 code bytes, low nibble first."""
    b = rows.reshape(rows.shape[0], K // 32, 20)
    s = b[:, :, 0:2].copy().view(np.float16)[:, :, 0].astype(np.float64)
    bias = b[:, :, 2:4].copy().view(np.float16)[:, :, 0].astype(np.float64)
    codes = b[:, :, 4:]
    q = np.stack([codes & 15, codes >> 4], axis=-1).reshape(rows.shape[0], K // 32, 32).astype(np.float64)
    return (s[:, :, None] * q + bias[:, :, None]).reshape(rows.shape[0], K), s, bias


def head(orc, N, K, seed=0):
    w = inputs.weights(N, K, seed=seed, tensor_id=900)
    return w, orc.quantize(Q8_0, w)


def test_small_copy_scale_and_bias_are_the_extremal_fp16_values(orc):
    N, K = 40, 256
    _, q8 = head(orc, N, K)
    small, _ = orc.shortlist_build(q8, N, K)
    w = np_q8_0(q8, K).reshape(N, K // 32, 32)
    wa, s, b = np_affine4(small.reshape(N, -1), K)
    wa = wa.reshape(N, K // 32, 32)
    mn, mx = w.min(axis=2), w.max(axis=2)
    s16, b16 = s.astype(np.float16), b.astype(np.float16)
    # b: the largest fp16 <= min w;  s: the smallest fp16 >= (max w - b) / 15
    assert np.all(b <= mn)
    assert np.all(np.nextafter(b16, np.float16(np.inf)).astype(np.float64) > mn)
    assert np.all(s >= (mx - b) / 15)
    assert np.all(np.nextafter(s16, np.float16(-np.inf)).astype(np.float64) < (mx - b) / 15)
    # every weight within half a step of its copy
    assert np.all(np.abs(w - wa) <= s[:, :, None] / 2 * (1 + 1e-12))


def test_bound_is_residual_norm_plus_rounding_allowance(orc):
    N, K = 64, 512
    _, q8 = head(orc, N, K, seed=1)
    small, bound = orc.shortlist_build(q8, N, K)
    w = np_q8_0(q8, K)
    wa, s, b = np_affine4(small.reshape(N, -1), K)
    r = np.linalg.norm(w - wa, axis=1)
    A = np.sqrt(32.0 * ((np.abs(b) + 15 * s) ** 2).sum(axis=1))
    want = r + K * 2.0 ** -22 * (np.linalg.norm(w, axis=1) + A)
    assert np.all(bound.astype(np.float64) >= want)
    assert np.all(bound.astype(np.float64) <= want * (1 + 2.0 ** -22))
    # with the N(0, 0.02) rows of a head the residual dominates: a few per cent of allowance
    assert np.all(want < 1.1 * r)


def test_bound_holds_and_is_attained(orc):
    """|y(W) - y(W')| <= B_n ||x|| for random x; for x along w_n - w'_n the residual part of the
    bound is attained (Cauchy-Schwarz with equality), so B_n is within the allowance of tight."""
    N, K = 48, 1024
    _, q8 = head(orc, N, K, seed=2)
    small, bound = orc.shortlist_build(q8, N, K)
    B = bound.astype(np.float64)
    x = inputs.activations_f32(6, K, seed=3)
    y8, _ = orc.gemv(Q8_0, q8, x, N, K)
    ya, _ = orc.gemv(AFFINE4, small, x, N, K)
    nx = np.linalg.norm(x.astype(np.float64), axis=1)
    assert np.all(np.abs(y8 - ya) <= B[None, :] * nx[:, None])
    w = np_q8_0(q8, K)
    wa, _, _ = np_affine4(small.reshape(N, -1), K)
    for n in (0, 17, 47):
        e = w[n] - wa[n]
        xe = (e / np.linalg.norm(e)).astype(np.float32)[None, :]
        d8, _ = orc.gemv(Q8_0, q8, xe, N, K)
        da, _ = orc.gemv(AFFINE4, small, xe, N, K)
        gap = abs(d8[0, n] - da[0, n])
        nxe = np.linalg.norm(xe.astype(np.float64))
        assert gap <= B[n] * nxe
        assert gap >= 0.9 * B[n] * nxe


def test_rows_the_copy_represents_exactly(orc):
    """Codes v = (i mod 16) - 8 with d = 1/2: the copy is exact (s = 1/2, b = -4), so r_n = 0
    and B_n is the rounding allowance alone, in closed form."""
    K = 256
    blk = np.frombuffer(np.float16(0.5).tobytes() + bytes(np.int8((i % 16) - 8).view(np.uint8)
                                                          for i in range(32)), np.uint8)
    q8 = np.tile(blk, K // 32)[None, :]
    small, bound = orc.shortlist_build(q8, 1, K)
    sb = small.reshape(K // 32, 20)
    assert np.all(sb[:, 0:2].copy().view(np.float16)[:, 0] == np.float16(0.5))
    assert np.all(sb[:, 2:4].copy().view(np.float16)[:, 0] == np.float16(-4.0))
    assert np.all(sb[:, 4:] == np.array([(2 * i) % 16 | (((2 * i + 1) % 16) << 4) for i in range(16)], np.uint8))
    wn = 0.5 * np.sqrt(K / 16 * 344.0)        # sum of v^2 over v = -8..7 is 344
    A = np.sqrt(K) * (4.0 + 15 * 0.5)         # sqrt(32 * (K/32) * (|b| + 15 s)^2)
    want = K * 2.0 ** -22 * (wn + A)
    assert want <= float(bound[0]) <= want * (1 + 2.0 ** -22)


def test_the_argmax_always_survives(orc):
    """The row with the largest exact score is never pruned; with a hidden state that favours
    one row (a confident next token) almost every other row is pruned."""
    N, K = 3000, 512
    w, q8 = head(orc, N, K, seed=4)
    small, bound = orc.shortlist_build(q8, N, K)
    B = bound.astype(np.float64)
    targets = [7, 1500, 2999]
    x_peak = inputs.to_bf16_bits(inputs.planted_activations_f32(w[targets], 0.5, seed=5))
    x_flat = inputs.activations_bf16(3, K, seed=6)
    for x, peaked in ((x_peak, True), (x_flat, False)):
        y8, _ = orc.gemv(Q8_0, q8, x, N, K)
        ya, _ = orc.gemv(AFFINE4, small, x, N, K)
        nx = np.linalg.norm(inputs.bf16_bits_to_f32(x).astype(np.float64), axis=1)
        for j in range(x.shape[0]):
            U = B * nx[j]
            cand = ya[j] + U >= (ya[j] - U).max()
            best = int(np.argmax(y8[j]))
            assert cand[best]
            if peaked:
                assert best == targets[j]
                assert cand.sum() <= 3
            else:
                assert cand.sum() > 10  # no favourite: many rows stay in play


def test_rejects_bad_K(orc):
    with pytest.raises(ValueError):
        orc.shortlist_build(np.zeros(34, np.uint8), 1, 48)
