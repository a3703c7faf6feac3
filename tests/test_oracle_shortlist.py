"""Pins of the shortlist oracle (oracle/shortlist.cpp): the small copy and the per-row score
bounds of a Q8_0 output head. Checked against things other than the oracle: Q8_0 and Q4_K
blocks decoded here with numpy from the byte layouts, the covering rules of the Q4_K copy
(half a step per weight, the min covering the most negative weight), the Cauchy-Schwarz
bound's tightness on the activation that attains it, a closed form for rows the small copy
represents exactly, and the property the method rests on (the true argmax always survives).
No GPU."""
import numpy as np
import pytest

from quantized_decode_gemv_block_gb300 import inputs

Q8_0, Q4_K = 1, 2


def np_q8_0(rows: np.ndarray, K: int) -> np.ndarray:
    """Q8_0 bytes (N x K/32*34) -> fp64 weights: fp16 d then 32 int8 codes per block."""
    b = rows.reshape(rows.shape[0], K // 32, 34)
    d = b[:, :, 0:2].copy().view(np.float16)[:, :, 0].astype(np.float64)
    q = b[:, :, 2:].copy().view(np.int8).astype(np.float64)
    return (d[:, :, None] * q).reshape(rows.shape[0], K)


def np_q4_k(rows: np.ndarray, K: int):
    """Q4_K bytes (N x K/256*144) -> (weights, step, low), step[n, g] = d * sc_g and
    low[n, g] = dmin * m_g for each 32-weight sub-block g. Layout: fp16 d, fp16 dmin, 12 bytes
    of 6-bit (sc, m) pairs (sub-blocks 0-3 in the low six bits of bytes 0-3 and 4-7; 4-7 in the
    nibbles of bytes 8-11 with their top two bits in the high bits of bytes 0-3 and 4-7), then
    128 bytes of codes: weight 64c + l is the low nibble of byte 32c + l, weight 64c + 32 + l
    its high nibble."""
    n = rows.shape[0]
    b = rows.reshape(n, K // 256, 144)
    d = b[:, :, 0:2].copy().view(np.float16)[:, :, 0].astype(np.float64)
    dmin = b[:, :, 2:4].copy().view(np.float16)[:, :, 0].astype(np.float64)
    s = b[:, :, 4:16].astype(np.int64)
    sc = np.zeros((n, K // 256, 8))
    m = np.zeros((n, K // 256, 8))
    for j in range(4):
        sc[:, :, j] = s[:, :, j] & 63
        m[:, :, j] = s[:, :, j + 4] & 63
        sc[:, :, j + 4] = (s[:, :, j + 8] & 15) | ((s[:, :, j] >> 6) << 4)
        m[:, :, j + 4] = (s[:, :, j + 8] >> 4) | ((s[:, :, j + 4] >> 6) << 4)
    qs = b[:, :, 16:].reshape(n, K // 256, 4, 32)
    q = np.stack([qs & 15, qs >> 4], axis=3).reshape(n, K // 256, 8, 32).astype(np.float64)
    step = d[:, :, None] * sc
    low = dmin[:, :, None] * m
    w = step[..., None] * q - low[..., None]
    return w.reshape(n, K), step.reshape(n, K // 32), low.reshape(n, K // 32)


def head(orc, N, K, seed=0):
    w = inputs.weights(N, K, seed=seed, tensor_id=900)
    return w, orc.quantize(Q8_0, w)


def test_small_copy_covers_every_weight_within_half_a_step(orc):
    N, K = 40, 512
    _, q8 = head(orc, N, K)
    small, _ = orc.shortlist_build(q8, N, K)
    w = np_q8_0(q8, K).reshape(N, K // 32, 32)
    wc, step, low = np_q4_k(small.reshape(N, -1), K)
    wc = wc.reshape(N, K // 32, 32)
    assert np.all(np.abs(w - wc) <= step[:, :, None] / 2 * (1 + 1e-12))
    assert np.all(low >= -np.minimum(0.0, w.min(axis=2)))  # the min reaches the lowest weight
    assert np.all(step > 0)


def test_bound_is_residual_norm_plus_rounding_allowance(orc):
    N, K = 64, 512
    _, q8 = head(orc, N, K, seed=1)
    small, bound = orc.shortlist_build(q8, N, K)
    w = np_q8_0(q8, K)
    wc, step, low = np_q4_k(small.reshape(N, -1), K)
    r = np.linalg.norm(w - wc, axis=1)
    A = np.sqrt(32.0 * ((15 * step + low) ** 2).sum(axis=1))
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
    ya, _ = orc.gemv(Q4_K, small, x, N, K)
    nx = np.linalg.norm(x.astype(np.float64), axis=1)
    assert np.all(np.abs(y8 - ya) <= B[None, :] * nx[:, None])
    w = np_q8_0(q8, K)
    wc, _, _ = np_q4_k(small.reshape(N, -1), K)
    for n in (0, 17, 47):
        e = w[n] - wc[n]
        xe = (e / np.linalg.norm(e)).astype(np.float32)[None, :]
        d8, _ = orc.gemv(Q8_0, q8, xe, N, K)
        da, _ = orc.gemv(Q4_K, small, xe, N, K)
        gap = abs(d8[0, n] - da[0, n])
        nxe = np.linalg.norm(xe.astype(np.float64))
        assert gap <= B[n] * nxe
        assert gap >= 0.9 * B[n] * nxe


def test_rows_the_copy_represents_exactly(orc):
    """Q8_0 codes 8k (k = i mod 16) with d = 63 * 2^-10, i.e. w = k * 63 * 2^-7: the Q4_K copy
    is exact (d = 2^-7, sc = 63, no min), so r_n = 0 and B_n is the rounding allowance alone,
    in closed form."""
    K = 512
    blk = np.frombuffer(np.float16(63 * 2.0 ** -10).tobytes() + bytes(8 * (i % 16) for i in range(32)), np.uint8)
    q8 = np.tile(blk, K // 32)[None, :]
    small, bound = orc.shortlist_build(q8, 1, K)
    wc, step, low = np_q4_k(small.reshape(1, -1), K)
    assert np.array_equal(wc[0], np_q8_0(q8, K)[0])
    assert np.all(step == 63 * 2.0 ** -7) and np.all(low == 0)
    wn = 63 * 2.0 ** -7 * np.sqrt(K / 16 * 1240.0)   # sum of k^2 over k = 0..15 is 1240
    A = np.sqrt(K) * 15 * 63 * 2.0 ** -7              # sqrt(32 * (K/32) * (15 d sc)^2)
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
        ya, _ = orc.gemv(Q4_K, small, x, N, K)
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
        orc.shortlist_build(np.zeros(68, np.uint8), 1, 64)
