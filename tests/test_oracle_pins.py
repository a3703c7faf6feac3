"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test names what fixes the expected value: a hand-derived closed form, an
independent library routine (numpy's fp16 conversion, numpy matmul, exact
rational arithmetic), a worked example in tests/golden, or an invariant of the
quantization scheme (the round-trip bound). No expected value here comes from
the CUDA path.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

from conftest import load_golden
from quantized_decode_gemv_block_gb300 import inputs

Q8_0, Q4_K, AFFINE4, Q5_K, Q6_K = 1, 2, 3, 4, 5


# ------------------------------------------------------------------- fp16 --
def test_fp16_decode_exhaustive(orc):
    """All 65536 binary16 codes decode exactly as numpy's float16 -> float64."""
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = codes.view(np.float16).astype(np.float64)
    got = np.array([orc.half_to_double(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros keep their sign
    assert math.copysign(1.0, orc.half_to_double(0x8000)) == -1.0


def test_fp16_round_trip_all_finite_codes(orc):
    for c in range(65536):
        if (c & 0x7C00) == 0x7C00 and (c & 0x3FF):
            continue  # NaN payloads are canonicalised
        assert orc.double_to_half_rn(orc.half_to_double(c)) == c


def test_fp16_rn_matches_numpy(orc):
    """Correct rounding from binary64, ties to even, checked against numpy's converter."""
    rng = np.random.default_rng(7)
    vals = list(rng.standard_normal(20000) * np.exp2(rng.uniform(-30, 17, 20000)))
    # exact midpoints between neighbouring fp16 values (ties) and points just off them
    for c in list(range(0, 0x7BFF, 97)) + [0, 1, 2, 0x3FF, 0x400, 0x401, 0x7BFE]:
        a, b = orc.half_to_double(c), orc.half_to_double(c + 1)
        mid = (a + b) / 2
        vals += [mid, np.nextafter(mid, 0), np.nextafter(mid, np.inf), -mid]
    vals += [65504.0, 65519.99, 65520.0, 65536.0, 1e300, -1e300, 2.0 ** -25, 2.0 ** -25 * 1.0000001,
             3 * 2.0 ** -26, 2.0 ** -26, 0.0, -0.0, float("inf"), float("-inf")]
    for v in vals:
        with np.errstate(over="ignore"):  # values past fp16's range round to inf, as intended
            ref = int(np.array([v], dtype=np.float64).astype(np.float16).view(np.uint16)[0])
        assert orc.double_to_half_rn(float(v)) == ref, v


def test_fp16_directed_rounding(orc):
    rng = np.random.default_rng(8)
    for v in list(rng.uniform(0, 2, 3000) * np.exp2(rng.uniform(-26, 14, 3000))):
        up, dn = orc.double_to_half_up(v), orc.double_to_half_down(v)
        vu, vd = orc.half_to_double(up), orc.half_to_double(dn)
        assert vd <= v <= vu
        assert vu - vd <= (orc.half_to_double(up + 1) - vu) * 1.0 + 1e-300 or vu == vd
        if vu != v:  # minimal: the code just below 'up' is already below v
            assert orc.half_to_double(up - 1) < v
        if vd != v and dn > 0:
            assert orc.half_to_double(dn + 1) > v


# ----------------------------------------------------------------- layout --
def test_block_sizes(orc):
    assert (orc.block_bytes(Q8_0), orc.block_weights(Q8_0)) == (34, 32)
    assert (orc.block_bytes(Q4_K), orc.block_weights(Q4_K)) == (144, 256)
    assert (orc.block_bytes(AFFINE4), orc.block_weights(AFFINE4)) == (20, 32)
    assert (orc.block_bytes(Q5_K), orc.block_weights(Q5_K)) == (176, 256)
    assert (orc.block_bytes(Q6_K), orc.block_weights(Q6_K)) == (210, 256)
    for K in (256, 2048, 2560, 9728):
        assert orc.row_bytes(Q5_K, K) == K * 11 // 16
        assert orc.row_bytes(Q6_K, K) == K * 105 // 128
        assert orc.row_bytes(Q8_0, K) == K * 17 // 16
        assert orc.row_bytes(Q4_K, K) == K * 9 // 16
        assert orc.row_bytes(AFFINE4, K) == K * 5 // 8


# --------------------------------------------------------- worked examples --
def test_q8_0_worked_example(orc):
    blk, f = load_golden("q8_0_e1.txt")
    assert len(blk) == 34
    w = orc.dequant(Q8_0, np.frombuffer(blk, np.uint8).reshape(1, 34), 1, 32)[0]
    assert np.array_equal(w, 0.5 * (np.arange(32) - 16.0))
    ones = np.ones((1, 32), np.float32)
    ramp = np.arange(32, dtype=np.float32)[None]
    y, ay = orc.gemv(Q8_0, np.frombuffer(blk, np.uint8).reshape(1, 34), ones, 1, 32)
    assert (y[0, 0], ay[0, 0]) == (-8.0, 128.0)
    y, ay = orc.gemv(Q8_0, np.frombuffer(blk, np.uint8).reshape(1, 34), ramp, 1, 32)
    assert (y[0, 0], ay[0, 0]) == (1240.0, 1920.0)


def test_q4_k_worked_example(orc):
    blk, f = load_golden("q4k_e2.txt")
    assert len(blk) == 144
    sc = [int(v) for v in f["sc"]]
    m = [int(v) for v in f["m"]]
    # the packed 6-bit scales decode to the stated (sc, m) for every sub-block
    for j in range(8):
        assert orc.unpack_scale_min(blk[4:16], j) == (sc[j], m[j])
    w = orc.dequant(Q4_K, np.frombuffer(blk, np.uint8).reshape(1, 144), 1, 256)[0]
    d, dmin = f["d"][0], f["dmin"][0]
    expect = np.array([d * sc[i // 32] * ((i + i // 32) % 16) - dmin * m[i // 32] for i in range(256)])
    assert np.array_equal(w, expect)
    assert (w[0], w[32], w[255]) == (0.0, -0.5, 377.5)
    b = np.frombuffer(blk, np.uint8).reshape(1, 144)
    y, ay = orc.gemv(Q4_K, b, np.ones((1, 256), np.float32), 1, 256)
    assert y[0, 0] == 240 * sum(sc) - 16 * sum(m) == 38480
    y, ay = orc.gemv(Q4_K, b, np.arange(256, dtype=np.float32)[None], 1, 256)
    assert (y[0, 0], ay[0, 0]) == (7768984.0, 7871992.0)


def _q5k_from_q4k(q4k_block: bytes, qh: bytes) -> bytes:
    """A Q5_K block with Q4_K's header (d, dmin, packed scales) and 4-bit codes plus the
    given 32 bytes of fifth bits: 16 header bytes, qh[32], then the 128 code bytes."""
    assert len(q4k_block) == 144 and len(qh) == 32
    return q4k_block[:16] + qh + q4k_block[16:]


def test_q5_k_reduces_to_q4_k_without_fifth_bits(orc):
    """With every fifth bit clear, Q5_K's w = d*sc*q - dmin*m is Q4_K's on the same bytes."""
    blk4, _ = load_golden("q4k_e2.txt")
    blk5 = _q5k_from_q4k(blk4, bytes(32))
    w4 = orc.dequant(Q4_K, np.frombuffer(blk4, np.uint8).reshape(1, 144), 1, 256)[0]
    w5 = orc.dequant(Q5_K, np.frombuffer(blk5, np.uint8).reshape(1, 176), 1, 256)[0]
    assert np.array_equal(w4, w5)


def test_q5_k_fifth_bit_positions(orc):
    """Hand-placed fifth bits. GGUF's Q5_K keeps the fifth bit of weight i in bit
    2c + h of qh[l], c = i // 64, h = 1 for the high-nibble half (i % 64 >= 32), l = i % 32:
    qh[0] bit 0 -> weight 0, qh[1] bit 1 -> weight 33, qh[2] bit 2 -> weight 66,
    qh[31] bit 7 -> weight 255. Exactly those weights gain 16*d*sc_j."""
    blk4, f = load_golden("q4k_e2.txt")
    d, sc = f["d"][0], [int(v) for v in f["sc"]]
    qh = bytearray(32)
    qh[0], qh[1], qh[2], qh[31] = 0x01, 0x02, 0x04, 0x80
    w4 = orc.dequant(Q4_K, np.frombuffer(blk4, np.uint8).reshape(1, 144), 1, 256)[0]
    w5 = orc.dequant(Q5_K, np.frombuffer(_q5k_from_q4k(blk4, bytes(qh)), np.uint8).reshape(1, 176), 1, 256)[0]
    diff = w5 - w4
    hit = {0, 33, 66, 255}
    for i in range(256):
        assert diff[i] == (16 * d * sc[i // 32] if i in hit else 0.0), i
    # every fifth bit set: every weight gains 16*d*sc_j; x = 1 then adds 16*32*d*sum(sc)
    w_all = orc.dequant(Q5_K, np.frombuffer(_q5k_from_q4k(blk4, bytes([0xFF] * 32)), np.uint8).reshape(1, 176),
                        1, 256)[0]
    assert np.array_equal(w_all - w4, np.array([16 * d * sc[i // 32] for i in range(256)]))
    b = np.frombuffer(_q5k_from_q4k(blk4, bytes([0xFF] * 32)), np.uint8).reshape(1, 176)
    y, _ = orc.gemv(Q5_K, b, np.ones((1, 256), np.float32), 1, 256)
    assert y[0, 0] == 38480 + 16 * 32 * d * sum(sc)  # Q4_K example's sum (tests/golden) + the fifth bits


def _q6k_block(ql=None, qh=None, scales=None, d_bits=0x3800):
    """Q6_K bytes: ql[128], qh[64], int8 scales[16], then fp16 d (0x3800 = 0.5) at byte 208."""
    ql = bytearray(128) if ql is None else ql
    qh = bytearray(64) if qh is None else qh
    sc = bytes((v & 0xFF) for v in (scales if scales is not None else range(16)))
    return bytes(ql) + bytes(qh) + sc + bytes([d_bits & 0xFF, d_bits >> 8])


def test_q6_k_zero_codes_and_signed_scales(orc):
    """All codes 0 (so q - 32 = -32) and scales[b] = b - 8 (negative ones included): weight i
    of sub-block b = i // 16 is d * (b - 8) * (-32) = -16 * (b - 8) with d = 0.5."""
    blk = _q6k_block(scales=[b - 8 for b in range(16)])
    w = orc.dequant(Q6_K, np.frombuffer(blk, np.uint8).reshape(1, 210), 1, 256)[0]
    assert np.array_equal(w, np.array([-16.0 * (i // 16 - 8) for i in range(256)]))


def test_q6_k_code_bit_positions(orc):
    """Hand-placed code bits. GGUF's Q6_K: weight 128n + 32k + l takes its low four bits from
    ql[64n + 32(k%2) + l] (low nibble for k < 2, high nibble otherwise) and its top two bits
    from bits 2k, 2k+1 of qh[32n + l]. So ql[0] = 0x0F sets weight 0 to 15 and ql[0] = 0xF0
    weight 64 to 15; ql[37] = 0x03 sets weight 37 (k = 1, l = 5) to 3; qh[39] = 0xC0 sets
    weight 231 (n = 1, k = 3, l = 7) to 48. Every other code stays 0."""
    ql, qh = bytearray(128), bytearray(64)
    ql[0] = 0xFF
    ql[37] = 0x03
    qh[39] = 0xC0
    scales = [1 + b for b in range(16)]
    blk = _q6k_block(ql, qh, scales)
    w = orc.dequant(Q6_K, np.frombuffer(blk, np.uint8).reshape(1, 210), 1, 256)[0]
    code = {0: 15, 64: 15, 37: 3, 231: 48}
    expect = np.array([0.5 * scales[i // 16] * (code.get(i, 0) - 32) for i in range(256)])
    assert np.array_equal(w, expect)


def test_affine4_nibble_order(orc):
    """Hand-built group: s = 2, b = -1, codes byte i = (2i mod 16) | ((2i+1 mod 16) << 4)."""
    blk = bytes([0x00, 0x40, 0x00, 0xBC]) + bytes(((2 * i) % 16) | ((((2 * i) + 1) % 16) << 4)
                                                 for i in range(16))
    w = orc.dequant(AFFINE4, np.frombuffer(blk, np.uint8).reshape(1, 20), 1, 32)[0]
    assert np.array_equal(w, 2.0 * (np.arange(32) % 16) - 1.0)


# --------------------------------------------------- quantizer invariants --
def _adversarial_blocks(bw, rng):
    rows = [
        np.zeros(bw), np.full(bw, 0.013), np.full(bw, -0.02), rng.uniform(0, 1, bw),
        -rng.uniform(0, 1, bw), np.where(np.arange(bw) == 5, 3.0, 1e-3 * rng.standard_normal(bw)),
        rng.standard_normal(bw) * 1e-7, rng.standard_normal(bw) * 60.0,
        np.where(np.arange(bw) % 32 == 0, -0.5, 0.0), np.linspace(-1, 1, bw),
    ]
    return np.stack(rows).astype(np.float32)


@pytest.mark.parametrize("fmt", [Q8_0, Q4_K, AFFINE4, Q5_K, Q6_K])
def test_round_trip_bound(orc, fmt):
    """|w - deq(q(w))| <= step/2 for every block (the quantizer's covering bound)."""
    bw, bb = orc.block_weights(fmt), orc.block_bytes(fmt)
    rng = np.random.default_rng(11)
    w = np.concatenate([inputs.weights(64, 512, seed=3, tensor_id=fmt).reshape(-1, bw),
                        _adversarial_blocks(bw, rng)]).astype(np.float32)
    nblk = w.shape[0]
    # one block per row so each row is one block
    blocks = orc.quantize(fmt, w)
    deq = orc.dequant(fmt, blocks, nblk, bw)
    err = np.abs(w.astype(np.float64) - deq)
    for r in range(nblk):
        b = blocks[r]
        if fmt == Q8_0:
            d = orc.half_to_double(int(b[0]) | (int(b[1]) << 8))
            amax = float(np.abs(w[r].astype(np.float64)).max())
            if d >= 2.0 ** -14:
                assert err[r].max() <= d / 2 * (1 + 1e-12)
            else:
                # fp16 d is subnormal or zero: relative rounding of d is coarse and the
                # +-127 clamp may bite, so only the covering bound of the clamp holds
                assert amax / 127 < 2.0 ** -14
                assert err[r].max() <= max(d / 2, amax - 127 * d) * (1 + 1e-12) + 1e-300
            q = b[2:].view(np.int8)
            assert q.min() >= -127
            assert d == float(np.float16(np.abs(w[r].astype(np.float64)).max() / 127))
        elif fmt in (Q4_K, Q5_K):
            d = orc.half_to_double(int(b[0]) | (int(b[1]) << 8))
            dmin = orc.half_to_double(int(b[2]) | (int(b[3]) << 8))
            for j in range(8):
                sc, m = orc.unpack_scale_min(bytes(b[4:16]), j)
                assert 0 <= sc <= 63 and 0 <= m <= 63
                seg = slice(32 * j, 32 * j + 32)
                assert err[r, seg].max() <= d * sc / 2 * (1 + 1e-12) + 1e-300
                # the min covers the most negative weight of the sub-block
                assert dmin * m >= -min(0.0, float(w[r, seg].min()))
        elif fmt == Q6_K:
            d = orc.half_to_double(int(b[208]) | (int(b[209]) << 8))
            for j in range(16):
                sc = int(np.int8(b[192 + j]))
                assert 0 <= sc <= 127
                seg = slice(16 * j, 16 * j + 16)
                assert err[r, seg].max() <= d * sc / 2 * (1 + 1e-12) + 1e-300
        else:
            s = orc.half_to_double(int(b[0]) | (int(b[1]) << 8))
            bias = orc.half_to_double(int(b[2]) | (int(b[3]) << 8))
            assert bias <= w[r].min()
            assert err[r].max() <= s / 2 * (1 + 1e-12) + 1e-300


def test_q8_0_codes_match_exact_rounding(orc):
    """Codes equal round-half-away-from-zero of the exact rational w/d (numpy fp16 for d)."""
    w = inputs.weights(16, 256, seed=5, tensor_id=2)
    blocks = orc.quantize(Q8_0, w).reshape(-1, 34)
    wb = w.reshape(-1, 32)
    for blk, ws in zip(blocks, wb):
        d = Fraction(orc.half_to_double(int(blk[0]) | (int(blk[1]) << 8)))
        for qi, wi in zip(blk[2:].view(np.int8), ws):
            r = Fraction(float(wi)) / d
            expect = int(math.floor(abs(r) + Fraction(1, 2))) * (1 if r >= 0 else -1)
            assert int(qi) == max(-127, min(127, expect))


# ------------------------------------------------------------------- gemv --
@pytest.mark.parametrize("fmt", [Q8_0, Q4_K, AFFINE4, Q5_K, Q6_K])
@pytest.mark.parametrize("K", [256, 512])
def test_gemv_brute_force(orc, fmt, K):
    """Oracle GEMV == numpy dense fp64 matmul of the dequantized matrix (other summation order)."""
    N, M = 8, 16
    w = inputs.weights(N, K, seed=1, tensor_id=K + fmt)
    blocks = orc.quantize(fmt, w)
    deq = orc.dequant(fmt, blocks, N, K)
    for xdt in ("f32", "bf16"):
        xf = inputs.activations_f32(M, K, seed=1, tensor_id=K)
        x = xf if xdt == "f32" else inputs.to_bf16_bits(xf)
        xv = xf.astype(np.float64) if xdt == "f32" else inputs.bf16_bits_to_f32(x).astype(np.float64)
        y, ay = orc.gemv(fmt, blocks, x, N, K)
        ref = xv @ deq.T
        aref = np.abs(xv) @ np.abs(deq).T
        assert np.all(np.abs(y - ref) <= 1e-12 * aref)
        assert np.allclose(ay, aref, rtol=1e-12, atol=0)


def test_gemv_exact_rational(orc):
    """fp64 oracle result is within K*eps*sum|w x| of the exact rational sum."""
    N, K, M = 3, 256, 2
    w = inputs.weights(N, K, seed=2, tensor_id=9)
    blocks = orc.quantize(Q4_K, w)
    deq = orc.dequant(Q4_K, blocks, N, K)
    x = inputs.activations_bf16(M, K, seed=2, tensor_id=10)
    xv = inputs.bf16_bits_to_f32(x)
    y, ay = orc.gemv(Q4_K, blocks, x, N, K)
    for j in range(M):
        for n in range(N):
            exact = sum(Fraction(float(deq[n, k])) * Fraction(float(xv[j, k])) for k in range(K))
            assert abs(Fraction(float(y[j, n])) - exact) <= Fraction(K * 2.0 ** -52) * Fraction(float(ay[j, n]))


def test_gemv_sampled_matches_full(orc):
    N, K, M = 40, 512, 5
    w = inputs.weights(N, K, seed=4, tensor_id=1)
    blocks = orc.quantize(Q4_K, w)
    x = inputs.activations_bf16(M, K, seed=4, tensor_id=2)
    y, ay = orc.gemv(Q4_K, blocks, x, N, K)
    js = np.array([0, 4, 2, 3, 1]); ns = np.array([0, 39, 17, 5, 22])
    ys, ays = orc.gemv_sampled(Q4_K, blocks, x, N, K, js, ns)
    assert np.array_equal(ys, y[js, ns]) and np.array_equal(ays, ay[js, ns])


def test_special_cases(orc):
    # zero scale -> zero output; NaN scale -> NaN only in that row
    K = 256
    w = inputs.weights(4, K, seed=6, tensor_id=3)
    blocks = orc.quantize(Q4_K, w)
    blocks[1, 0:2] = 0  # d = 0 and dmin = 0 in row 1's only super-block
    blocks[1, 2:4] = 0
    blocks[2, 0:2] = [0x00, 0x7E]  # d = NaN in row 2
    x = inputs.activations_bf16(3, K, seed=6, tensor_id=4)
    y, _ = orc.gemv(Q4_K, blocks, x, 4, K)
    assert np.all(y[:, 1] == 0.0)
    assert np.all(np.isnan(y[:, 2]))
    assert np.all(np.isfinite(y[:, [0, 3]]))
    # all codes equal, x = 1: y = n_blocks * 32 * d * q (Q8_0 closed form)
    blk = bytes([0x00, 0x34]) + bytes([7]) * 32  # d = 0.25, q = 7
    b = np.frombuffer(blk * 4, np.uint8).reshape(1, 136)
    y, _ = orc.gemv(Q8_0, b, np.ones((1, 128), np.float32), 1, 128)
    assert y[0, 0] == 4 * 32 * 0.25 * 7
