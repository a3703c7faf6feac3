"""Pins for the decode-step oracle (oracle/decode.cpp), on the CPU.

bf16 rounding against torch's converter; RMSNorm against its closed form; the step against
cases that reduce to pinned pieces (zero layers, zero layer weights); and the composition's
indexing (q/k/v split, GQA mapping, gate/up split) against a numpy restatement on tiny
shapes built from the oracle's own dequantized matrices.
"""
import numpy as np
import pytest
import torch

from quantized_decode_gemv_block_gb300 import inputs

Q4_K, Q8_0 = 2, 1


def test_bf16_rounding_matches_torch(orc):
    rng = np.random.default_rng(3)
    vals = list((rng.standard_normal(20000) * np.exp2(rng.uniform(-140, 120, 20000))).astype(np.float32))
    bits = np.arange(0, 0x7F7F, 37, dtype=np.uint32)
    for b in bits:  # midpoints between neighbouring bf16 values and their neighbours
        lo = np.array([b << 16], dtype=np.uint32).view(np.float32)[0]
        hi = np.array([(b + 1) << 16], dtype=np.uint32).view(np.float32)[0]
        mid = np.float32((np.float64(lo) + np.float64(hi)) / 2)
        vals += [mid, np.nextafter(mid, np.float32(0)), np.nextafter(mid, np.float32(np.inf)), -mid]
    vals += [np.float32(0.0), np.float32(-0.0), np.float32(3.4e38), np.float32(1e-40), np.float32(-1e-44)]
    v32 = np.array(vals, dtype=np.float32)
    ref = torch.from_numpy(v32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.double_to_bf16_rn(float(v)) for v in v32], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_rounding_of_arrays_matches_torch(orc):
    """The array form rounds exactly like the scalar one, which torch's converter pins above
    (the same midpoints, their neighbours, signed zeros, the top of the range)."""
    rng = np.random.default_rng(4)
    bits = np.arange(0, 0x7F7F, 53, dtype=np.uint32)
    lo = (bits << 16).view(np.float32).astype(np.float64)
    hi = ((bits + 1) << 16).view(np.float32).astype(np.float64)
    mid = ((lo + hi) / 2).astype(np.float32)
    vals = np.concatenate([mid, np.nextafter(mid, np.float32(0)), np.nextafter(mid, np.float32(np.inf)), -mid,
                           (rng.standard_normal(5000) * np.exp2(rng.uniform(-130, 120, 5000))).astype(np.float32),
                           np.array([0.0, -0.0, 3.39e38, 1e-41], np.float32)])
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = orc.bf16_rn(vals.astype(np.float64).reshape(2, -1)).reshape(-1)
    assert np.array_equal(got, ref)


def test_swiglu_closed_forms(orc):
    """silu(0) * u = 0; silu(g) = g once exp(-g) vanishes against 1 (g = 40), so act = bf16(g u)
    (a swap of gate and up gives silu(1.5) * 40 = 49.1 there instead of 60); silu of a very
    negative gate is -0; and random rows equal the formula in numpy fp64 rounded by the pinned
    scalar rounding."""
    gu = np.array([[0.0, 40.0, -800.0, 5.0, 1.5, 3.0]], dtype=np.float64)  # g = [0, 40, -800], u = [5, 1.5, 3]
    act = orc.swiglu_bf16(gu)
    assert act[0, 0] == 0x0000
    assert act[0, 1] == orc.double_to_bf16_rn(60.0) == 0x4270
    assert act[0, 2] == 0x8000
    rng = np.random.default_rng(8)
    gu = rng.standard_normal((3, 2 * 96)) * 3.0
    g, u = gu[:, :96], gu[:, 96:]
    expect = np.vectorize(orc.double_to_bf16_rn, otypes=[np.uint16])(g / (1.0 + np.exp(-g)) * u)
    assert np.array_equal(orc.swiglu_bf16(gu), expect)


def test_rmsnorm_closed_form(orc):
    eps = 1e-6
    h = np.array([[2.0] * 256, [-0.5] * 256], dtype=np.float64)
    out = orc.rmsnorm_bf16(h, eps)
    for r, c in enumerate([2.0, -0.5]):
        expect = orc.double_to_bf16_rn(c / np.sqrt(c * c + eps))
        assert np.all(out[r] == expect)
    # scale invariance (for eps = 0): rmsnorm(s*h) == rmsnorm(h) for powers of two s
    hr = np.random.default_rng(1).standard_normal((3, 512))
    assert np.array_equal(orc.rmsnorm_bf16(hr, 0.0), orc.rmsnorm_bf16(hr * 8.0, 0.0))


TINY = dict(n_layers=2, hidden=256, q_dim=256, kv_dim=128, head_dim=64, ffn=512, vocab=300,
            layer_fmt=Q4_K, head_fmt=Q8_0, eps=1e-6)


def tiny_model(orc, d, seed=0, zero_layers=False):
    h, q, kv, f = d["hidden"], d["q_dim"], d["kv_dim"], d["ffn"]
    shapes = [(q + 2 * kv, h), (h, q), (2 * f, h), (h, f)]
    layers, tid = [], 0
    for _ in range(d["n_layers"]):
        lay = []
        for N, K in shapes:
            w = inputs.weights(N, K, seed=seed, tensor_id=tid)
            if zero_layers:
                w[:] = 0
            lay.append(orc.quantize(d["layer_fmt"], w))
            tid += 1
        layers.append(tuple(lay))
    head = orc.quantize(d["head_fmt"], inputs.weights(d["vocab"], h, seed=seed, tensor_id=tid))
    return layers, head


def test_decode_without_layer_work_reduces_to_norm_and_head(orc):
    x = inputs.activations_bf16(3, TINY["hidden"], seed=5)
    layers, head = tiny_model(orc, TINY, zero_layers=True)
    got = orc.decode_step(TINY, layers, head, x)
    xn = orc.rmsnorm_bf16(inputs.bf16_bits_to_f32(x).astype(np.float64), TINY["eps"])
    ref, _ = orc.gemv(Q8_0, head, xn, TINY["vocab"], TINY["hidden"])
    assert np.array_equal(got, ref)
    d0 = dict(TINY, n_layers=0)
    assert np.array_equal(orc.decode_step(d0, [], head, x), ref)


def test_decode_composition_against_numpy_restatement(orc):
    d = TINY
    layers, head = tiny_model(orc, d, seed=2)
    x = inputs.activations_bf16(2, d["hidden"], seed=6)
    got = orc.decode_step(d, layers, head, x)
    H, Q, KV, F, hd = d["hidden"], d["q_dim"], d["kv_dim"], d["ffn"], d["head_dim"]
    group = (Q // hd) // (KV // hd)

    def bf(a):
        return inputs.bf16_bits_to_f32(np.vectorize(orc.double_to_bf16_rn, otypes=[np.uint16])(a)).astype(np.float64)

    def norm(h):
        return h / np.sqrt((h * h).mean(axis=1, keepdims=True) + d["eps"])

    h = inputs.bf16_bits_to_f32(x).astype(np.float64)
    for (wqkv, wo, wgu, wd) in layers:
        Wqkv = orc.dequant(Q4_K, wqkv, Q + 2 * KV, H)
        Wo, Wgu, Wd = orc.dequant(Q4_K, wo, H, Q), orc.dequant(Q4_K, wgu, 2 * F, H), orc.dequant(Q4_K, wd, H, F)
        qkv = bf(norm(h)) @ Wqkv.T
        v = qkv[:, Q + KV:]
        oin = np.concatenate([v[:, (hq // group) * hd:(hq // group + 1) * hd] for hq in range(Q // hd)], axis=1)
        h = h + bf(oin) @ Wo.T
        gu = bf(norm(h)) @ Wgu.T
        g, u = gu[:, :F], gu[:, F:]
        h = h + bf(g / (1 + np.exp(-g)) * u) @ Wd.T
    ref = bf(norm(h)) @ orc.dequant(Q8_0, head, d["vocab"], H).T
    # numpy sums in another order: allow a few ulps, and the rare bf16 tie flip upstream
    err = np.abs(got - ref) / (np.abs(ref).max() + 1e-30)
    assert np.quantile(err, 0.99) < 1e-9 and err.max() < 1e-2


def test_attention_step_with_self_only_visibility_is_the_stand_in(orc):
    """With no cached context and each token seeing only itself, attention over the cache is
    the stand-in (softmax weight 1 on the token's own value): identical fp64 logits."""
    layers, head = tiny_model(orc, TINY, seed=4)
    M = 3
    x = inputs.activations_bf16(M, TINY["hidden"], seed=5)
    ref = orc.decode_step(TINY, layers, head, x)
    empty = [np.zeros((0, TINY["kv_dim"]), np.uint16)] * TINY["n_layers"]
    got = orc.decode_step_attn(TINY, layers, head, empty, empty, 0, x, 0.125,
                               mask=np.array([1 << i for i in range(M)], np.uint32))
    assert np.array_equal(got, ref)
    # one token, causal: the same
    got1 = orc.decode_step_attn(TINY, layers, head, empty, empty, 0, x[:1], 0.125)
    assert np.array_equal(got1, ref[:1])


def test_attention_step_depends_on_the_cache_and_the_window(orc):
    layers, head = tiny_model(orc, TINY, seed=6)
    M, L = 4, 9
    x = inputs.activations_bf16(M, TINY["hidden"], seed=7)
    rng = np.random.default_rng(8)
    kc = [(rng.standard_normal((L, TINY["kv_dim"])).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
          for _ in range(TINY["n_layers"])]
    vc = [(rng.standard_normal((L, TINY["kv_dim"])).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
          for _ in range(TINY["n_layers"])]
    a = orc.decode_step_attn(TINY, layers, head, kc, vc, L, x, 0.125)
    # causal: token 0 alone and token 0 inside the window agree; later tokens see the earlier ones
    a0 = orc.decode_step_attn(TINY, layers, head, kc, vc, L, x[:1], 0.125)
    assert np.array_equal(a0[0], a[0])
    b = orc.decode_step_attn(TINY, layers, head, kc, vc, L, x[[0, 2, 1, 3]], 0.125)
    assert np.array_equal(b[0], a[0]) and not np.allclose(b[3], a[3])
    # the cached values matter
    vc2 = [v.copy() for v in vc]
    vc2[0][3] ^= 0x0100
    c = orc.decode_step_attn(TINY, layers, head, kc, vc2, L, x, 0.125)
    assert not np.array_equal(c, a)
