"""GPU decode attention (kq_attention) against the fp64 oracle, and its batch invariance.

Tolerance: |o - o_ref| <= 1e-4 * sum_p w_p |v_p| per element (the contract's scale: the
softmax-weighted magnitude of what is summed). The kernel's products of bf16 values are exact
in fp32, the softmax weights enter the second product as bf16 hi + lo pairs (2^-16
relative), so its error is fp32 rounding of the scores (a few 1e-7 relative, amplified by
|score| through exp) and of the sums.
"""
import numpy as np
import pytest
import torch

import quantized_decode_gemv_block_gb300 as kq
from quantized_decode_gemv_block_gb300 import inputs

pytestmark = pytest.mark.gpu
TOL = 1e-4


@pytest.fixture(scope="module")
def built():
    from quantized_decode_gemv_block_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def make(M, L, n_q, n_kv, hd, seed):
    q = inputs.activations_f32(M, n_q * hd, seed=seed, tensor_id=7000)
    k = inputs.activations_bf16(L + M, n_kv * hd, seed=seed, tensor_id=7001)
    v = inputs.activations_bf16(L + M, n_kv * hd, seed=seed, tensor_id=7002)
    return q, k, v


def dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def run(q, k, v, L, n_q, n_kv, hd, scale, mask=None):
    md = torch.from_numpy(mask.view(np.int32)).cuda() if mask is not None else None
    o = kq.attention(torch.from_numpy(q).cuda(), dev_bf16(k), dev_bf16(v), L, n_q, n_kv, hd, scale, mask=md)
    torch.cuda.synchronize()
    return o.cpu().numpy()


def check(o, ref, base, what):
    err = np.abs(o.astype(np.float64) - ref)
    bad = err > TOL * base
    assert not bad.any(), f"{what}: {bad.sum()} outside; worst {(err / np.maximum(base, 1e-300)).max():.3g}"


# (M, L, n_q, n_kv, head_dim): one token and no context; a partial chunk; exactly one chunk;
# one past a chunk; head_dim 64; 128 query rows (4 heads x 32 tokens); many chunks; no GQA;
# 94 chunks (the combine's groups then go past its prefetched chunks into both later loops)
SHAPES = [(1, 0, 16, 4, 128), (1, 1, 16, 4, 128), (4, 63, 16, 4, 128), (8, 64, 16, 4, 128),
          (16, 65, 8, 2, 64), (32, 200, 8, 2, 128), (5, 1000, 16, 4, 128), (32, 4096, 4, 4, 128),
          (3, 12000, 16, 4, 128)]


@pytest.mark.parametrize("M,L,n_q,n_kv,hd", SHAPES)
def test_attention_matches_oracle(built, orc, M, L, n_q, n_kv, hd):
    q, k, v = make(M, L, n_q, n_kv, hd, seed=M + L)
    scale = float(np.float32(1.0 / np.sqrt(hd)))
    o = run(q, k, v, L, n_q, n_kv, hd, scale)
    ref, base = orc.attention(q, k, v, L, n_q, n_kv, hd, scale)
    check(o, ref, base, f"attention M={M} L={L} {n_q}/{n_kv} hd={hd}")
    assert kq.device_errors() == 0


def test_tree_mask_and_tokens_that_see_nothing(built, orc):
    M, L, n_q, n_kv, hd = 12, 100, 16, 4, 128
    q, k, v = make(M, L, n_q, n_kv, hd, seed=3)
    rng = np.random.default_rng(5)
    mask = np.array([(int(rng.integers(0, 1 << 12)) | (1 << i)) & ((2 << i) - 1) for i in range(M)], np.uint32)
    o = run(q, k, v, L, n_q, n_kv, hd, 0.09, mask)
    ref, base = orc.attention(q, k, v, L, n_q, n_kv, hd, 0.09, mask=mask)
    check(o, ref, base, "tree mask")
    # no context and an empty mask row: zeros
    mask0 = np.array([0] + [1 << i for i in range(1, 4)], np.uint32)
    q4, k4, v4 = make(4, 0, 4, 2, 64, seed=9)
    o = run(q4, k4, v4, 0, 4, 2, 64, 0.125, mask0)
    assert np.all(o[0] == 0.0)
    ref, base = orc.attention(q4, k4, v4, 0, 4, 2, 64, 0.125, mask=mask0)
    check(o, ref, base, "empty row")


def test_a_tokens_output_is_the_same_for_every_window_size(built):
    """Bit equality across window sizes, including across the kernel's two work splits (warps
    over positions for up to 3 row blocks of 16 query rows, warps over row blocks from 4 on:
    M <= 12 and M >= 13 here, with 4 query rows per token)."""
    L, n_q, n_kv, hd = 777, 16, 4, 128
    q, k, v = make(32, L, n_q, n_kv, hd, seed=11)
    full = run(q[:32], k[:L + 32], v[:L + 32], L, n_q, n_kv, hd, 0.0883)
    for M in (1, 3, 5, 8, 12, 13, 20, 24):
        o = run(q[:M], k[:L + M], v[:L + M], L, n_q, n_kv, hd, 0.0883)
        assert np.array_equal(o.view(np.uint32), full[:M].view(np.uint32)), f"M={M}"


@pytest.mark.parametrize("M,L,hd", [(8, 300, 128), (5, 125, 64), (3, 0, 128), (4, 128, 128), (3, 12000, 128)])
def test_window_equals_one_token_at_a_time(built, M, L, hd):
    """Token i of a window over L cached positions equals token i alone over L + i cached
    positions (the window's earlier rows now part of the cache), bit for bit."""
    n_q, n_kv = 16, 4
    q, k, v = make(M, L, n_q, n_kv, hd, seed=M + L + hd)
    win = run(q, k, v, L, n_q, n_kv, hd, 0.0883)
    for i in range(M):
        o = run(q[i:i + 1], k[:L + i + 1], v[:L + i + 1], L + i, n_q, n_kv, hd, 0.0883)
        assert np.array_equal(o.view(np.uint32), win[i:i + 1].view(np.uint32)), f"token {i}"


def test_extreme_finite_values_in_a_later_guess_leave_earlier_tokens_unchanged(built):
    """A later guess's key and value rows at the largest finite bf16 magnitude (0x7F7F, about
    3.39e38) enter the chunk's products with weight 0 for the earlier tokens: those tokens keep
    the bits they get decoded alone. (Non-finite keys or values are outside the guarantee, as
    the header states: 0 * Inf is NaN.)"""
    M, L, n_q, n_kv, hd = 4, 130, 16, 4, 128
    q, k, v = make(M, L, n_q, n_kv, hd, seed=21)
    k = k.copy()
    v = v.copy()
    k[L + 3, ::2] = 0x7F7F   # +max finite bf16 in half of the last guess's key
    v[L + 3, ::3] = 0xFF7F   # -max finite bf16 in a third of its value
    win = run(q, k, v, L, n_q, n_kv, hd, 0.0883)
    assert np.all(np.isfinite(win[:3]))
    for i in range(3):
        o = run(q[i:i + 1], k[:L + i + 1], v[:L + i + 1], L + i, n_q, n_kv, hd, 0.0883)
        assert np.array_equal(o.view(np.uint32), win[i:i + 1].view(np.uint32)), f"token {i}"
