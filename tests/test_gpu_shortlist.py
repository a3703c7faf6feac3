"""GPU shortlist output head (kq_shortlist_build, kq_head_argmax) against the oracle.

The small copy's bytes must equal the oracle's exactly (byte work); its bounds may differ
from the oracle's by one fp32 ulp (both evaluate fp64 sums, in different orders, and round
up) and must not lie below the bound computed here from the decoded arrays. The greedy token
must be the same with the shortlist as with every row scored exactly (bit-identical token and
score), the same for every M, and valid against the fp64 oracle: its oracle score within the
tolerance of the largest oracle score, its exact score within 1e-4 * sum |w x| of the oracle's.
"""
import numpy as np
import pytest
import torch

import quantized_decode_gemv_block_gb300 as kq
from quantized_decode_gemv_block_gb300 import inputs
from test_oracle_shortlist import np_q4_k, np_q8_0

pytestmark = pytest.mark.gpu
Q8_0 = 1
TOL = 1e-4


@pytest.fixture(scope="module")
def built():
    from quantized_decode_gemv_block_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def cuda_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def x_device(x_f32, dtype):
    if dtype == "bf16":
        return inputs.to_bf16_bits(x_f32), cuda_bf16(inputs.to_bf16_bits(x_f32))
    return x_f32, torch.from_numpy(x_f32).cuda()


def run_both(w_dev, sl, xd, N, K):
    t1, s1, r1 = kq.head_argmax(w_dev, sl, xd, N, K)
    t0, s0, r0 = kq.head_argmax(w_dev, None, xd, N, K, all_rows=True)
    torch.cuda.synchronize()
    assert kq.device_errors() == 0
    t1, s1, t0, s0 = t1.cpu().numpy(), s1.cpu().numpy(), t0.cpu().numpy(), s0.cpu().numpy()
    assert np.array_equal(t1, t0), (t1, t0)
    assert np.array_equal(s1.view(np.uint32), s0.view(np.uint32))
    assert int(r0.item()) == N
    return t1, s1, int(r1.item())


def check_against_oracle(orc, q8, x_host, N, K, tok, sc):
    y, ay = orc.gemv(Q8_0, q8, x_host, N, K)
    for j in range(len(tok)):
        t = int(tok[j])
        tol = TOL * ay[j]
        assert abs(float(sc[j]) - y[j, t]) <= tol[t], (j, t)
        assert y[j, t] >= y[j].max() - tol[t] - tol[int(np.argmax(y[j]))], (j, t, int(np.argmax(y[j])))


@pytest.mark.parametrize("N,K", [(3000, 512), (777, 2048), (1, 256), (33, 256)])
def test_small_copy_matches_the_oracle(built, orc, N, K):
    w = inputs.weights(N, K, seed=N, tensor_id=900)
    q8 = orc.quantize(Q8_0, w)
    buf = kq.shortlist_build(torch.from_numpy(q8).cuda(), N, K)
    small, bound = kq.shortlist_parts(buf, N, K)
    small, bound = small.cpu().numpy(), bound.cpu().numpy()
    osmall, obound = orc.shortlist_build(q8, N, K)
    assert np.array_equal(small.reshape(-1), osmall)
    ulp = np.spacing(obound)
    assert np.all(np.abs(bound.astype(np.float64) - obound) <= ulp)
    wq = np_q8_0(q8, K)
    wc, step, low = np_q4_k(osmall.reshape(N, -1), K)
    want = np.linalg.norm(wq - wc, axis=1) + K * 2.0 ** -22 * (
        np.linalg.norm(wq, axis=1) + np.sqrt(32.0 * ((15 * step + low) ** 2).sum(axis=1)))
    assert np.all(bound.astype(np.float64) >= want)


@pytest.mark.parametrize("M,dtype", [(1, "bf16"), (4, "bf16"), (16, "bf16"), (3, "f32")])
def test_planted_tokens(built, orc, M, dtype):
    N, K = 5000, 512
    w = inputs.weights(N, K, seed=7, tensor_id=900)
    q8 = orc.quantize(Q8_0, w)
    w_dev = torch.from_numpy(q8).cuda()
    sl = kq.shortlist_build(w_dev, N, K)
    targets = np.random.default_rng(M).choice(N, M, replace=False)
    xh, xd = x_device(inputs.planted_activations_f32(w[targets], 0.5, seed=M), dtype)
    tok, sc, scored = run_both(w_dev, sl, xd, N, K)
    assert np.array_equal(tok, targets)
    assert scored <= 3 * M  # the shortlist prunes nearly every row
    check_against_oracle(orc, q8, xh, N, K, tok, sc)


def test_unpeaked_activations_fall_back_to_many_exact_rows(built, orc):
    N, K = 4000, 512
    w = inputs.weights(N, K, seed=8, tensor_id=900)
    q8 = orc.quantize(Q8_0, w)
    w_dev = torch.from_numpy(q8).cuda()
    sl = kq.shortlist_build(w_dev, N, K)
    xh = inputs.activations_bf16(5, K, seed=9)
    tok, sc, scored = run_both(w_dev, sl, cuda_bf16(xh), N, K)
    assert scored > 50
    check_against_oracle(orc, q8, xh, N, K, tok, sc)


def test_every_row_keeps_its_token_for_every_m(built, orc):
    N, K = 2500, 1024
    w = inputs.weights(N, K, seed=10, tensor_id=900)
    q8 = orc.quantize(Q8_0, w)
    w_dev = torch.from_numpy(q8).cuda()
    sl = kq.shortlist_build(w_dev, N, K)
    targets = np.arange(16) * 150 + 3
    x = inputs.planted_activations_f32(w[targets], 0.35, seed=11)
    x[::3] = inputs.activations_f32(6, K, seed=12)  # a third of the rows without a favourite
    xd = cuda_bf16(inputs.to_bf16_bits(x))
    t16, s16, _ = kq.head_argmax(w_dev, sl, xd, N, K)
    t16, s16 = t16.cpu().numpy(), s16.cpu().numpy()
    for M in (1, 2, 5, 8):
        for r0 in (0, 16 - M):
            t, s, _ = kq.head_argmax(w_dev, sl, xd[r0:r0 + M].contiguous(), N, K)
            assert np.array_equal(t.cpu().numpy(), t16[r0:r0 + M])
            assert np.array_equal(s.cpu().numpy().view(np.uint32), s16[r0:r0 + M].view(np.uint32))


def test_ties_go_to_the_lowest_row(built, orc):
    N, K = 300, 256
    w = inputs.weights(N, K, seed=13, tensor_id=900)
    w[40] = w[200]  # identical rows: identical exact scores
    w[41] = w[200]
    q8 = orc.quantize(Q8_0, w)
    w_dev = torch.from_numpy(q8).cuda()
    sl = kq.shortlist_build(w_dev, N, K)
    xh, xd = x_device(inputs.planted_activations_f32(w[[200, 200]], 0.5, seed=14), "bf16")
    tok, sc, _ = run_both(w_dev, sl, xd, N, K)
    assert list(tok) == [40, 40]


@pytest.mark.parametrize("M", [1, 8])
def test_full_size_head(built, orc, M):
    """Q8_0 head 151936 x 2048 (the decode step's output layer), hidden states favouring
    one row each: the tokens, the shortlist against every row scored, and the oracle's
    full scores of the head."""
    N, K = 151936, 2048
    wf = inputs.weights_cuda(N, K, seed=0, tensor_id=901)
    w_dev = kq.quantize("q8_0", wf)
    targets = torch.tensor(np.random.default_rng(M).choice(N, M, replace=False), device="cuda")
    xd = inputs.planted_activations_cuda(wf[targets], 0.5, seed=M)
    del wf
    sl = kq.shortlist_build(w_dev, N, K)
    tok, sc, scored = run_both(w_dev, sl, xd, N, K)
    assert np.array_equal(tok, targets.cpu().numpy())
    assert scored <= 3 * M
    xh = xd.view(torch.int16).cpu().numpy().view(np.uint16)
    check_against_oracle(orc, w_dev.cpu().numpy(), xh, N, K, tok, sc)


def test_activations_too_large_for_shared_memory_give_the_same_bits(built, orc):
    """M = 16 fp32 rows of K = 3072 (192 KB) are read from global memory, one row (12 KB) from
    shared memory: the exact scores are the same instructions, so the same bits."""
    N, K = 1200, 3072
    w = inputs.weights(N, K, seed=15, tensor_id=900)
    q8 = orc.quantize(Q8_0, w)
    w_dev = torch.from_numpy(q8).cuda()
    sl = kq.shortlist_build(w_dev, N, K)
    targets = np.arange(16) * 70 + 1
    x = inputs.planted_activations_f32(w[targets], 0.5, seed=16)
    xd = torch.from_numpy(x).cuda()
    t16, s16, _ = run_both(w_dev, sl, xd, N, K)
    assert np.array_equal(t16, targets)
    for j in (0, 7, 15):
        t, s, _ = kq.head_argmax(w_dev, sl, xd[j:j + 1].contiguous(), N, K)
        assert int(t.item()) == int(t16[j])
        assert np.array_equal(s.cpu().numpy().view(np.uint32), s16[j:j + 1].view(np.uint32))
    check_against_oracle(orc, q8, x, N, K, t16, s16)


@pytest.mark.parametrize("N,M", [(2047, 3), (1, 2), (5, 1), (1025, 16)])
def test_ragged_and_tiny_heads(built, orc, N, M):
    """N not a multiple of 4 (the exact pass's scalar row loads) or of the 1024-row chunks,
    a one-row head (its only row wins), a head smaller than one warp's rows."""
    K = 512
    w = inputs.weights(N, K, seed=N + 17, tensor_id=900)
    q8 = orc.quantize(Q8_0, w)
    w_dev = torch.from_numpy(q8).cuda()
    sl = kq.shortlist_build(w_dev, N, K)
    targets = np.random.default_rng(N).integers(0, N, M)
    xh, xd = x_device(inputs.planted_activations_f32(w[targets], 0.5, seed=N), "bf16")
    tok, sc, scored = run_both(w_dev, sl, xd, N, K)
    if N == 1:
        assert list(tok) == [0] * M
    else:
        assert np.array_equal(tok, targets)
    check_against_oracle(orc, q8, xh, N, K, tok, sc)


def test_nan_scores_never_win(built, orc):
    """A row whose Q8_0 scale is NaN scores NaN: it is never the token, with or without the
    shortlist; hidden states that are NaN give no comparable score at all: token -1."""
    N, K, M = 600, 256, 2
    w = inputs.weights(N, K, seed=21, tensor_id=900)
    q8 = orc.quantize(Q8_0, w)
    q8[123, 0:2] = np.frombuffer(np.float16(np.nan).tobytes(), np.uint8)  # d of block 0 = NaN
    w_dev = torch.from_numpy(q8).cuda()
    sl = kq.shortlist_build(w_dev, N, K)
    xh, xd = x_device(inputs.planted_activations_f32(w[[123, 400]], 0.5, seed=22), "bf16")
    tok, sc, _ = run_both(w_dev, sl, xd, N, K)
    y, _ = orc.gemv(Q8_0, q8, xh, N, K)
    assert np.isnan(y[:, 123]).all()
    assert tok[1] == 400 and tok[0] != 123
    assert tok[0] == int(np.nanargmax(y[0]))
    xn = xd.clone()
    xn[0, 5] = float("nan")
    tok, sc, _ = run_both(w_dev, sl, xn, N, K)
    assert tok[0] == -1 and np.isnan(sc[0])
    assert tok[1] == 400
