"""GPU parity of kq_gemm against the fp64 oracle: the tensor-core prefill product (Q4_K x
bf16, M > 32) and the 16-row GEMV passes (16 < M <= 32, and every M > 16 of the other pairs).

Tolerance (the contract of the method): |y_gpu - y_ref| <= 1e-4 * sum_k |w_k x_k| per
output element. The prefill path forms only exact products (X as fp16 under an exact
per-token power of two; weights as the integers sc*q with d applied in fp32 per
super-block; the min term through fp16 hi/lo splits good to 2^-22), so its error is fp32
summation alone: a CPU model of the same arithmetic with exact sums lands near 1e-8 of
sum |w x|. Beyond the contract the tests ask for a median below 1e-6, which fp16-rounded
weights (median about 1e-5 on these data) could not reach.
"""
import numpy as np
import pytest
import torch

from quantized_decode_gemv_block_gb300 import inputs

pytestmark = pytest.mark.gpu

Q4_K = 2
TOL = 1e-4


@pytest.fixture(scope="module")
def kq():
    from quantized_decode_gemv_block_gb300 import build
    build.build()
    import quantized_decode_gemv_block_gb300 as m
    assert torch.cuda.is_available()
    return m


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bf16(x_bits):
    return dev(x_bits.view(np.int16)).view(torch.bfloat16)


def assert_close(y, yref, ay, what=""):
    err = np.abs(y - yref)
    bad = err > TOL * ay
    rel = err / np.maximum(ay, 1e-300)
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside 1e-4*sum|wx|; worst ratio "
                           f"{rel.max():.3g}")
    assert np.median(rel) < 1e-6, f"{what}: median error {np.median(rel):.3g} of sum|wx|"


def run_gemm(kq, blocks, x_bits, N, K):
    y = kq.gemm("q4_k", dev(blocks), bf16(x_bits), N, K)
    torch.cuda.synchronize()
    return y.cpu().numpy().astype(np.float64)


# (M, N, K) of the tensor-core route (M > 32): one tile; ragged M (tails of 33, 72, 1 and 16
# tokens); ragged N (tails of 8 and 232 rows of a 256-row pair tile, where rank 1 of the pair
# has no rows); several K super-blocks; N % 4 != 0 (rows not 16-byte aligned); more pair tiles
# (80) than co-resident pairs, so some pairs take a second tile.
SHAPES = [(33, 256, 256), (200, 520, 1024), (129, 300, 512), (257, 1000, 2560), (384, 2048, 768),
          (130, 258, 512), (784, 5120, 256)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_gemm_matches_oracle(kq, orc, M, N, K):
    w = inputs.weights(N, K, seed=M + N, tensor_id=Q4_K)
    blocks = orc.quantize(Q4_K, w)
    x = inputs.activations_bf16(M, K, seed=M, tensor_id=3000)
    y = run_gemm(kq, blocks, x, N, K)
    yref, ay = orc.gemv(Q4_K, blocks, x, N, K)
    assert_close(y, yref, ay, f"gemm {M}x{N}x{K}")
    assert kq.device_errors() == 0


def test_gemm_rows_of_any_magnitude(kq, orc):
    """Per-token scaling: rows scaled by 2^-60 .. 2^60, a zero row and a row with one nonzero."""
    M, N, K = 40, 512, 1024
    blocks = orc.quantize(Q4_K, inputs.weights(N, K, seed=5, tensor_id=Q4_K))
    xf = inputs.activations_f32(M, K, seed=6, tensor_id=3001)
    for j in range(M):
        xf[j] *= np.float32(2.0 ** (3 * (j - 20)))
    xf[7] = 0.0
    xf[9] = 0.0
    xf[9, 300] = 1.5
    x = inputs.to_bf16_bits(xf)
    y = run_gemm(kq, blocks, x, N, K)
    yref, ay = orc.gemv(Q4_K, blocks, x, N, K)
    assert np.all(y[7] == 0.0)
    live = np.ones(M, bool)
    live[7] = False
    assert_close(y[live], yref[live], ay[live], "scaled rows")


def test_gemm_is_deterministic_and_small_m_is_gemv(kq, orc):
    M, N, K = 300, 768, 1536
    blocks = orc.quantize(Q4_K, inputs.weights(N, K, seed=8, tensor_id=Q4_K))
    wd = dev(blocks)
    x = bf16(inputs.activations_bf16(M, K, seed=9, tensor_id=3002))
    a = kq.gemm("q4_k", wd, x, N, K)
    b = kq.gemm("q4_k", wd, x, N, K)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    # M <= 16 goes to the GEMV kernels: same bits as kq_gemv
    g = kq.gemm("q4_k", wd, x[:16], N, K)
    v = kq.gemv("q4_k", wd, x[:16], N, K)
    torch.cuda.synchronize()
    assert torch.equal(g.view(torch.int32), v.view(torch.int32))


def test_gemm_errors(kq):
    M, N, K = 64, 256, 512
    w = torch.zeros((N, 144 * K // 256), dtype=torch.uint8, device="cuda")
    x = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    need = kq.gemm_workspace_size("q4_k", torch.bfloat16, M, N, K)
    assert need >= M * K * 2 + M * 4
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(kq.KQError) as e:
        kq.gemm("q4_k", w, x, N, K, y=y, workspace=small)
    assert e.value.code == kq.KQ_ERR_WORKSPACE
    big = torch.empty(need + 512, dtype=torch.uint8, device="cuda")
    with pytest.raises(kq.KQError) as e:
        kq.gemm("q4_k", w, x, N, K, y=y, workspace=big[16:])  # not 256-byte aligned
    assert e.value.code == kq.KQ_ERR_WORKSPACE
    assert kq.gemm_workspace_size("q8_0", torch.bfloat16, M, N, K) == 0  # GEMV passes
    assert kq.gemm_workspace_size("q4_k", torch.bfloat16, 16, N, K) == 0
    assert kq.gemm_workspace_size("q4_k", torch.bfloat16, 32, N, K) == 0  # GEMV passes
    assert kq.gemm_workspace_size("q4_k", torch.bfloat16, 33, N, K) > 0   # tensor cores


def test_full_prefill_9728x2560_m2048(kq, orc):
    """Q4_K W 9728 x 2560 times X 2048 x 2560 bf16: sampled outputs, every tile corner included."""
    M, N, K = 2048, 9728, 2560
    blocks = orc.quantize(Q4_K, inputs.weights(N, K, seed=0, tensor_id=Q4_K))
    x = inputs.activations_bf16(M, K, seed=0, tensor_id=3003)
    y = kq.gemm("q4_k", dev(blocks), bf16(x), N, K)
    torch.cuda.synchronize()
    y = y.cpu().numpy()
    rng = np.random.default_rng(0)
    js = list(rng.integers(0, M, 3000))
    ns = list(rng.integers(0, N, 3000))
    for mt in range(0, M, 128):  # corners of every 128 x 256 output tile along the diagonal band
        for nt in range(0, N, 256 * 5):
            for dj, dn in ((0, 0), (127, 255), (0, 255), (127, 0)):
                js.append(min(M - 1, mt + dj))
                ns.append(min(N - 1, nt + dn))
    js, ns = np.array(js), np.array(ns)
    yref, ay = orc.gemv_sampled(Q4_K, blocks, x, N, K, js, ns)
    got = y[js, ns].astype(np.float64)
    assert_close(got, yref, ay, "prefill 2048x9728x2560")
    assert kq.device_errors() == 0


def _gemv_rows_equal(kq, fmt, wd, x, y, N, K):
    """Every row of y has the bits kq_gemv gives that row alone (M = 1)."""
    for j in range(x.shape[0]):
        r = kq.gemv(fmt, wd, x[j:j + 1].contiguous(), N, K)
        torch.cuda.synchronize()
        assert torch.equal(r.view(torch.int32)[0], y.view(torch.int32)[j]), f"{fmt} row {j}"


@pytest.mark.parametrize("M", [17, 24, 32])
def test_batched_verify_up_to_32_rows_is_gemv_bitwise(kq, orc, M):
    """16 < M <= 32 (Q4_K, bf16): 16-row GEMV passes; each row keeps its M = 1 bits."""
    N, K = 600, 1024  # ragged row tiles, four super-blocks
    blocks = orc.quantize(Q4_K, inputs.weights(N, K, seed=M, tensor_id=Q4_K))
    x_bits = inputs.activations_bf16(M, K, seed=M, tensor_id=3004)
    wd, x = dev(blocks), bf16(x_bits)
    assert kq.gemm_workspace_size("q4_k", torch.bfloat16, M, N, K) == 0
    y = kq.gemm("q4_k", wd, x, N, K)
    torch.cuda.synchronize()
    yref, ay = orc.gemv(Q4_K, blocks, x_bits, N, K)
    err = np.abs(y.cpu().numpy().astype(np.float64) - yref)
    assert np.all(err <= TOL * ay), f"worst ratio {(err / ay).max():.3g}"
    _gemv_rows_equal(kq, "q4_k", wd, x, y, N, K)
    assert kq.device_errors() == 0


@pytest.mark.parametrize("fmt,code,dtype,M", [("q8_0", 1, "f32", 20), ("q5_k", 4, "bf16", 40),
                                              ("affine4", 3, "bf16", 18), ("q6_k", 5, "bf16", 33)])
def test_gemm_passes_for_pairs_without_tensor_core_product(kq, orc, fmt, code, dtype, M):
    """M > 16 for every other format / dtype pair: 16-row GEMV passes, within the contract
    against the oracle and bit-identical, row by row, to kq_gemv."""
    N, K = 300, 512
    blocks = orc.quantize(code, inputs.weights(N, K, seed=M + code, tensor_id=code))
    if dtype == "f32":
        xh = inputs.activations_f32(M, K, seed=M, tensor_id=3005)
        x = dev(xh)
    else:
        xh = inputs.activations_bf16(M, K, seed=M, tensor_id=3005)
        x = bf16(xh)
    wd = dev(blocks)
    y = kq.gemm(fmt, wd, x, N, K)
    torch.cuda.synchronize()
    yref, ay = orc.gemv(code, blocks, xh, N, K)
    err = np.abs(y.cpu().numpy().astype(np.float64) - yref)
    assert np.all(err <= TOL * ay), f"{fmt}: worst ratio {(err / ay).max():.3g}"
    _gemv_rows_equal(kq, fmt, wd, x, y, N, K)
    assert kq.device_errors() == 0
