"""GPU parity of kq_gemv / kq_quantize against the fp64 oracle, and batch invariance.

Tolerance (the contract of the method): |y_gpu - y_ref| <= 1e-4 * sum_k |w_k x_k| per
output element, y_ref and the sum from the oracle on the same inputs. Quantizer bytes
and batch-invariance are bit-exact.
"""
import numpy as np
import pytest
import torch

from quantized_decode_gemv_block_gb300 import inputs

pytestmark = pytest.mark.gpu

FMTS = {"q8_0": 1, "q4_k": 2, "affine4": 3, "q5_k": 4, "q6_k": 5}
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


def x_tensor(x_np, dtype):
    if dtype == "bf16":
        return dev(x_np.view(np.int16)).view(torch.bfloat16)
    return dev(x_np)


def make_x(M, K, dtype, seed, tid=1000):
    xf = inputs.activations_f32(M, K, seed=seed, tensor_id=tid)
    return xf if dtype == "f32" else inputs.to_bf16_bits(xf)


def run_gemv(kq, fmt, blocks_np, x_np, dtype, N, K):
    y = kq.gemv(fmt, dev(blocks_np), x_tensor(x_np, dtype), N, K)
    torch.cuda.synchronize()
    return y.cpu().numpy().astype(np.float64)


def assert_close(y, yref, ay, what=""):
    err = np.abs(y - yref)
    bad = err > TOL * ay
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside 1e-4*sum|wx|; worst ratio "
                           f"{(err / np.maximum(ay, 1e-300)).max():.3g}")


# ------------------------------------------------------------- quantizer --
@pytest.mark.parametrize("fmt", list(FMTS))
def test_quantizer_bytes_match_oracle(kq, orc, fmt):
    f = FMTS[fmt]
    N, K = 96, 1024
    w = inputs.weights(N, K, seed=21, tensor_id=f)
    w[3, :256] = 0.0                       # all-zero block(s)
    w[4, :256] = 0.013                     # constant, positive
    w[5, :256] = -0.02                     # constant, negative
    w[6, 5] = 3.0                          # outlier
    w[7, :] *= 1e-6                        # tiny values (subnormal fp16 scales)
    w[8, :] *= 1e3                         # large values
    ref = orc.quantize(f, w)
    got = kq.quantize(fmt, dev(w))
    torch.cuda.synchronize()
    got = got.cpu().numpy()
    assert got.shape == ref.shape
    diff = np.argwhere(got != ref)
    assert diff.size == 0, f"{len(diff)} bytes differ, first at {diff[:4].tolist()}"


# ------------------------------------------------------------------ gemv --
SHAPES = [(1, 256), (37, 512), (300, 2560), (1000, 1024), (129, 4096), (700, 3072), (90, 20736)]


@pytest.mark.parametrize("fmt", list(FMTS))
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("N,K", SHAPES)
def test_gemv_matches_oracle(kq, orc, fmt, dtype, N, K):
    f = FMTS[fmt]
    w = inputs.weights(N, K, seed=N + K, tensor_id=f)
    blocks = orc.quantize(f, w)
    for M in (1, 3, 8, 13, 16):
        x = make_x(M, K, dtype, seed=M + 7 * N)
        yref, ay = orc.gemv(f, blocks, x, N, K)
        y = run_gemv(kq, fmt, blocks, x, dtype, N, K)
        assert_close(y, yref, ay, f"{fmt} {dtype} N={N} K={K} M={M}")


@pytest.mark.parametrize("fmt", list(FMTS))
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_batch_invariance(kq, orc, fmt, dtype):
    """Row j's bits are the same for every M in 1..16 and every slot position."""
    f = FMTS[fmt]
    N, K = 700, 3072
    blocks = orc.quantize(f, inputs.weights(N, K, seed=3, tensor_id=f))
    x16 = make_x(16, K, dtype, seed=99)
    wd = dev(blocks)
    full = kq.gemv(fmt, wd, x_tensor(x16, dtype), N, K).cpu().numpy()
    for M in range(1, 17):
        y = kq.gemv(fmt, wd, x_tensor(x16[:M].copy(), dtype), N, K).cpu().numpy()
        assert np.array_equal(y.view(np.uint32), full[:M].view(np.uint32)), f"M={M}"
    rng = np.random.default_rng(5)
    for M in (2, 7, 9, 16):
        perm = rng.permutation(16)[:M]
        y = kq.gemv(fmt, wd, x_tensor(x16[perm].copy(), dtype), N, K).cpu().numpy()
        assert np.array_equal(y.view(np.uint32), full[perm].view(np.uint32)), f"perm M={M}"


def test_k_zero_writes_zeros_and_empty_is_noop(kq):
    y = torch.full((3, 5), 7.0, device="cuda")
    w = torch.zeros(16, dtype=torch.uint8, device="cuda")
    x = torch.zeros((3, 16), dtype=torch.bfloat16, device="cuda")
    kq.gemv("q4_k", w, x, 5, 0, y=y)
    torch.cuda.synchronize()
    assert torch.all(y == 0)
    y2 = torch.full((0, 5), 7.0, device="cuda")
    kq.gemv("q4_k", w, x[:0], 5, 256, y=y2)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_guard_bands_untouched(kq, orc, dtype):
    """Y is written only inside M x N: a canary around it survives."""
    N, K, M = 77, 512, 5
    blocks = orc.quantize(2, inputs.weights(N, K, seed=8, tensor_id=2))
    x = make_x(M, K, dtype, seed=8)
    pad = 1024
    buf = torch.full((pad + M * N + pad,), 12345.0, device="cuda")
    y = buf[pad:pad + M * N].view(M, N)
    kq.gemv("q4_k", dev(blocks), x_tensor(x, dtype), N, K, y=y)
    torch.cuda.synchronize()
    b = buf.cpu().numpy()
    assert np.all(b[:pad] == 12345.0) and np.all(b[pad + M * N:] == 12345.0)
    yref, ay = orc.gemv(2, blocks, x, N, K)
    assert_close(y.cpu().numpy().astype(np.float64), yref, ay)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_nan_scale_stays_in_its_row(kq, orc, dtype):
    N, K, M = 40, 512, 3
    blocks = orc.quantize(2, inputs.weights(N, K, seed=9, tensor_id=2))
    blocks[11, 0:2] = [0x00, 0x7E]  # d = NaN in row 11's first super-block
    x = make_x(M, K, dtype, seed=9)
    y = run_gemv(kq, "q4_k", blocks, x, dtype, N, K)
    assert np.all(np.isnan(y[:, 11]))
    others = np.delete(y, 11, axis=1)
    assert np.all(np.isfinite(others))
    yref, ay = orc.gemv(2, blocks, x, N, K)
    assert_close(np.delete(y, 11, axis=1), np.delete(yref, 11, axis=1), np.delete(ay, 11, axis=1))


def test_no_device_errors_recorded(kq):
    assert kq.device_errors() == 0


def test_errors_reported(kq):
    w = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    x = torch.zeros((17, 256), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(kq.KQError) as e:
        kq.gemv("q4_k", w, x, 4, 256)
    assert e.value.code == kq.KQ_ERR_ARG


# ------------------------------------------------------ full-size workloads --
def sampled_check(kq, orc, f, fmt, N, K, Ms, dtype, seed, nsamp=1500):
    w = inputs.weights(N, K, seed=seed, tensor_id=f)
    blocks = orc.quantize(f, w)
    wd = dev(blocks)
    rng = np.random.default_rng(seed)
    ys = {}
    for M in Ms:
        x = make_x(M, K, dtype, seed=seed, tid=2000)  # rows of smaller M are a prefix of larger M
        y = kq.gemv(fmt, wd, x_tensor(x, dtype), N, K)
        torch.cuda.synchronize()
        y = y.cpu().numpy()
        js = rng.integers(0, M, nsamp)
        ns = rng.integers(0, N, nsamp)
        ns[:4] = [0, N - 1, N // 2, 1]
        yref, ay = orc.gemv_sampled(f, blocks, x, N, K, js, ns)
        assert_close(y[js, ns].astype(np.float64), yref, ay, f"{fmt} {N}x{K} M={M}")
        ys[M] = y
    Mmax = max(Ms)
    for M in Ms:
        assert np.array_equal(ys[M].view(np.uint32), ys[Mmax][:M].view(np.uint32))


def test_full_q8_0_gemv_1024_fp32(kq, orc):
    N = K = 1024
    blocks = orc.quantize(1, inputs.weights(N, K, seed=0, tensor_id=0))
    x = inputs.activations_f32(1, K, seed=0)
    yref, ay = orc.gemv(1, blocks, x, N, K)
    y = run_gemv(kq, "q8_0", blocks, x, "f32", N, K)
    assert_close(y, yref, ay, "q8_0 1024x1024 fp32")


@pytest.mark.parametrize("N,K", [(9728, 2560), (2560, 9728)])
def test_full_q4_k_ffn_gemv(kq, orc, N, K):
    sampled_check(kq, orc, 2, "q4_k", N, K, [1], "bf16", seed=0)


@pytest.mark.parametrize("N,K", [(9728, 2560), (2560, 9728)])
def test_full_q5_k_ffn_gemv(kq, orc, N, K):
    sampled_check(kq, orc, 4, "q5_k", N, K, [1, 16], "bf16", seed=0)


@pytest.mark.parametrize("N,K", [(9728, 2560), (2560, 9728)])
def test_full_q6_k_ffn_gemv(kq, orc, N, K):
    sampled_check(kq, orc, 5, "q6_k", N, K, [1, 16], "bf16", seed=0)


def test_full_q4_k_verify_12288x4096(kq, orc):
    sampled_check(kq, orc, 2, "q4_k", 12288, 4096, [1, 2, 4, 8, 16], "bf16", seed=0)


def test_overlap_flag_gives_identical_results_in_a_chain(kq, orc):
    """KQ_OVERLAP_PREVIOUS (programmatic dependent launch): a chain of GEMVs where each reads
    the previous one's output gives the same bits as the plain chain, and matches the oracle."""
    dims = [2048, 3072, 1024, 2048]
    blocks = [orc.quantize(2, inputs.weights(dims[i + 1], dims[i], seed=40 + i, tensor_id=2))
              for i in range(len(dims) - 1)]
    wd = [dev(b) for b in blocks]
    x0 = make_x(4, dims[0], "bf16", seed=41)

    def chain(overlap):
        x = x_tensor(x0, "bf16")
        outs = []
        for i, w in enumerate(wd):
            y = kq.gemv("q4_k", w, x, dims[i + 1], dims[i], overlap=overlap)
            outs.append(y)
            x = y.to(torch.bfloat16)
        torch.cuda.synchronize()
        return [o.cpu().numpy() for o in outs]

    plain, over = chain(False), chain(True)
    for a, b in zip(plain, over):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    # the first link against the oracle
    yref, ay = orc.gemv(2, blocks[0], x0, dims[1], dims[0])
    assert_close(over[0].astype(np.float64), yref, ay, "chain link 0")
    # back-to-back GEMVs on the same input with overlap, in a CUDA graph
    x = x_tensor(x0, "bf16")
    ys = [torch.empty((4, dims[1]), device="cuda") for _ in range(6)]
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        kq.gemv("q4_k", wd[0], x, dims[1], dims[0], y=ys[0], overlap=True)
        s.synchronize()
        with torch.cuda.graph(g, stream=s):
            for y in ys:
                kq.gemv("q4_k", wd[0], x, dims[1], dims[0], y=y, overlap=True)
    g.replay()
    torch.cuda.synchronize()
    for y in ys:
        assert np.array_equal(y.cpu().numpy().view(np.uint32), plain[0].view(np.uint32))
    assert kq.device_errors() == 0


@pytest.mark.parametrize("fmt", ["q8_0", "q4_k", "q6_k"])
def test_overlap_flag_on_the_fp32_path(kq, orc, fmt):
    """KQ_OVERLAP_PREVIOUS on the CUDA-core (fp32 x) kernels: a chain where each GEMV reads
    the previous one's output gives the same bits with and without the flag (eager and in a
    CUDA graph), and the first link matches the oracle."""
    f = FMTS[fmt]
    dims = [1024, 2048, 512, 1024]
    blocks = [orc.quantize(f, inputs.weights(dims[i + 1], dims[i], seed=60 + i, tensor_id=3))
              for i in range(len(dims) - 1)]
    wd = [dev(b) for b in blocks]
    x0 = make_x(3, dims[0], "f32", seed=61)

    def chain(overlap):
        x = x_tensor(x0, "f32")
        outs = []
        for i, w in enumerate(wd):
            y = kq.gemv(fmt, w, x, dims[i + 1], dims[i], overlap=overlap)
            outs.append(y)
            x = y
        torch.cuda.synchronize()
        return [o.cpu().numpy() for o in outs]

    plain, over = chain(False), chain(True)
    for a, b in zip(plain, over):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    yref, ay = orc.gemv(f, blocks[0], x0, dims[1], dims[0])
    assert_close(over[0].astype(np.float64), yref, ay, f"{fmt} fp32 chain link 0")
    x = x_tensor(x0, "f32")
    ys = [torch.empty((3, dims[1]), device="cuda") for _ in range(6)]
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        kq.gemv(fmt, wd[0], x, dims[1], dims[0], y=ys[0], overlap=True)
        s.synchronize()
        with torch.cuda.graph(g, stream=s):
            for y in ys:
                kq.gemv(fmt, wd[0], x, dims[1], dims[0], y=y, overlap=True)
    g.replay()
    torch.cuda.synchronize()
    for y in ys:
        assert np.array_equal(y.cpu().numpy().view(np.uint32), plain[0].view(np.uint32))


@pytest.mark.parametrize("fmt", ["q4_k", "q8_0", "q6_k"])
def test_pinned_host_buffers(kq, orc, fmt):
    """x in and y out in pinned host memory (device-addressable under unified addressing): the
    kernels read and write them directly, with the same bits as device buffers."""
    f = FMTS[fmt]
    N, K, M = 700, 3072, 3
    blocks = orc.quantize(f, inputs.weights(N, K, seed=31, tensor_id=f))
    wd = dev(blocks)
    x = make_x(M, K, "bf16", seed=31)
    xd = x_tensor(x, "bf16")
    ref = kq.gemv(fmt, wd, xd, N, K)
    xh = xd.cpu().pin_memory()
    yh = torch.full((M, N), 7.0, dtype=torch.float32).pin_memory()
    kq.gemv(fmt, wd, xh, N, K, y=yh)
    torch.cuda.synchronize()
    assert np.array_equal(yh.numpy().view(np.uint32), ref.cpu().numpy().view(np.uint32))
