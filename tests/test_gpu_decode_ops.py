"""The decode step checked op by op at the contract's tolerance (kq_decode_step_trace).

The end-to-end test of the step (test_gpu_decode.py) compares logits after 28 layers, where
bf16 roundings of intermediate activations may differ between the fp32 GPU and the fp64
oracle and the difference compounds. Here every op of the GPU step is given to the oracle
with the GPU's own input (teacher forcing), so each op meets its own bar:
  - every GEMV (qkv, o, gate|up, down of every layer, and the head):
    |y_gpu - y_ref| <= 1e-4 * sum_k |w_k x_k| per element, all elements;
  - the GQA expand (the attention stand-in) and the residual adds: bit-exact (a bf16
    rounding of an fp32 value; an fp32 addition, the exact sum rounded once);
  - RMSNorm and SwiGLU: the GPU computes in fp32 and rounds to bf16, the oracle in fp64; the
    two agree except where the exact value lies within fp32 rounding of a bf16 rounding
    boundary, where they pick the neighbouring bf16 values: at most 1 bf16 ulp apart, and
    such ties are rare (at most 1 % of the elements of an op).
The model and sizes are the dense 28-layer decoder of the benchmark (hidden 2048, q 2048,
kv 512, FFN 6144, vocab 151936 Q8_0 head, every other linear Q4_K), M = 1 and 8.
"""
import numpy as np
import pytest
import torch

import quantized_decode_gemv_block_gb300 as kq
from quantized_decode_gemv_block_gb300 import decode as kqd
from quantized_decode_gemv_block_gb300 import inputs

pytestmark = pytest.mark.gpu
FMT = {"q4_k": 2, "q8_0": 1, "affine4": 3}
TOL = 1e-4


@pytest.fixture(scope="module")
def built():
    from quantized_decode_gemv_block_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def bits(t):
    return t.cpu().numpy().view(np.uint16)


def f32(t):
    return t.cpu().numpy()


def check_gemv(orc, fmt, blocks, x_bits, y_gpu, N, K, what):
    y_ref, base = orc.gemv(fmt, blocks, x_bits, N, K)
    err = np.abs(y_gpu.astype(np.float64) - y_ref)
    bad = err > TOL * base
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside 1e-4; worst " \
                          f"{(err / np.maximum(base, 1e-300)).max():.3g}"
    return float((err / np.maximum(base, 1e-300)).max())


def check_bf16_op(got, ref, what):
    """got, ref: bf16 bits. Equal, or 1 ulp apart (same sign) on at most 1 % of elements."""
    g, r = got.astype(np.int32), ref.astype(np.int32)
    same_sign = (g & 0x8000) == (r & 0x8000)
    d = np.where(same_sign, np.abs(g - r), 1 << 20)
    d = np.where((g & 0x7FFF) + (r & 0x7FFF) == 0, 0, d)  # +0 and -0
    assert d.max() <= 1, f"{what}: {int((d > 1).sum())} elements more than 1 ulp apart"
    assert (d == 1).mean() <= 0.01, f"{what}: {(d == 1).mean():.3%} one ulp apart"
    return int((d == 1).sum())


def residual_add(h, y):
    """fp32(h + y): the exact sum of two fp32 values (exact in fp64) rounded once."""
    return (h.astype(np.float64) + y.astype(np.float64)).astype(np.float32)


def make_model(orc, d, seed):
    hl, dl, tid = [], [], 0
    for _ in range(d["n_layers"]):
        lay = []
        for _, N, K in kqd.matrix_shapes(d):
            lay.append(orc.quantize(FMT[d["layer_fmt"]], inputs.weights(N, K, seed=seed, tensor_id=tid)))
            tid += 1
        hl.append(tuple(lay))
        dl.append(tuple(torch.from_numpy(b).cuda() for b in lay))
    head = orc.quantize(FMT[d["head_fmt"]], inputs.weights(d["vocab"], d["hidden"], seed=seed, tensor_id=tid))
    model = kq.DecodeModel(d["n_layers"], d["hidden"], d["q_dim"], d["kv_dim"], d["head_dim"], d["ffn"],
                           d["vocab"], dl, torch.from_numpy(head).cuda(), d["layer_fmt"], d["head_fmt"], d["eps"])
    return model, hl, head


def run_ops(orc, d, M, seed):
    model, hl, head = make_model(orc, d, seed)
    x = inputs.activations_bf16(M, d["hidden"], seed=seed, tensor_id=6000 + M)
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    logits, tr = model.step_trace(xd)
    plain = model.step(xd)
    torch.cuda.synchronize()
    # the traced step is the step: the same logits, bit for bit
    assert np.array_equal(f32(logits).view(np.uint32), f32(plain).view(np.uint32))

    lf, hf = FMT[d["layer_fmt"]], FMT[d["head_fmt"]]
    D, Q, KV, F, hd = d["hidden"], d["q_dim"], d["kv_dim"], d["ffn"], d["head_dim"]
    group = (Q // hd) // (KV // hd)
    eps = d["eps"]
    worst, ties = 0.0, 0
    h = f32(tr["h0"])
    assert np.array_equal(h, inputs.bf16_bits_to_f32(x)), "h0 = the input as fp32"
    xin = bits(tr["x0"])
    ties += check_bf16_op(xin, orc.rmsnorm_bf16(h.astype(np.float64), eps), "rmsnorm 0")
    for l, ops in enumerate(tr["layers"]):
        wqkv, wo, wgu, wd = hl[l]
        qkv = f32(ops["qkv"])
        worst = max(worst, check_gemv(orc, lf, wqkv, xin, qkv, Q + 2 * KV, D, f"layer {l} qkv"))
        # the stand-in: query head hq reads v of kv head hq // group, rounded to bf16
        v = qkv[:, Q + KV:].reshape(M, KV // hd, hd)
        o_ref = orc.bf16_rn(np.repeat(v, group, axis=1).reshape(M, Q).astype(np.float64))
        o_in = bits(ops["o_in"])
        assert np.array_equal(o_in, o_ref), f"layer {l} gqa expand"
        y_o = f32(ops["y_o"])
        worst = max(worst, check_gemv(orc, lf, wo, o_in, y_o, D, Q, f"layer {l} o"))
        h_mid = f32(ops["h_mid"])
        assert np.array_equal(h_mid.view(np.uint32), residual_add(h, y_o).view(np.uint32)), f"layer {l} add 1"
        x_mid = bits(ops["x_mid"])
        ties += check_bf16_op(x_mid, orc.rmsnorm_bf16(h_mid.astype(np.float64), eps), f"layer {l} rmsnorm 1")
        gu = f32(ops["gu"])
        worst = max(worst, check_gemv(orc, lf, wgu, x_mid, gu, 2 * F, D, f"layer {l} gate|up"))
        act = bits(ops["act"])
        ties += check_bf16_op(act, orc.swiglu_bf16(gu.astype(np.float64)), f"layer {l} swiglu")
        y_d = f32(ops["y_d"])
        worst = max(worst, check_gemv(orc, lf, wd, act, y_d, D, F, f"layer {l} down"))
        h = f32(ops["h_out"])
        assert np.array_equal(h.view(np.uint32), residual_add(h_mid, y_d).view(np.uint32)), f"layer {l} add 2"
        xin = bits(ops["x_out"])
        ties += check_bf16_op(xin, orc.rmsnorm_bf16(h.astype(np.float64), eps), f"layer {l} rmsnorm 2")
    worst = max(worst, check_gemv(orc, hf, head, xin, f32(logits), d["vocab"], D, "head"))
    assert kq.device_errors() == 0
    return worst, ties


TINY = dict(n_layers=2, hidden=256, q_dim=256, kv_dim=128, head_dim=64, ffn=512, vocab=1000,
            layer_fmt="q4_k", head_fmt="q8_0", eps=1e-6)


@pytest.mark.parametrize("M", [1, 5, 16])
def test_tiny_decode_step_op_by_op(built, orc, M):
    run_ops(orc, TINY, M, seed=40 + M)


@pytest.mark.parametrize("M", [1, 8])
def test_dense_28_layer_decode_step_op_by_op(built, orc, M):
    worst, ties = run_ops(orc, kqd.DENSE_28L, M, seed=0)
    print(f"M={M}: worst GEMV error {worst:.3g} of sum|w x|; {ties} bf16 ties at 1 ulp")
