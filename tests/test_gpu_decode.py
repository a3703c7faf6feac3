"""GPU decode step (kq_decode_step) against the fp64 oracle step, and batch invariance.

Tolerance, and where it comes from: every GEMV input is rounded to bf16, and the GPU (fp32
arithmetic) and the oracle (fp64) round an activation lying within the GEMV's ~1e-6
relative error of a bf16 rounding boundary to neighbouring bf16 values (about 1e-6 / 2^-8,
i.e. 2.6e-4 of the elements at each rounding point). One flip in the head's input moves a
logit by at most 2^-8 |w_k x_k|; flips upstream move the residual stream by a similar
relative amount and accumulate over layers. Per logit the test allows 1e-2 * sum_k |w_k x_k|
(sum over the head row, x = the oracle's final activations) and a median of 1e-5 per layer
of depth (2 layers: 2e-5; 28 layers: 2.8e-4).
"""
import numpy as np
import pytest
import torch

import quantized_decode_gemv_block_gb300 as kq
from quantized_decode_gemv_block_gb300 import decode as kqd
from quantized_decode_gemv_block_gb300 import inputs

pytestmark = pytest.mark.gpu
FMT = {"q4_k": 2, "q8_0": 1, "affine4": 3}


@pytest.fixture(scope="module")
def built():
    from quantized_decode_gemv_block_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def make(orc, d, seed):
    """Weights from numpy, quantized by the oracle; the same blocks go to the GPU."""
    host_layers, dev_layers, tid = [], [], 0
    for _ in range(d["n_layers"]):
        hl = []
        for _, N, K in kqd.matrix_shapes(d):
            hl.append(orc.quantize(FMT[d["layer_fmt"]], inputs.weights(N, K, seed=seed, tensor_id=tid)))
            tid += 1
        host_layers.append(tuple(hl))
        dev_layers.append(tuple(torch.from_numpy(b).cuda() for b in hl))
    head = orc.quantize(FMT[d["head_fmt"]], inputs.weights(d["vocab"], d["hidden"], seed=seed, tensor_id=tid))
    model = kq.DecodeModel(d["n_layers"], d["hidden"], d["q_dim"], d["kv_dim"], d["head_dim"], d["ffn"],
                           d["vocab"], dev_layers, torch.from_numpy(head).cuda(), d["layer_fmt"],
                           d["head_fmt"], d["eps"])
    odims = dict(d, layer_fmt=FMT[d["layer_fmt"]], head_fmt=FMT[d["head_fmt"]])
    return model, host_layers, head, odims


def check_logits(orc, odims, head, logits_gpu, ref, xfinal):
    depth = max(1, odims["n_layers"])
    # tolerance base: sum_k |w_k x_k| over the head row, x = the oracle's final activations
    W = orc.dequant(odims["head_fmt"], head, odims["vocab"], odims["hidden"])
    base = np.abs(inputs.bf16_bits_to_f32(xfinal).astype(np.float64)) @ np.abs(W).T
    err = np.abs(logits_gpu.astype(np.float64) - ref)
    assert np.all(err <= 1e-2 * base), f"max err/base {(err / base).max():.3g}"
    assert np.median(err / base) < 1e-5 * depth, f"median err/base {np.median(err / base):.3g}"


TINY = dict(n_layers=2, hidden=256, q_dim=256, kv_dim=128, head_dim=64, ffn=512, vocab=1000,
            layer_fmt="q4_k", head_fmt="q8_0", eps=1e-6)


def test_tiny_decode_matches_oracle_and_is_batch_invariant(built, orc):
    model, hl, head, od = make(orc, TINY, seed=11)
    x = inputs.activations_bf16(16, TINY["hidden"], seed=12)
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    full = model.step(xd).cpu().numpy()
    ref, xf = orc.decode_step(od, hl, head, x, return_head_input=True)
    check_logits(orc, od, head, full, ref, xf)
    for M in (1, 3, 8):
        y = model.step(xd[:M].contiguous()).cpu().numpy()
        assert np.array_equal(y.view(np.uint32), full[:M].view(np.uint32)), f"M={M}"
    assert kq.device_errors() == 0


def test_decode_graph_replay_matches_eager(built, orc):
    model, hl, head, od = make(orc, dict(TINY, head_fmt="q4_k", vocab=512), seed=13)
    g = kqd.GraphStep(model, 4)
    x = inputs.activations_bf16(4, TINY["hidden"], seed=14)
    g.x.copy_(torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16))
    g.replay()
    torch.cuda.synchronize()
    eager = model.step(g.x.clone()).cpu().numpy()
    assert np.array_equal(g.logits.cpu().numpy().view(np.uint32), eager.view(np.uint32))


@pytest.mark.parametrize("M", [1, 8])
def test_full_dense_28_layer_decode_step(built, orc, M):
    d = kqd.DENSE_28L
    model, hl, head, od = make(orc, d, seed=0)
    x = inputs.activations_bf16(M, d["hidden"], seed=0, tensor_id=5000)
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    logits = model.step(xd).cpu().numpy()
    ref, xf = orc.decode_step(od, hl, head, x, return_head_input=True)
    check_logits(orc, od, head, logits, ref, xf)
    assert kq.device_errors() == 0


# ---- the step with attention over a KV cache (kq_decode_step_attn) ----

def make_cache(d, L, M, seed):
    """Random bf16 context rows (host bits) and a device cache holding them (capacity L + M)."""
    kh, vh = [], []
    for l in range(d["n_layers"]):
        kh.append(inputs.activations_bf16(L, d["kv_dim"], seed=seed, tensor_id=8000 + 2 * l) if L else
                  np.zeros((0, d["kv_dim"]), np.uint16))
        vh.append(inputs.activations_bf16(L, d["kv_dim"], seed=seed, tensor_id=8001 + 2 * l) if L else
                  np.zeros((0, d["kv_dim"]), np.uint16))
    cache = kq.KVCache(d["n_layers"], L + M, d["kv_dim"])
    for l in range(d["n_layers"]):
        if L:
            cache.k[l][:L].copy_(torch.from_numpy(kh[l].view(np.int16)).cuda().view(torch.bfloat16))
            cache.v[l][:L].copy_(torch.from_numpy(vh[l].view(np.int16)).cuda().view(torch.bfloat16))
    cache.length = L
    return cache, kh, vh


def attn_scale(hd):
    return float(np.float32(1.0) / np.sqrt(np.float32(hd)))  # as the kernels form it


def test_tiny_decode_with_attention_matches_oracle_and_is_batch_invariant(built, orc):
    model, hl, head, od = make(orc, TINY, seed=31)
    M, L = 5, 37
    cache, kh, vh = make_cache(TINY, L, M, seed=32)
    x = inputs.activations_bf16(M, TINY["hidden"], seed=33)
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    sc = attn_scale(TINY["head_dim"])
    full = model.step_attn(xd, cache).cpu().numpy()
    ref, xf = orc.decode_step_attn(od, hl, head, kh, vh, L, x, sc, return_head_input=True)
    check_logits(orc, od, head, full, ref, xf)
    for m in (1, 2):  # the first tokens alone: the same bits
        y = model.step_attn(xd[:m].contiguous(), cache).cpu().numpy()
        assert np.array_equal(y.view(np.uint32), full[:m].view(np.uint32)), f"M={m}"
    # a tree of guesses: token i sees window tokens 0 and i
    mask = np.array([1 | (1 << i) for i in range(M)], np.uint32)
    yt = model.step_attn(xd, cache, mask=torch.from_numpy(mask.view(np.int32)).cuda()).cpu().numpy()
    ref_t, xf_t = orc.decode_step_attn(od, hl, head, kh, vh, L, x, sc, mask=mask, return_head_input=True)
    check_logits(orc, od, head, yt, ref_t, xf_t)
    assert kq.device_errors() == 0


@pytest.mark.parametrize("M,L", [(6, 125), (4, 0), (3, 256)])
def test_verify_window_equals_plain_decoding(built, orc, M, L):
    """The rule the pages' speed-ups rest on (Kinetic README, "What makes it fast"): checking M
    guesses in one pass gives the bits plain decoding gives. One step over a window of M tokens
    at cache length L against M steps of one token each, the cache growing by one row per step:
    the same logits, bit for bit (the window may cross a 128-position chunk boundary)."""
    model, hl, head, od = make(orc, TINY, seed=37 + L)
    cache, _, _ = make_cache(TINY, L, M, seed=38 + L)
    x = inputs.activations_bf16(M, TINY["hidden"], seed=39 + L)
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    win = model.step_attn(xd, cache).cpu().numpy()
    for i in range(M):
        cache.length = L + i  # the earlier guesses are now cached (their rows were just written)
        y = model.step_attn(xd[i:i + 1].contiguous(), cache).cpu().numpy()
        assert np.array_equal(y.view(np.uint32), win[i:i + 1].view(np.uint32)), f"token {i}"
    assert kq.device_errors() == 0


def test_decode_with_attention_and_no_context_is_the_stand_in_step(built, orc):
    """L = 0 and each token seeing only itself: the same logits as kq_decode_step (both
    paths round the same values the same way)."""
    model, hl, head, od = make(orc, TINY, seed=34)
    M = 3
    cache, _, _ = make_cache(TINY, 0, M, seed=35)
    x = inputs.activations_bf16(M, TINY["hidden"], seed=36)
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    mask = torch.from_numpy(np.array([1 << i for i in range(M)], np.uint32).view(np.int32)).cuda()
    a = model.step_attn(xd, cache, mask=mask).cpu().numpy()
    b = model.step(xd).cpu().numpy()
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("M", [1, 8])
def test_full_dense_28_layer_decode_with_attention(built, orc, M):
    d = kqd.DENSE_28L
    model, hl, head, od = make(orc, d, seed=0)
    L = 200
    cache, kh, vh = make_cache(d, L, M, seed=37)
    x = inputs.activations_bf16(M, d["hidden"], seed=0, tensor_id=5001)
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    logits = model.step_attn(xd, cache).cpu().numpy()
    ref, xf = orc.decode_step_attn(od, hl, head, kh, vh, L, x, attn_scale(d["head_dim"]), return_head_input=True)
    check_logits(orc, od, head, logits, ref, xf)
    assert kq.device_errors() == 0
