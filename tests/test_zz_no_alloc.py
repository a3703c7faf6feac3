"""kq_decode_step_static: the decode step with library-held scratch (no allocation per call).

Callers that cannot allocate device memory (they borrow the GPU from a framework that owns
every allocation, or must not allocate on a latency-critical path or during stream capture)
use this entry point instead of kq_decode_step. This test checks, through the C-ABI, that two
calls in a row give the same logits as kq_decode_step with a caller workspace, and that a
model too large for the fixed scratch is refused. It sits last in collection order so that a
run stopping at the first failure has run every other test first.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kq():
    from quantized_decode_gemv_block_gb300 import build
    build.build()
    import quantized_decode_gemv_block_gb300 as m
    assert torch.cuda.is_available()
    return m


SMALL = dict(n_layers=2, hidden=512, q_dim=512, kv_dim=256, head_dim=128, ffn=1024, vocab=2000,
             layer_fmt="q4_k", head_fmt="q8_0", eps=1e-6)


def test_static_scratch_step_matches_workspace_step(kq):
    from quantized_decode_gemv_block_gb300 import decode as kqd
    model = kqd.random_model(SMALL, seed=7)
    M = 5
    x = torch.randn((M, SMALL["hidden"]), device="cuda").to(torch.bfloat16)
    ref = model.step(x).clone()  # kq_decode_step with a caller workspace
    L = kq.lib()
    for call in range(2):
        out = torch.full((M, SMALL["vocab"]), float("nan"), device="cuda")
        rc = L.kq_decode_step_static(ctypes.byref(model.c), x.data_ptr(), out.data_ptr(), M,
                                     torch.cuda.current_stream().cuda_stream)
        assert rc == 0, L.kq_last_error().decode()
        torch.cuda.synchronize()
        # same kernels and split as kq_decode_step: identical bits (inside any tolerance)
        assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.cpu().numpy().view(np.uint32)), call
    assert kq.device_errors() == 0


def test_static_scratch_refuses_models_beyond_its_size(kq):
    from quantized_decode_gemv_block_gb300 import decode as kqd
    big = dict(SMALL, ffn=65536, n_layers=0)  # gate/up workspace alone: 16 x 131072 x 4 bytes > 4 MiB
    model = kqd.random_model(big, seed=8)
    need = model.workspace_size(16)
    assert need > 4 * 2**20
    x = torch.zeros((16, big["hidden"]), device="cuda").to(torch.bfloat16)
    out = torch.empty((16, big["vocab"]), device="cuda")
    rc = kq.lib().kq_decode_step_static(ctypes.byref(model.c), x.data_ptr(), out.data_ptr(), 16, None)
    assert rc == kq.KQ_ERR_WORKSPACE
    assert "static scratch" in kq.lib().kq_last_error().decode()


def test_static_scratch_holds_the_dense_28_layer_model_at_16_tokens(kq):
    """The 4 MiB array is sized for the dense 28-layer decoder (hidden 2048, ffn 6144, vocab
    151936) up to 16 tokens: its step runs from the array and gives kq_decode_step's bits."""
    from quantized_decode_gemv_block_gb300 import decode as kqd
    model = kqd.random_model(kqd.DENSE_28L, seed=9)
    M = 16
    assert model.workspace_size(M) <= 4 * 2**20
    x = torch.randn((M, kqd.DENSE_28L["hidden"]), device="cuda").to(torch.bfloat16)
    ref = model.step(x).clone()
    out = torch.full((M, kqd.DENSE_28L["vocab"]), float("nan"), device="cuda")
    L = kq.lib()
    rc = L.kq_decode_step_static(ctypes.byref(model.c), x.data_ptr(), out.data_ptr(), M,
                                 torch.cuda.current_stream().cuda_stream)
    assert rc == 0, L.kq_last_error().decode()
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.cpu().numpy().view(np.uint32))
    assert kq.device_errors() == 0
