"""Decode-step driver: random block-quantized dense decoders and CUDA-graph replay.

The step itself is the library's kq_decode_step (all kernels native); this module only
allocates device buffers, quantizes synthetic weights with kq_quantize, and captures the
step in a CUDA graph (Kinetic README, "What makes it fast": the decode step is recorded once
and launched with one call per token).
"""
from __future__ import annotations

import torch

from . import DecodeModel, quantize
from .inputs import weights_cuda

# Dense 28-layer decoder: hidden 2048, q 2048 (16 heads x 128), kv 512 (4 heads x 128),
# gated FFN 6144, vocab 151936 (Q8_0 head); every other linear Q4_K.
DENSE_28L = dict(n_layers=28, hidden=2048, q_dim=2048, kv_dim=512, head_dim=128, ffn=6144,
                 vocab=151936, layer_fmt="q4_k", head_fmt="q8_0", eps=1e-6)


def matrix_shapes(d: dict):
    """(name, N, K) of every weight matrix of one layer, then the head."""
    h, q, kv, f = d["hidden"], d["q_dim"], d["kv_dim"], d["ffn"]
    return [("qkv", q + 2 * kv, h), ("o", h, q), ("gate_up", 2 * f, h), ("down", h, f)]


def random_model(d: dict, seed: int = 0, device: str = "cuda") -> DecodeModel:
    """N(0, 0.02) weights drawn on the GPU and quantized there (kq_quantize)."""
    layers = []
    tid = 0
    for _ in range(d["n_layers"]):
        lay = []
        for _, N, K in matrix_shapes(d):
            w = weights_cuda(N, K, seed=seed, tensor_id=tid, device=device)
            lay.append(quantize(d["layer_fmt"], w))
            del w
            tid += 1
        layers.append(tuple(lay))
    w = weights_cuda(d["vocab"], d["hidden"], seed=seed, tensor_id=tid, device=device)
    head = quantize(d["head_fmt"], w)
    del w
    return DecodeModel(d["n_layers"], d["hidden"], d["q_dim"], d["kv_dim"], d["head_dim"], d["ffn"],
                       d["vocab"], layers, head, d["layer_fmt"], d["head_fmt"], d["eps"])


def weight_bytes(model: DecodeModel) -> int:
    return sum(t.numel() for lay in model.layers for t in lay) + model.head.numel()


class GraphStep:
    """One decode step for M tokens captured in a CUDA graph over fixed buffers."""

    def __init__(self, model: DecodeModel, M: int, stream: torch.cuda.Stream | None = None, cache=None):
        """cache: a KVCache to run kq_decode_step_attn over (its length fixed at capture time)."""
        self.model, self.M, self.cache = model, M, cache
        dev = model.head.device
        self.x = torch.zeros((M, model.hidden), dtype=torch.bfloat16, device=dev)
        self.logits = torch.empty((M, model.vocab), dtype=torch.float32, device=dev)
        nbytes = model.attn_workspace_size(M, cache.length) if cache is not None else model.workspace_size(M)
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self.stream = stream or torch.cuda.Stream(device=dev)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(self.stream):
            self._step()  # first call outside capture (lazy set-up)
            self.stream.synchronize()
            with torch.cuda.graph(self.graph, stream=self.stream):
                self._step()

    def _step(self):
        if self.cache is None:
            self.model.step(self.x, self.logits, self.ws)
        else:
            self.model.step_attn(self.x, self.cache, logits=self.logits, workspace=self.ws)

    def replay(self):
        with torch.cuda.stream(self.stream):
            self.graph.replay()
