"""Seeded synthetic inputs shared by the tests, the oracle checks and the benchmark.

This module holds no arithmetic of the method: it draws normal numbers and
converts fp32 activations to bf16 (round to nearest even, done by torch). The
shapes and distributions are those of the workloads this library is measured on:
weights N(0, 0.02) fp32 (quantized afterwards by a quantizer), activations
N(0, 1), one row per token.

Every tensor is identified by (seed, tensor_id) so that a workload's tensors are
independent and reproducible on any machine.
"""
from __future__ import annotations

import numpy as np
import torch

WEIGHT_STD = 0.02

# Workloads (W is N x K: N output rows, K inputs).
Q8_0_GEMV_1024 = dict(name="q8_0 gemv 1024x1024 fp32 x", fmt="q8_0", shapes=[(1024, 1024)], M=[1],
                      x_dtype="f32")
Q4_K_FFN_GEMV = dict(name="q4_k gemv ffn 9728x2560 + 2560x9728 bf16 x",
                     fmt="q4_k", shapes=[(9728, 2560), (2560, 9728)], M=[1], x_dtype="bf16")
Q4_K_VERIFY = dict(name="q4_k verify 12288x4096 bf16 M in 1,2,4,8,16", fmt="q4_k",
                   shapes=[(12288, 4096)], M=[1, 2, 4, 8, 16], x_dtype="bf16")
Q4_K_PREFILL = dict(name="q4_k prefill 9728x2560 x 2048 bf16", fmt="q4_k", shapes=[(9728, 2560)],
                    M=[2048], x_dtype="bf16")
# Dense 28-layer decoder: hidden 2048, q 2048 (16 heads x 128), kv 512 (4 heads x 128),
# gated FFN 6144, vocab 151936 with a Q8_0 output head; every other linear Q4_K.
DECODE_28L = dict(name="decode step 28 layers hidden 2048 ffn 6144 vocab 151936",
                  layers=28, hidden=2048, q_dim=2048, kv_dim=512, head_dim=128, ffn=6144,
                  vocab=151936, M=[1, 8])


def _rng(seed: int, tensor_id: int) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(tensor_id)])


def weights(N: int, K: int, seed: int = 0, tensor_id: int = 0, std: float = WEIGHT_STD) -> np.ndarray:
    """N x K fp32 drawn from N(0, std^2)."""
    w = _rng(seed, tensor_id).standard_normal((N, K), dtype=np.float32)
    w *= np.float32(std)
    return w


def activations_f32(M: int, K: int, seed: int = 0, tensor_id: int = 1000) -> np.ndarray:
    """M x K fp32 drawn from N(0, 1)."""
    return _rng(seed, tensor_id).standard_normal((M, K), dtype=np.float32)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 (round to nearest even), returned as uint16 bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def activations_bf16(M: int, K: int, seed: int = 0, tensor_id: int = 1000) -> np.ndarray:
    """M x K bf16 bit patterns of N(0, 1) draws."""
    return to_bf16_bits(activations_f32(M, K, seed, tensor_id))


def weights_cuda(N: int, K: int, seed: int = 0, tensor_id: int = 0, std: float = WEIGHT_STD,
                 device: str = "cuda") -> torch.Tensor:
    """N x K fp32 N(0, std^2) drawn on the GPU by torch's Philox generator (large workloads)."""
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) << 20) ^ int(tensor_id))
    w = torch.randn((N, K), generator=g, device=device, dtype=torch.float32)
    return w.mul_(std)


def activations_cuda(M: int, K: int, seed: int = 0, tensor_id: int = 1000, dtype=torch.bfloat16,
                     device: str = "cuda") -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) << 20) ^ int(tensor_id))
    return torch.randn((M, K), generator=g, device=device, dtype=torch.float32).to(dtype)


def planted_activations_f32(targets: np.ndarray, gain: float, seed: int = 0, tensor_id: int = 1000) -> np.ndarray:
    """M x K fp32 hidden states that favour one output row each, the way a trained model's
    last hidden state favours its next token: x_j = z_j + gain * ||z_j|| * t_j / ||t_j||, with
    z_j ~ N(0, 1) and t_j row j of `targets` (the fp32 weights of the row to favour)."""
    t = np.ascontiguousarray(targets, dtype=np.float32)
    z = activations_f32(t.shape[0], t.shape[1], seed, tensor_id).astype(np.float64)
    td = t.astype(np.float64)
    zn = np.linalg.norm(z, axis=1, keepdims=True)
    tn = np.linalg.norm(td, axis=1, keepdims=True)
    return (z + gain * zn * td / np.where(tn > 0, tn, 1.0)).astype(np.float32)


def planted_activations_cuda(targets: torch.Tensor, gain: float, seed: int = 0, tensor_id: int = 1000,
                             dtype=torch.bfloat16) -> torch.Tensor:
    """The same recipe on the GPU (torch's generator for z), for full-size workloads."""
    t = targets.to(torch.float32)
    z = activations_cuda(t.shape[0], t.shape[1], seed, tensor_id, dtype=torch.float32, device=t.device)
    zn = z.norm(dim=1, keepdim=True)
    tn = t.norm(dim=1, keepdim=True).clamp_min(1e-30)
    return (z + gain * zn * t / tn).to(dtype)
