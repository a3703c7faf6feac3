"""Scalar fp64 CPU oracle for block-quantized GEMV -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package. The CUDA product path never calls it and shares no
code with it. The arithmetic lives in ``oracle.cpp`` (plain C++, fp64, built
without contraction); this module only marshals numpy arrays through ctypes.

Each function states what it computes; the definitions and their sources are in
the headers of ``oracle.cpp``, ``decode.cpp``, ``attention.cpp`` and ``shortlist.cpp``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
_SOURCES = [os.path.join(_HERE, "oracle.cpp"), os.path.join(_HERE, "decode.cpp"),
            os.path.join(_HERE, "attention.cpp"), os.path.join(_HERE, "shortlist.cpp")]

Q8_0, Q4_K, AFFINE4, Q5_K, Q6_K = 1, 2, 3, 4, 5
F32, BF16 = 1, 2

_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so in place with g++ (-O2, OpenMP, no fp contraction)."""
    srcs = [s for s in _SOURCES if os.path.exists(s)]
    newest = max(os.path.getmtime(s) for s in srcs)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < newest:
        cmd = ["g++", "-std=c++17", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-o", _SO + ".tmp"] + srcs
        subprocess.run(cmd, check=True)
        os.replace(_SO + ".tmp", _SO)
    return _SO


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO)
        P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.orc_block_bytes.argtypes = [I]
        L.orc_block_weights.argtypes = [I]
        L.orc_half_to_double.argtypes = [ctypes.c_uint16]
        L.orc_half_to_double.restype = ctypes.c_double
        for f in (L.orc_double_to_half_rn, L.orc_double_to_half_up, L.orc_double_to_half_down):
            f.argtypes = [ctypes.c_double]
            f.restype = ctypes.c_uint16
        L.orc_unpack_scale_min.argtypes = [P, I, P, P]
        L.orc_quantize.argtypes = [I, P, I64, I64, P, I]
        L.orc_dequant.argtypes = [I, P, I64, I64, P]
        L.orc_gemv.argtypes = [I, P, I, P, I64, I64, I64, P, P, I]
        L.orc_gemv_sampled.argtypes = [I, P, I, P, I64, I64, I64, I64, P, P, P, P, I]
        L.orc_double_to_bf16_rn.argtypes = [ctypes.c_double]
        L.orc_double_to_bf16_rn.restype = ctypes.c_uint16
        L.orc_rmsnorm.argtypes = [P, P, I64, I64, ctypes.c_double]
        L.orc_bf16_rn_n.argtypes = [P, I64, P]
        L.orc_swiglu.argtypes = [P, I64, I64, P]
        L.orc_decode_step.argtypes = [I, I, I, I, I, I, I, I, I, ctypes.c_double, P, P, P, P, P, P, I64,
                                      P, I, P]
        L.orc_attention.argtypes = [I, I, I, I, I, P, P, P, P, ctypes.c_float, P, P]
        L.orc_attention.restype = I
        L.orc_decode_step_attn.argtypes = [I, I, I, I, I, I, I, I, I, ctypes.c_double, P, P, P, P, P, P, P, I,
                                           P, ctypes.c_float, P, I64, P, I, P]
        L.orc_decode_step_attn.restype = I
        L.orc_shortlist_build.argtypes = [P, I64, I64, P, P, I]
        L.orc_shortlist_build.restype = I
        _lib = L
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def block_bytes(fmt: int) -> int:
    return lib().orc_block_bytes(fmt)


def block_weights(fmt: int) -> int:
    return lib().orc_block_weights(fmt)


def row_bytes(fmt: int, K: int) -> int:
    return K // block_weights(fmt) * block_bytes(fmt)


def half_to_double(h: int) -> float:
    return lib().orc_half_to_double(h)


def double_to_half_rn(v: float) -> int:
    return lib().orc_double_to_half_rn(v)


def double_to_half_up(v: float) -> int:
    return lib().orc_double_to_half_up(v)


def double_to_half_down(v: float) -> int:
    return lib().orc_double_to_half_down(v)


def unpack_scale_min(sc12: bytes, j: int):
    a = np.frombuffer(bytes(sc12), dtype=np.uint8).copy()
    sc, m = ctypes.c_int(), ctypes.c_int()
    lib().orc_unpack_scale_min(_ptr(a), j, ctypes.byref(sc), ctypes.byref(m))
    return sc.value, m.value


def quantize(fmt: int, w: np.ndarray, nthreads: int = 0) -> np.ndarray:
    """fp32 N x K -> uint8 N x row_bytes blocks (the oracle's own quantizer)."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    N, K = w.shape
    out = np.empty((N, row_bytes(fmt, K)), dtype=np.uint8)
    nt = nthreads or os.cpu_count() or 1
    if lib().orc_quantize(fmt, _ptr(w), N, K, _ptr(out), nt) != 0:
        raise ValueError("orc_quantize: bad format or K")
    return out


def dequant(fmt: int, blocks: np.ndarray, N: int, K: int) -> np.ndarray:
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    out = np.empty((N, K), dtype=np.float64)
    if lib().orc_dequant(fmt, _ptr(blocks), N, K, _ptr(out)) != 0:
        raise ValueError("orc_dequant: bad format or K")
    return out


def _x_code(x: np.ndarray):
    if x.dtype == np.float32:
        return F32
    if x.dtype == np.uint16:  # bf16 bit patterns
        return BF16
    raise TypeError("x must be float32 or uint16 (bf16 bits)")


def gemv(fmt: int, blocks: np.ndarray, x: np.ndarray, N: int, K: int, nthreads: int = 0):
    """Return (y, absy), both M x N fp64: y = x @ deq(W)^T, absy = |x| @ |deq(W)|^T."""
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    x = np.ascontiguousarray(x)
    M = x.shape[0]
    y = np.empty((M, N), dtype=np.float64)
    ay = np.empty((M, N), dtype=np.float64)
    nt = nthreads or os.cpu_count() or 1
    if lib().orc_gemv(fmt, _ptr(blocks), _x_code(x), _ptr(x), M, N, K, _ptr(y), _ptr(ay), nt) != 0:
        raise ValueError("orc_gemv: bad arguments")
    return y, ay


def gemv_sampled(fmt: int, blocks: np.ndarray, x: np.ndarray, N: int, K: int, js, ns,
                 nthreads: int = 0):
    """(y, absy) at the output coordinates (js[p], ns[p]) only."""
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    x = np.ascontiguousarray(x)
    M = x.shape[0]
    js = np.ascontiguousarray(js, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    y = np.empty(len(js), dtype=np.float64)
    ay = np.empty(len(js), dtype=np.float64)
    nt = nthreads or os.cpu_count() or 1
    rc = lib().orc_gemv_sampled(fmt, _ptr(blocks), _x_code(x), _ptr(x), M, N, K, len(js),
                                _ptr(js), _ptr(ns), _ptr(y), _ptr(ay), nt)
    if rc != 0:
        raise ValueError(f"orc_gemv_sampled: bad arguments ({rc})")
    return y, ay


def double_to_bf16_rn(v: float) -> int:
    return lib().orc_double_to_bf16_rn(v)


def bf16_rn(v: np.ndarray) -> np.ndarray:
    """bf16 bits of every value of v (fp64 in, nearest, ties to even), same shape."""
    a = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(a.shape, dtype=np.uint16)
    lib().orc_bf16_rn_n(_ptr(a), a.size, _ptr(out))
    return out


def swiglu_bf16(gu: np.ndarray) -> np.ndarray:
    """bf16 bits of silu(g) * u for gu = [g | u] (M x 2F, fp64 arithmetic) -> M x F."""
    gu = np.ascontiguousarray(gu, dtype=np.float64)
    M, F2 = gu.shape
    out = np.empty((M, F2 // 2), dtype=np.uint16)
    lib().orc_swiglu(_ptr(gu), M, F2 // 2, _ptr(out))
    return out


def rmsnorm_bf16(h: np.ndarray, eps: float) -> np.ndarray:
    """bf16 bits of h / sqrt(mean(h^2) + eps), row by row (fp64 arithmetic)."""
    h = np.ascontiguousarray(h, dtype=np.float64)
    M, D = h.shape
    out = np.empty((M, D), dtype=np.uint16)
    lib().orc_rmsnorm(_ptr(h), _ptr(out), M, D, eps)
    return out


def decode_step(dims: dict, layers: list, head: np.ndarray, x_bf16: np.ndarray, nthreads: int = 0,
                return_head_input: bool = False):
    """Logits (M x vocab, fp64) of one decode step (definition in decode.cpp); optionally
    also the head's input (bf16 bits of the final RMSNorm).

    dims: n_layers, hidden, q_dim, kv_dim, head_dim, ffn, vocab, layer_fmt, head_fmt, eps.
    layers: per layer (w_qkv, w_o, w_gate_up, w_down) blocks (uint8 arrays); head: blocks."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    M = x.shape[0]
    keep = [np.ascontiguousarray(a, dtype=np.uint8) for lay in layers for a in lay]
    ptrs = [[keep[4 * l + i].ctypes.data for l in range(len(layers))] for i in range(4)]
    arrs = [(ctypes.c_void_p * max(1, len(layers)))(*p) for p in ptrs]
    headb = np.ascontiguousarray(head, dtype=np.uint8)
    out = np.empty((M, dims["vocab"]), dtype=np.float64)
    xf = np.empty((M, dims["hidden"]), dtype=np.uint16)
    nt = nthreads or os.cpu_count() or 1
    rc = lib().orc_decode_step(dims["n_layers"], dims["hidden"], dims["q_dim"], dims["kv_dim"],
                               dims["head_dim"], dims["ffn"], dims["vocab"], dims["layer_fmt"],
                               dims["head_fmt"], dims["eps"], *[ctypes.cast(a, ctypes.c_void_p) for a in arrs],
                               _ptr(headb), _ptr(x), M, _ptr(out), nt, _ptr(xf))
    if rc != 0:
        raise ValueError("orc_decode_step failed")
    return (out, xf) if return_head_input else out


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, L: int, n_q: int, n_kv: int, hd: int,
              scale: float, mask: np.ndarray | None = None):
    """(out, base), both M x (n_q*hd) fp64: decode attention of the M window tokens (definition
    in attention.cpp). q: M x (n_q*hd) fp32; k, v: (L+M) x (n_kv*hd) bf16 bits (uint16);
    mask: M uint32 words (bit j of word i: token i sees window token j) or None (causal)."""
    q = np.ascontiguousarray(q, dtype=np.float32)
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = np.ascontiguousarray(v, dtype=np.uint16)
    M = q.shape[0]
    out = np.empty((M, n_q * hd), dtype=np.float64)
    base = np.empty((M, n_q * hd), dtype=np.float64)
    mp = None
    if mask is not None:
        mask = np.ascontiguousarray(mask, dtype=np.uint32)
        mp = _ptr(mask)
    if lib().orc_attention(M, L, n_q, n_kv, hd, _ptr(q), _ptr(k), _ptr(v), mp, scale, _ptr(out), _ptr(base)) != 0:
        raise ValueError("orc_attention: bad arguments")
    return out, base


def decode_step_attn(dims: dict, layers: list, head: np.ndarray, k_cache: list, v_cache: list, L: int,
                     x_bf16: np.ndarray, scale: float, mask: np.ndarray | None = None, nthreads: int = 0,
                     return_head_input: bool = False):
    """Logits (M x vocab, fp64) of one decode step with attention over a KV cache (definition in
    decode.cpp, orc_decode_step_attn). k_cache[l], v_cache[l]: L x kv_dim bf16 bits (uint16)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    M = x.shape[0]
    keep = [np.ascontiguousarray(a, dtype=np.uint8) for lay in layers for a in lay]
    n = max(1, len(layers))
    ptrs = [[keep[4 * l + i].ctypes.data for l in range(len(layers))] for i in range(4)]
    arrs = [(ctypes.c_void_p * n)(*p) for p in ptrs]
    kk = [np.ascontiguousarray(a, dtype=np.uint16) for a in k_cache]
    vv = [np.ascontiguousarray(a, dtype=np.uint16) for a in v_cache]
    karr = (ctypes.c_void_p * n)(*[a.ctypes.data for a in kk])
    varr = (ctypes.c_void_p * n)(*[a.ctypes.data for a in vv])
    headb = np.ascontiguousarray(head, dtype=np.uint8)
    out = np.empty((M, dims["vocab"]), dtype=np.float64)
    xf = np.empty((M, dims["hidden"]), dtype=np.uint16)
    mp = None
    if mask is not None:
        mask = np.ascontiguousarray(mask, dtype=np.uint32)
        mp = _ptr(mask)
    nt = nthreads or os.cpu_count() or 1
    rc = lib().orc_decode_step_attn(dims["n_layers"], dims["hidden"], dims["q_dim"], dims["kv_dim"],
                                    dims["head_dim"], dims["ffn"], dims["vocab"], dims["layer_fmt"],
                                    dims["head_fmt"], dims["eps"], *[ctypes.cast(a, ctypes.c_void_p) for a in arrs],
                                    _ptr(headb), ctypes.cast(karr, ctypes.c_void_p), ctypes.cast(varr, ctypes.c_void_p),
                                    L, mp, scale, _ptr(x), M, _ptr(out), nt, _ptr(xf))
    if rc != 0:
        raise ValueError("orc_decode_step_attn failed")
    return (out, xf) if return_head_input else out


def shortlist_build(w_q8: np.ndarray, N: int, K: int, nthreads: int = 0):
    """Small copy (Q4_K bytes, N x K/256 x 144) and per-row score bounds B_n (fp32) of a Q8_0
    head (definition in shortlist.cpp). A row can win only if approx_n + B_n ||x|| >=
    max_m (approx_m - B_m ||x||), approx being the small copy's product."""
    w = np.ascontiguousarray(w_q8, dtype=np.uint8)
    small = np.empty(N * (K // 256) * 144, dtype=np.uint8)
    bound = np.empty(N, dtype=np.float32)
    nt = nthreads or os.cpu_count() or 1
    if lib().orc_shortlist_build(_ptr(w), N, K, _ptr(small), _ptr(bound), nt) != 0:
        raise ValueError("orc_shortlist_build: bad arguments")
    return small, bound
