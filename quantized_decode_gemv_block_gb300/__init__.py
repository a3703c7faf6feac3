"""kq: fused dequantize-and-multiply of block-quantized weights on GB300 (sm_103a).

A thin ctypes binding over the C-ABI library ``libkq.so`` (declared in
``include/kq.h``). This module only marshals arguments: it passes device pointers
and the current CUDA stream to the library and raises on a nonzero status. Every
step of the computation runs in the library's CUDA kernels; there is no CPU or
PyTorch fallback, and importing fails loudly if ``libkq.so`` has not been built
(``python -m quantized_decode_gemv_block_gb300.build``).
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkq.so")

Q8_0, Q4_K, AFFINE4, Q5_K, Q6_K = 1, 2, 3, 4, 5
F32, BF16 = 1, 2
FORMATS = {"q8_0": Q8_0, "q4_k": Q4_K, "affine4": AFFINE4, "q5_k": Q5_K, "q6_k": Q6_K}
KQ_OK, KQ_ERR_ARG, KQ_ERR_UNSUPPORTED, KQ_ERR_WORKSPACE, KQ_ERR_CUDA, KQ_ERR_TIMEOUT = 0, -1, -2, -3, -4, -5


class KQError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"kq error {code}: {msg}")
        self.code = code


class DecodeModelC(ctypes.Structure):
    """Mirror of kq_decode_model (include/kq.h)."""
    _fields_ = [("n_layers", ctypes.c_int), ("hidden", ctypes.c_int), ("q_dim", ctypes.c_int),
                ("kv_dim", ctypes.c_int), ("head_dim", ctypes.c_int), ("ffn", ctypes.c_int),
                ("vocab", ctypes.c_int), ("layer_fmt", ctypes.c_int), ("head_fmt", ctypes.c_int),
                ("rms_eps", ctypes.c_float), ("w_qkv", ctypes.POINTER(ctypes.c_void_p)),
                ("w_o", ctypes.POINTER(ctypes.c_void_p)), ("w_gate_up", ctypes.POINTER(ctypes.c_void_p)),
                ("w_down", ctypes.POINTER(ctypes.c_void_p)), ("w_head", ctypes.c_void_p)]


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libkq.so and declare its C signatures. Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with "
                          "`python -m quantized_decode_gemv_block_gb300.build` (needs nvcc)")
    L = ctypes.CDLL(path)
    P, I, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    L.kq_block_bytes.argtypes = [I]
    L.kq_block_bytes.restype = SZ
    L.kq_block_weights.argtypes = [I]
    L.kq_block_weights.restype = SZ
    L.kq_row_bytes.argtypes = [I, I]
    L.kq_row_bytes.restype = SZ
    L.kq_last_error.restype = ctypes.c_char_p
    L.kq_version.restype = ctypes.c_char_p
    L.kq_gemv.argtypes = [I, P, I, P, P, I, I, I, P]
    L.kq_gemv.restype = I
    L.kq_gemv_ex.argtypes = [I, P, I, P, P, I, I, I, ctypes.c_uint, P]
    L.kq_gemv_ex.restype = I
    L.kq_gemm.argtypes = [I, P, I, P, P, I, I, I, P, SZ, P]
    L.kq_gemm.restype = I
    L.kq_gemm_workspace_size.argtypes = [I, I, I, I, I]
    L.kq_gemm_workspace_size.restype = SZ
    L.kq_quantize.argtypes = [I, P, P, I, I, P]
    L.kq_quantize.restype = I
    L.kq_device_errors.restype = I
    L.kq_decode_workspace_size.argtypes = [ctypes.POINTER(DecodeModelC), I]
    L.kq_decode_workspace_size.restype = SZ
    L.kq_attention_workspace_size.argtypes = [I, I, I, I, I]
    L.kq_attention_workspace_size.restype = SZ
    L.kq_attention.argtypes = [P, P, P, P, I, I, I, I, I, P, ctypes.c_float, P, SZ, P]
    L.kq_attention.restype = I
    L.kq_decode_attn_workspace_size.argtypes = [ctypes.POINTER(DecodeModelC), I, I]
    L.kq_decode_attn_workspace_size.restype = SZ
    L.kq_decode_step_attn.argtypes = [ctypes.POINTER(DecodeModelC), ctypes.POINTER(KVCacheC), P, P, I, P, P, SZ, P]
    L.kq_decode_step_attn.restype = I
    L.kq_decode_step.argtypes = [ctypes.POINTER(DecodeModelC), P, P, I, P, SZ, P]
    L.kq_decode_step.restype = I
    L.kq_decode_step_static.argtypes = [ctypes.POINTER(DecodeModelC), P, P, I, P]
    L.kq_decode_trace_size.argtypes = [ctypes.POINTER(DecodeModelC), I]
    L.kq_decode_trace_size.restype = SZ
    L.kq_decode_step_trace.argtypes = [ctypes.POINTER(DecodeModelC), P, P, I, P, SZ, P, SZ, P]
    L.kq_decode_step_trace.restype = I
    L.kq_decode_step_static.restype = I
    L.kq_shortlist_bytes.argtypes = [I, I]
    L.kq_shortlist_bytes.restype = SZ
    L.kq_shortlist_build.argtypes = [P, I, I, P, SZ, P]
    L.kq_shortlist_build.restype = I
    L.kq_head_argmax_workspace_size.argtypes = [I, I]
    L.kq_head_argmax_workspace_size.restype = SZ
    L.kq_head_argmax.argtypes = [P, P, I, P, I, I, I, P, P, P, P, SZ, ctypes.c_uint, P]
    L.kq_head_argmax.restype = I
    _lib = L
    return L


def lib():
    return load_library()


def _fmt(fmt) -> int:
    return FORMATS[fmt] if isinstance(fmt, str) else int(fmt)


def _check(rc: int):
    if rc != KQ_OK:
        raise KQError(rc, lib().kq_last_error().decode())


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def block_bytes(fmt) -> int:
    return lib().kq_block_bytes(_fmt(fmt))


def block_weights(fmt) -> int:
    return lib().kq_block_weights(_fmt(fmt))


def row_bytes(fmt, K: int) -> int:
    return lib().kq_row_bytes(_fmt(fmt), K)


def version() -> str:
    return lib().kq_version().decode()


def _x_dtype(x: torch.Tensor) -> int:
    if x.dtype == torch.bfloat16:
        return BF16
    if x.dtype == torch.float32:
        return F32
    raise TypeError("x must be torch.bfloat16 or torch.float32")


KQ_OVERLAP_PREVIOUS = 1


def gemv(fmt, w: torch.Tensor, x: torch.Tensor, N: int, K: int, y: torch.Tensor | None = None,
         stream=None, overlap: bool = False) -> torch.Tensor:
    """Y (M x N fp32) = X (M x K) @ deq(W)^T for M <= 16, through kq_gemv / kq_gemv_ex.

    overlap=True passes KQ_OVERLAP_PREVIOUS: the previous kernel on the stream must not
    write w (it may still be running while this one streams w)."""
    M = x.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    if overlap:
        rc = lib().kq_gemv_ex(_fmt(fmt), w.data_ptr(), _x_dtype(x), x.data_ptr(), y.data_ptr(), M, N, K,
                              KQ_OVERLAP_PREVIOUS, _stream(stream))
    else:
        rc = lib().kq_gemv(_fmt(fmt), w.data_ptr(), _x_dtype(x), x.data_ptr(), y.data_ptr(), M, N, K,
                           _stream(stream))
    _check(rc)
    return y


def gemm_workspace_size(fmt, x_dtype, M: int, N: int, K: int) -> int:
    xd = x_dtype if isinstance(x_dtype, int) else (BF16 if x_dtype == torch.bfloat16 else F32)
    return lib().kq_gemm_workspace_size(_fmt(fmt), xd, M, N, K)


def gemm(fmt, w: torch.Tensor, x: torch.Tensor, N: int, K: int, y: torch.Tensor | None = None,
         workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Y = X @ deq(W)^T for any M, through kq_gemm (tensor cores for M > 16)."""
    M = x.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    need = gemm_workspace_size(fmt, _x_dtype(x), M, N, K)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    wp = workspace.data_ptr() if workspace is not None else None
    wn = workspace.numel() if workspace is not None else 0
    _check(lib().kq_gemm(_fmt(fmt), w.data_ptr(), _x_dtype(x), x.data_ptr(), y.data_ptr(), M, N, K,
                         wp, wn, _stream(stream)))
    return y


def attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, L: int, n_q: int, n_kv: int,
              head_dim: int, scale: float, mask: torch.Tensor | None = None, out: torch.Tensor | None = None,
              workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Decode attention of the M window tokens (kq_attention): q M x (n_q*head_dim) fp32,
    k_cache / v_cache (L+M) x (n_kv*head_dim) bf16, mask None (causal) or M int32 words."""
    M = q.shape[0]
    if out is None:
        out = torch.empty((M, n_q * head_dim), dtype=torch.float32, device=q.device)
    need = lib().kq_attention_workspace_size(M, L, n_q, n_kv, head_dim)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _check(lib().kq_attention(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), out.data_ptr(), M, L, n_q,
                              n_kv, head_dim, mask.data_ptr() if mask is not None else None, scale,
                              workspace.data_ptr(), workspace.numel(), _stream(stream)))
    return out


KQ_HEAD_ALL_ROWS = 1


def shortlist_build(w_q8: torch.Tensor, N: int, K: int, out: torch.Tensor | None = None,
                    stream=None) -> torch.Tensor:
    """The shortlist buffer of a Q8_0 head (kq_shortlist_build): the small Q4_K copy, then
    N fp32 score bounds (see shortlist_parts)."""
    need = lib().kq_shortlist_bytes(N, K)
    if need == 0:
        raise KQError(KQ_ERR_ARG, "bad head shape for the shortlist")
    if out is None:
        out = torch.empty(need, dtype=torch.uint8, device=w_q8.device)
    _check(lib().kq_shortlist_build(w_q8.data_ptr(), N, K, out.data_ptr(), out.numel(), _stream(stream)))
    return out


def shortlist_parts(buf: torch.Tensor, N: int, K: int):
    """(small copy bytes N x K/256*144, bounds N fp32): views into a shortlist buffer."""
    small = N * (K // 256) * 144
    s = (small + 255) // 256 * 256
    return buf[:small].view(N, K // 256 * 144), buf[s:s + 4 * N].view(torch.float32)


def head_argmax(w_q8: torch.Tensor, shortlist: torch.Tensor | None, x: torch.Tensor, N: int, K: int,
                all_rows: bool = False, workspace: torch.Tensor | None = None, token: torch.Tensor | None = None,
                score: torch.Tensor | None = None, rows_scored: torch.Tensor | None = None, stream=None):
    """Greedy next token of each hidden-state row of x over a Q8_0 head (kq_head_argmax).
    Returns (token int32 [M], score fp32 [M], rows_scored int32 [1]) device tensors."""
    M = x.shape[0]
    dev = x.device
    if workspace is None:
        workspace = torch.empty(lib().kq_head_argmax_workspace_size(M, N), dtype=torch.uint8, device=dev)
    if token is None:
        token = torch.empty(M, dtype=torch.int32, device=dev)
    if score is None:
        score = torch.empty(M, dtype=torch.float32, device=dev)
    if rows_scored is None:
        rows_scored = torch.empty(1, dtype=torch.int32, device=dev)
    _check(lib().kq_head_argmax(w_q8.data_ptr(), shortlist.data_ptr() if shortlist is not None else None,
                                _x_dtype(x), x.data_ptr(), M, N, K, token.data_ptr(), score.data_ptr(),
                                rows_scored.data_ptr(), workspace.data_ptr(), workspace.numel(),
                                KQ_HEAD_ALL_ROWS if all_rows else 0, _stream(stream)))
    return token, score, rows_scored


def device_errors() -> int:
    """Read and clear the device error word (bit 0: a bounded in-kernel wait gave up)."""
    rc = lib().kq_device_errors()
    if rc < 0:
        _check(rc)
    return rc


def quantize(fmt, w: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """fp32 N x K device matrix -> N x row_bytes uint8 blocks, through kq_quantize."""
    N, K = w.shape
    if out is None:
        out = torch.empty((N, row_bytes(fmt, K)), dtype=torch.uint8, device=w.device)
    _check(lib().kq_quantize(_fmt(fmt), w.data_ptr(), out.data_ptr(), N, K, _stream(stream)))
    return out


class KVCacheC(ctypes.Structure):
    """Mirror of kq_kv_cache (include/kq.h)."""
    _fields_ = [("k", ctypes.POINTER(ctypes.c_void_p)), ("v", ctypes.POINTER(ctypes.c_void_p)),
                ("length", ctypes.c_int), ("capacity", ctypes.c_int)]


class KVCache:
    """Per-layer bf16 K and V arrays (capacity x kv_dim device tensors) and the cached length."""

    def __init__(self, n_layers: int, capacity: int, kv_dim: int, device="cuda", k=None, v=None):
        self.k = k if k is not None else [torch.zeros((capacity, kv_dim), dtype=torch.bfloat16, device=device)
                                          for _ in range(n_layers)]
        self.v = v if v is not None else [torch.zeros((capacity, kv_dim), dtype=torch.bfloat16, device=device)
                                          for _ in range(n_layers)]
        self.capacity, self.length = capacity, 0
        n = max(1, n_layers)
        self._ka = (ctypes.c_void_p * n)(*[t.data_ptr() for t in self.k])
        self._va = (ctypes.c_void_p * n)(*[t.data_ptr() for t in self.v])

    def c(self) -> KVCacheC:
        return KVCacheC(ctypes.cast(self._ka, ctypes.POINTER(ctypes.c_void_p)),
                        ctypes.cast(self._va, ctypes.POINTER(ctypes.c_void_p)), self.length, self.capacity)


class DecodeModel:
    """A dense decoder whose weights are block-quantized device tensors (kq_decode_step).

    layers: list of (w_qkv, w_o, w_gate_up, w_down) uint8 CUDA tensors; head: uint8 CUDA tensor.
    The model struct and pointer arrays are kept alive by this object."""

    def __init__(self, n_layers, hidden, q_dim, kv_dim, head_dim, ffn, vocab, layers, head,
                 layer_fmt="q4_k", head_fmt="q8_0", eps=1e-6):
        self.layers, self.head = layers, head
        n = max(1, n_layers)
        self._arrs = [(ctypes.c_void_p * n)(*[lay[i].data_ptr() for lay in layers]) for i in range(4)]
        self.c = DecodeModelC(n_layers, hidden, q_dim, kv_dim, head_dim, ffn, vocab, _fmt(layer_fmt),
                              _fmt(head_fmt), eps,
                              *[ctypes.cast(a, ctypes.POINTER(ctypes.c_void_p)) for a in self._arrs],
                              head.data_ptr())
        self.hidden, self.vocab = hidden, vocab

    def workspace_size(self, M: int) -> int:
        return lib().kq_decode_workspace_size(ctypes.byref(self.c), M)

    def step(self, x: torch.Tensor, logits: torch.Tensor | None = None,
             workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """logits (M x vocab fp32) for M bf16 token rows x (M x hidden)."""
        M = x.shape[0]
        if logits is None:
            logits = torch.empty((M, self.vocab), dtype=torch.float32, device=x.device)
        if workspace is None:
            workspace = torch.empty(self.workspace_size(M), dtype=torch.uint8, device=x.device)
        _check(lib().kq_decode_step(ctypes.byref(self.c), x.data_ptr(), logits.data_ptr(), M,
                                    workspace.data_ptr(), workspace.numel(), _stream(stream)))
        return logits

    def step_trace(self, x: torch.Tensor, stream=None):
        """kq_decode_step_trace: (logits, trace) where trace holds every op's output as torch
        device tensors: "h0", "x0", and per layer l a dict "layers"[l] with "qkv", "o_in", "y_o",
        "h_mid", "x_mid", "gu", "act", "y_d", "h_out", "x_out" (bf16 fields as int16 bits)."""
        M = x.shape[0]
        c = self.c
        D, Q, KV, F = c.hidden, c.q_dim, c.kv_dim, c.ffn
        logits = torch.empty((M, self.vocab), dtype=torch.float32, device=x.device)
        ws = torch.empty(self.workspace_size(M), dtype=torch.uint8, device=x.device)
        need = lib().kq_decode_trace_size(ctypes.byref(c), M)
        buf = torch.empty(need, dtype=torch.uint8, device=x.device)
        _check(lib().kq_decode_step_trace(ctypes.byref(c), x.data_ptr(), logits.data_ptr(), M, ws.data_ptr(),
                                          ws.numel(), buf.data_ptr(), buf.numel(), _stream(stream)))
        al = lambda n: (n + 255) // 256 * 256
        off = 0

        def take(cols, f32):
            nonlocal off
            nb = M * cols * (4 if f32 else 2)
            t = buf[off:off + nb].view(torch.float32 if f32 else torch.int16).view(M, cols)
            off = al(off + nb)
            return t

        tr = {"h0": take(D, True), "x0": take(D, False), "layers": []}
        for _ in range(c.n_layers):
            tr["layers"].append({"qkv": take(Q + 2 * KV, True), "o_in": take(Q, False), "y_o": take(D, True),
                                 "h_mid": take(D, True), "x_mid": take(D, False), "gu": take(2 * F, True),
                                 "act": take(F, False), "y_d": take(D, True), "h_out": take(D, True),
                                 "x_out": take(D, False)})
        assert off <= need
        return logits, tr

    def attn_workspace_size(self, M: int, L: int) -> int:
        return lib().kq_decode_attn_workspace_size(ctypes.byref(self.c), M, L)

    def step_attn(self, x: torch.Tensor, cache: "KVCache", mask: torch.Tensor | None = None,
                  logits: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                  stream=None) -> torch.Tensor:
        """kq_decode_step_attn: logits for M bf16 token rows attending to cache.length cached
        positions (the window's k, v are written at rows length..length+M-1; length is not
        advanced here). mask: None (causal) or M int32 words."""
        M = x.shape[0]
        if logits is None:
            logits = torch.empty((M, self.vocab), dtype=torch.float32, device=x.device)
        if workspace is None:
            workspace = torch.empty(self.attn_workspace_size(M, cache.length), dtype=torch.uint8, device=x.device)
        cc = cache.c()
        _check(lib().kq_decode_step_attn(ctypes.byref(self.c), ctypes.byref(cc), x.data_ptr(), logits.data_ptr(), M,
                                         mask.data_ptr() if mask is not None else None, workspace.data_ptr(),
                                         workspace.numel(), _stream(stream)))
        return logits

    def step_static(self, x: torch.Tensor, logits: torch.Tensor, stream=None) -> torch.Tensor:
        """The same step through kq_decode_step_static (library-held scratch, no allocation)."""
        _check(lib().kq_decode_step_static(ctypes.byref(self.c), x.data_ptr(), logits.data_ptr(),
                                           x.shape[0], _stream(stream)))
        return logits
