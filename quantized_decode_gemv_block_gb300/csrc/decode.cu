// Decode step of a dense transformer on block-quantized weights (the composition of the
// GEMVs; Kinetic README, "What makes it fast": a decode step is hundreds of small kernels,
// recorded once and replayed with one launch per token; all of a dense model's weights
// are read once per token).
//
// Model (per layer): x = RMSNorm(h) -> [q k v] = x Wqkv^T -> attention stand-in (each row
// attends only to itself, so the output of head hq is v of kv head hq / (n_q / n_kv)) ->
// h += o Wo^T -> x = RMSNorm(h) -> [g u] = x Wgu^T -> a = silu(g) * u -> h += a Wd^T.
// Then logits = RMSNorm(h) Whead^T. RMSNorm has unit weight. Activations entering a GEMV
// are rounded to bf16 (round to nearest even); the residual stream h and every GEMV
// output stay fp32.
//
// Every kernel here takes part in programmatic dependent launch: it lets the next launch
// begin at once and waits for the previous grid before touching what that grid wrote.
// The GEMVs are launched with KQ_OVERLAP_PREVIOUS (no kernel of the step writes weights),
// so each one streams its weights while the glue before it still runs.
#include <cuda_bf16.h>

#include <cmath>
#include <vector>

#include "kq.h"
#include "kq_device.cuh"
#include "kq_internal.h"

namespace kq {
namespace {

constexpr int kGlueThreads = 256;

__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint16_t f2bf(float v) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

// Fixed-order block sum (same tree for every launch): warp butterflies, then warp 0.
__device__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    v = lane < (kGlueThreads / 32) ? red[lane] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    if (lane == 0) red[0] = v;
  }
  __syncthreads();
  const float r = red[0];
  __syncthreads();
  return r;
}

// h[j] = x[j] (bf16 -> fp32) if x != null; then, if add != null, h[j] += add[j]; then
// out[j] = bf16(h[j] / sqrt(mean(h[j]^2) + eps)). One CTA per token; D % 4 == 0 (the hidden
// size is a multiple of 256). Thread t takes the 4-element chunks t, t + 256, ... of the row;
// the first kNormChunks of them stay in registers, so every load of a row up to 4096 wide is
// in flight at once (this kernel sits between two GEMVs on the decode step's critical path)
// and the normalisation reads nothing back. Sum of squares: per thread in chunk order,
// elements in order, then a fixed block tree.
constexpr int kNormChunks = 4;
__global__ void __launch_bounds__(kGlueThreads) add_rmsnorm_kernel(float* __restrict__ h,
                                                                   const uint16_t* __restrict__ x,
                                                                   const float* __restrict__ add,
                                                                   uint16_t* __restrict__ out, int D,
                                                                   float eps) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[kGlueThreads / 32];
  const int j = blockIdx.x, nch = D / 4;
  float* hj = h + (long long)j * D;
  const float* aj = add ? add + (long long)j * D : nullptr;
  const uint16_t* xj = x ? x + (long long)j * D : nullptr;
  float4 v[kNormChunks], a[kNormChunks];
#pragma unroll
  for (int r = 0; r < kNormChunks; ++r) {
    const int c = threadIdx.x + r * kGlueThreads;
    v[r] = a[r] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (c < nch) {
      if (xj) {
        const uint2 u = *reinterpret_cast<const uint2*>(xj + 4 * c);
        v[r] = make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                           __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
      } else {
        v[r] = *reinterpret_cast<const float4*>(hj + 4 * c);
      }
      if (aj) a[r] = *reinterpret_cast<const float4*>(aj + 4 * c);
    }
  }
  float ss = 0.f;
#pragma unroll
  for (int r = 0; r < kNormChunks; ++r) {
    const int c = threadIdx.x + r * kGlueThreads;
    if (c < nch) {
      if (aj) {
        v[r].x = v[r].x + a[r].x;
        v[r].y = v[r].y + a[r].y;
        v[r].z = v[r].z + a[r].z;
        v[r].w = v[r].w + a[r].w;
      }
      *reinterpret_cast<float4*>(hj + 4 * c) = v[r];
      ss = __fmaf_rn(v[r].x, v[r].x, ss);
      ss = __fmaf_rn(v[r].y, v[r].y, ss);
      ss = __fmaf_rn(v[r].z, v[r].z, ss);
      ss = __fmaf_rn(v[r].w, v[r].w, ss);
    }
  }
  for (int c = threadIdx.x + kNormChunks * kGlueThreads; c < nch; c += kGlueThreads) {  // rows > 4096
    float4 w = xj ? make_float4(0.f, 0.f, 0.f, 0.f) : *reinterpret_cast<const float4*>(hj + 4 * c);
    if (xj) {
      const uint2 u = *reinterpret_cast<const uint2*>(xj + 4 * c);
      w = make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u), __uint_as_float(u.y << 16),
                      __uint_as_float(u.y & 0xFFFF0000u));
    }
    if (aj) {
      const float4 b = *reinterpret_cast<const float4*>(aj + 4 * c);
      w.x = w.x + b.x;
      w.y = w.y + b.y;
      w.z = w.z + b.z;
      w.w = w.w + b.w;
    }
    *reinterpret_cast<float4*>(hj + 4 * c) = w;
    ss = __fmaf_rn(w.x, w.x, ss);
    ss = __fmaf_rn(w.y, w.y, ss);
    ss = __fmaf_rn(w.z, w.z, ss);
    ss = __fmaf_rn(w.w, w.w, ss);
  }
  const float tot = block_sum(ss, red);
  const float inv = 1.0f / sqrtf(tot / (float)D + eps);
#pragma unroll
  for (int r = 0; r < kNormChunks; ++r) {
    const int c = threadIdx.x + r * kGlueThreads;
    if (c < nch)
      *reinterpret_cast<uint2*>(out + (long long)j * D + 4 * c) =
          make_uint2((uint32_t)f2bf(v[r].x * inv) | ((uint32_t)f2bf(v[r].y * inv) << 16),
                     (uint32_t)f2bf(v[r].z * inv) | ((uint32_t)f2bf(v[r].w * inv) << 16));
  }
  for (int c = threadIdx.x + kNormChunks * kGlueThreads; c < nch; c += kGlueThreads) {
    const float4 w = *reinterpret_cast<const float4*>(hj + 4 * c);
    *reinterpret_cast<uint2*>(out + (long long)j * D + 4 * c) =
        make_uint2((uint32_t)f2bf(w.x * inv) | ((uint32_t)f2bf(w.y * inv) << 16),
                   (uint32_t)f2bf(w.z * inv) | ((uint32_t)f2bf(w.w * inv) << 16));
  }
}

// out[j][hq*hd + d] = bf16(qkv[j][q_dim + kv_dim + (hq / group)*hd + d]): the attention
// stand-in with a context of one token (softmax weight 1 on the token's own value).
__global__ void __launch_bounds__(kGlueThreads) gqa_expand_kernel(const float* __restrict__ qkv,
                                                                  uint16_t* __restrict__ out, int M,
                                                                  int q_dim, int kv_dim, int hd,
                                                                  int group) {
  pdl_trigger();
  pdl_wait();
  const int qkv_dim = q_dim + 2 * kv_dim;
  const long long total = (long long)M * q_dim;
  for (long long e = blockIdx.x * (long long)kGlueThreads + threadIdx.x; e < total;
       e += (long long)gridDim.x * kGlueThreads) {
    const int j = (int)(e / q_dim), c = (int)(e - (long long)j * q_dim);
    const int hq = c / hd, d = c - hq * hd;
    out[e] = f2bf(qkv[(long long)j * qkv_dim + q_dim + kv_dim + (hq / group) * hd + d]);
  }
}

// out[j][i] = bf16(silu(gu[j][i]) * gu[j][F + i]), silu(g) = g / (1 + exp(-g)).
__global__ void __launch_bounds__(kGlueThreads) swiglu_kernel(const float* __restrict__ gu,
                                                              uint16_t* __restrict__ out, int M, int F) {
  pdl_trigger();
  pdl_wait();
  const long long total = (long long)M * F;
  for (long long e = blockIdx.x * (long long)kGlueThreads + threadIdx.x; e < total;
       e += (long long)gridDim.x * kGlueThreads) {
    const int j = (int)(e / F), i = (int)(e - (long long)j * F);
    out[e] = silu_mul_bf16(gu[(long long)j * 2 * F + i], gu[(long long)j * 2 * F + F + i]);
  }
}

// Rows L..L+M-1 of a layer's cache: k = bf16(qkv[:, q_dim : q_dim+kv_dim]), v = the next kv_dim.
__global__ void __launch_bounds__(kGlueThreads) kv_append_kernel(const float* __restrict__ qkv,
                                                                 uint16_t* __restrict__ kc, uint16_t* __restrict__ vc,
                                                                 int M, int q_dim, int kv_dim, int L) {
  pdl_trigger();
  pdl_wait();
  const int qkv_dim = q_dim + 2 * kv_dim;
  const long long total = (long long)M * kv_dim;
  for (long long e = blockIdx.x * (long long)kGlueThreads + threadIdx.x; e < total;
       e += (long long)gridDim.x * kGlueThreads) {
    const int j = (int)(e / kv_dim), c = (int)(e - (long long)j * kv_dim);
    const float* row = qkv + (long long)j * qkv_dim + q_dim;
    kc[(long long)(L + j) * kv_dim + c] = f2bf(row[c]);
    vc[(long long)(L + j) * kv_dim + c] = f2bf(row[kv_dim + c]);
  }
}

template <class... Args>
cudaError_t launch_pdl(void (*kern)(Args...), int grid, cudaStream_t s, bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kGlueThreads, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

size_t al256(size_t v) { return (v + 255) & ~size_t(255); }

struct Ws {  // workspace carve-up
  float* h;     // M x hidden      residual stream
  uint16_t* x;  // M x max(hidden, q_dim, ffn) bf16 GEMV input
  uint16_t* x2; // M x max(q_dim, ffn) bf16: the input of Wo and of the down projection
  float* qkv;   // M x (q_dim + 2 kv_dim)
  float* y;     // M x hidden      o / down outputs
  float* gu;    // M x 2 ffn
  size_t bytes;
};

Ws carve(const kq_decode_model* m, int M, void* base) {
  Ws w;
  const int xw = std::max(m->hidden, std::max(m->q_dim, m->ffn));
  size_t off = 0;
  auto take = [&](size_t bytes) {
    void* p = base ? static_cast<uint8_t*>(base) + off : nullptr;
    off = al256(off + bytes);
    return p;
  };
  w.h = static_cast<float*>(take(sizeof(float) * (size_t)M * m->hidden));
  w.x = static_cast<uint16_t*>(take(sizeof(uint16_t) * (size_t)M * xw));
  w.x2 = static_cast<uint16_t*>(take(sizeof(uint16_t) * (size_t)M * std::max(m->q_dim, m->ffn)));
  w.qkv = static_cast<float*>(take(sizeof(float) * (size_t)M * (m->q_dim + 2 * m->kv_dim)));
  w.y = static_cast<float*>(take(sizeof(float) * (size_t)M * m->hidden));
  w.gu = static_cast<float*>(take(sizeof(float) * (size_t)M * 2 * m->ffn));
  w.bytes = off;
  return w;
}

// The trace buffer of kq_decode_step_trace: h0 and x0, then per layer qkv, o_in, y_o, h_mid,
// x_mid, gu, act, y_d, h_out, x_out, each field 256-byte aligned, in that order.
struct TraceLayout {
  size_t h0, x0, layer0, layer_bytes, bytes;
  size_t qkv, o_in, y_o, h_mid, x_mid, gu, act, y_d, h_out, x_out;  // offsets within a layer
};

TraceLayout trace_layout(const kq_decode_model* m, int M) {
  TraceLayout t;
  const size_t D = m->hidden, QKV = m->q_dim + 2 * m->kv_dim, F = m->ffn, Q = m->q_dim;
  size_t off = 0;
  auto take = [&](size_t bytes) { const size_t o = off; off = al256(off + bytes); return o; };
  t.h0 = take(4 * M * D);
  t.x0 = take(2 * M * D);
  t.layer0 = off;
  off = 0;
  t.qkv = take(4 * M * QKV);
  t.o_in = take(2 * M * Q);
  t.y_o = take(4 * M * D);
  t.h_mid = take(4 * M * D);
  t.x_mid = take(2 * M * D);
  t.gu = take(4 * M * 2 * F);
  t.act = take(2 * M * F);
  t.y_d = take(4 * M * D);
  t.h_out = take(4 * M * D);
  t.x_out = take(2 * M * D);
  t.layer_bytes = off;
  t.bytes = t.layer0 + (size_t)m->n_layers * t.layer_bytes;
  return t;
}

}  // namespace

size_t decode_trace_size(const kq_decode_model* m, int M) { return trace_layout(m, M).bytes; }

int decode_check(const kq_decode_model* m, int M, std::string* err) {
  if (!m) { *err = "model is NULL"; return -1; }
  if (m->n_layers < 0 || m->hidden <= 0 || m->q_dim <= 0 || m->kv_dim <= 0 || m->head_dim <= 0 ||
      m->ffn <= 0 || m->vocab <= 0) { *err = "model dimensions must be positive"; return -1; }
  if (m->q_dim % m->head_dim || m->kv_dim % m->head_dim) { *err = "q_dim and kv_dim must be multiples of head_dim"; return -1; }
  if ((m->q_dim / m->head_dim) % (m->kv_dim / m->head_dim)) { *err = "query heads must be a multiple of kv heads"; return -1; }
  if (m->hidden % 256 || m->q_dim % 256 || m->ffn % 256) { *err = "hidden, q_dim and ffn must be multiples of 256"; return -1; }
  if (M < 1 || M > 16) { *err = "M must be in 1..16"; return -1; }
  if (m->n_layers > 0 && (!m->w_qkv || !m->w_o || !m->w_gate_up || !m->w_down)) { *err = "layer weight arrays are NULL"; return -1; }
  if (!m->w_head) { *err = "w_head is NULL"; return -1; }
  return 0;
}

size_t decode_workspace_size(const kq_decode_model* m, int M) { return carve(m, M, nullptr).bytes; }

int decode_step(const kq_decode_model* m, const uint16_t* x, float* logits, int M, void* ws, int num_sms,
                cudaStream_t s, std::string* err, void* trace) {
  const Ws w = carve(m, M, ws);
  const TraceLayout tl = trace_layout(m, M);
  // trace: after an op, a device-to-device copy of what it wrote (stream-ordered; the kernels
  // and their arguments are those of the untraced step)
  auto keep = [&](size_t off, const void* src, size_t bytes) -> int {
    if (!trace) return 0;
    const cudaError_t e = cudaMemcpyAsync(static_cast<uint8_t*>(trace) + off, src, bytes, cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) { *err = std::string("trace copy: ") + cudaGetErrorString(e); return -1; }
    return 0;
  };
  const size_t MD = (size_t)M * m->hidden;
  const int qkv_dim = m->q_dim + 2 * m->kv_dim;
  const int group = (m->q_dim / m->head_dim) / (m->kv_dim / m->head_dim);
  auto rowb = [](int fmt, int K) { return (long long)kq_row_bytes(fmt, K); };
  auto ew_grid = [&](long long n) { return (int)std::min<long long>(4 * (long long)num_sms, (n + kGlueThreads - 1) / kGlueThreads); };
  auto ck = [&](cudaError_t e, const char* what) {
    if (e != cudaSuccess) { *err = std::string(what) + ": " + cudaGetErrorString(e); return -1; }
    return 0;
  };
  auto gemv = [&](int fmt, const void* wt, const uint16_t* xin, float* y, int N, int K,
                  const GemvEpilogue* epi = nullptr) {
    return launch_gemv_mma(fmt, wt, xin, y, M, N, K, rowb(fmt, K), num_sms, s, true, err, epi);
  };
  // The attention stand-in and the SwiGLU run inside the GEMVs that produce their inputs when
  // the streaming kernel takes those shapes (its epilogue writes the bf16 input of Wo, resp. of
  // the down projection); otherwise as separate kernels. Both give the same bits.
  GemvEpilogue expand, swiglu;
  expand.kind = 1;
  expand.out = w.x2;
  expand.v0 = m->q_dim + m->kv_dim;
  expand.vn = m->kv_dim;
  expand.hd = m->head_dim;
  expand.group = group;
  expand.out_w = m->q_dim;
  swiglu.kind = 2;
  swiglu.out = w.x2;
  const bool fuse_expand = gemv_epilogue_ok(m->layer_fmt, qkv_dim, m->hidden, 1, num_sms);
  const bool fuse_swiglu = gemv_epilogue_ok(m->layer_fmt, 2 * m->ffn, m->hidden, 2, num_sms);
  // h = x (bf16 -> fp32); x_norm = RMSNorm(h)
  if (ck(launch_pdl(add_rmsnorm_kernel, M, s, false, w.h, x, (const float*)nullptr, w.x, m->hidden, m->rms_eps),
         "add_rmsnorm"))
    return -1;
  if (keep(tl.h0, w.h, 4 * MD) || keep(tl.x0, w.x, 2 * MD)) return -1;
  for (int l = 0; l < m->n_layers; ++l) {
    const size_t L0 = tl.layer0 + (size_t)l * tl.layer_bytes;
    if (gemv(m->layer_fmt, m->w_qkv[l], w.x, w.qkv, qkv_dim, m->hidden, fuse_expand ? &expand : nullptr)) return -1;
    if (keep(L0 + tl.qkv, w.qkv, 4 * (size_t)M * qkv_dim)) return -1;
    if (!fuse_expand &&
        ck(launch_pdl(gqa_expand_kernel, ew_grid((long long)M * m->q_dim), s, true, (const float*)w.qkv, w.x2, M,
                      m->q_dim, m->kv_dim, m->head_dim, group),
           "gqa_expand"))
      return -1;
    if (keep(L0 + tl.o_in, w.x2, 2 * (size_t)M * m->q_dim)) return -1;
    if (gemv(m->layer_fmt, m->w_o[l], w.x2, w.y, m->hidden, m->q_dim)) return -1;
    if (keep(L0 + tl.y_o, w.y, 4 * MD)) return -1;
    if (ck(launch_pdl(add_rmsnorm_kernel, M, s, true, w.h, (const uint16_t*)nullptr, (const float*)w.y, w.x,
                      m->hidden, m->rms_eps),
           "add_rmsnorm"))
      return -1;
    if (keep(L0 + tl.h_mid, w.h, 4 * MD) || keep(L0 + tl.x_mid, w.x, 2 * MD)) return -1;
    if (fuse_swiglu) {  // gate|up outputs in fp32 only when traced
      if (gemv(m->layer_fmt, m->w_gate_up[l], w.x, trace ? w.gu : nullptr, 2 * m->ffn, m->hidden, &swiglu)) return -1;
      if (keep(L0 + tl.gu, w.gu, 4 * (size_t)M * 2 * m->ffn)) return -1;
    } else {
      if (gemv(m->layer_fmt, m->w_gate_up[l], w.x, w.gu, 2 * m->ffn, m->hidden)) return -1;
      if (keep(L0 + tl.gu, w.gu, 4 * (size_t)M * 2 * m->ffn)) return -1;
      if (ck(launch_pdl(swiglu_kernel, ew_grid((long long)M * m->ffn), s, true, (const float*)w.gu, w.x2, M, m->ffn),
             "swiglu"))
        return -1;
    }
    if (keep(L0 + tl.act, w.x2, 2 * (size_t)M * m->ffn)) return -1;
    if (gemv(m->layer_fmt, m->w_down[l], w.x2, w.y, m->hidden, m->ffn)) return -1;
    if (keep(L0 + tl.y_d, w.y, 4 * MD)) return -1;
    if (ck(launch_pdl(add_rmsnorm_kernel, M, s, true, w.h, (const uint16_t*)nullptr, (const float*)w.y, w.x,
                      m->hidden, m->rms_eps),
           "add_rmsnorm"))
      return -1;
    if (keep(L0 + tl.h_out, w.h, 4 * MD) || keep(L0 + tl.x_out, w.x, 2 * MD)) return -1;
  }
  return gemv(m->head_fmt, m->w_head, w.x, logits, m->vocab, m->hidden);
}

size_t decode_attn_workspace_size(const kq_decode_model* m, int M, int L) {
  return al256(carve(m, M, nullptr).bytes) +
         attention_workspace(M, L, m->q_dim / m->head_dim, m->kv_dim / m->head_dim, m->head_dim);
}

int decode_step_attn(const kq_decode_model* m, const kq_kv_cache* c, const uint16_t* x, float* logits, int M,
                     const uint32_t* mask, void* ws, int num_sms, cudaStream_t s, std::string* err) {
  const Ws w = carve(m, M, ws);
  void* aws = static_cast<uint8_t*>(ws) + al256(w.bytes);
  const int qkv_dim = m->q_dim + 2 * m->kv_dim;
  const int n_q = m->q_dim / m->head_dim, n_kv = m->kv_dim / m->head_dim;
  const float scale = 1.0f / sqrtf((float)m->head_dim);
  auto rowb = [](int fmt, int K) { return (long long)kq_row_bytes(fmt, K); };
  auto ew_grid = [&](long long n) { return (int)std::min<long long>(4 * (long long)num_sms, (n + kGlueThreads - 1) / kGlueThreads); };
  auto ck = [&](cudaError_t e, const char* what) {
    if (e != cudaSuccess) { *err = std::string(what) + ": " + cudaGetErrorString(e); return -1; }
    return 0;
  };
  auto gemv = [&](int fmt, const void* wt, const uint16_t* xin, float* y, int N, int K,
                  const GemvEpilogue* epi = nullptr) {
    return launch_gemv_mma(fmt, wt, xin, y, M, N, K, rowb(fmt, K), num_sms, s, true, err, epi);
  };
  GemvEpilogue swiglu;  // the SwiGLU inside the gate|up GEMV when its plan allows (see decode_step)
  swiglu.kind = 2;
  swiglu.out = w.x2;
  const bool fuse_swiglu = gemv_epilogue_ok(m->layer_fmt, 2 * m->ffn, m->hidden, 2, num_sms);
  // the window's k and v go into the cache from the qkv GEMV's stores (same bf16 rounding as the
  // append kernel, which runs instead where the streaming kernel does not take the shape)
  GemvEpilogue append;
  append.kind = 3;
  append.v0 = m->q_dim;
  append.hd = m->kv_dim;
  append.row0 = c->length;
  const bool fuse_append = gemv_epilogue_ok(m->layer_fmt, qkv_dim, m->hidden, 3, num_sms);
  if (ck(launch_pdl(add_rmsnorm_kernel, M, s, false, w.h, x, (const float*)nullptr, w.x, m->hidden, m->rms_eps),
         "add_rmsnorm"))
    return -1;
  for (int l = 0; l < m->n_layers; ++l) {
    uint16_t* kc = static_cast<uint16_t*>(c->k[l]);
    uint16_t* vc = static_cast<uint16_t*>(c->v[l]);
    append.out = kc;
    append.out_b = vc;
    if (gemv(m->layer_fmt, m->w_qkv[l], w.x, w.qkv, qkv_dim, m->hidden, fuse_append ? &append : nullptr)) return -1;
    if (!fuse_append &&
        ck(launch_pdl(kv_append_kernel, ew_grid((long long)M * m->kv_dim), s, true, (const float*)w.qkv, kc, vc, M,
                      m->q_dim, m->kv_dim, c->length),
           "kv_append"))
      return -1;
    // attention over the cache; its output goes to the Wo GEMV's input as bf16. A plain launch
    // here: starting its CTAs early behind the small append kernel measured slower at M = 8
    if (launch_attention(w.qkv, qkv_dim, kc, vc, nullptr, w.x, M, c->length, n_q, n_kv, m->head_dim, mask, scale,
                         aws, s, false, err))
      return -1;
    if (gemv(m->layer_fmt, m->w_o[l], w.x, w.y, m->hidden, m->q_dim)) return -1;
    if (ck(launch_pdl(add_rmsnorm_kernel, M, s, true, w.h, (const uint16_t*)nullptr, (const float*)w.y, w.x,
                      m->hidden, m->rms_eps),
           "add_rmsnorm"))
      return -1;
    if (fuse_swiglu) {
      if (gemv(m->layer_fmt, m->w_gate_up[l], w.x, nullptr, 2 * m->ffn, m->hidden, &swiglu)) return -1;
    } else {
      if (gemv(m->layer_fmt, m->w_gate_up[l], w.x, w.gu, 2 * m->ffn, m->hidden)) return -1;
      if (ck(launch_pdl(swiglu_kernel, ew_grid((long long)M * m->ffn), s, true, (const float*)w.gu, w.x2, M, m->ffn),
             "swiglu"))
        return -1;
    }
    if (gemv(m->layer_fmt, m->w_down[l], w.x2, w.y, m->hidden, m->ffn)) return -1;
    if (ck(launch_pdl(add_rmsnorm_kernel, M, s, true, w.h, (const uint16_t*)nullptr, (const float*)w.y, w.x,
                      m->hidden, m->rms_eps),
           "add_rmsnorm"))
      return -1;
  }
  return gemv(m->head_fmt, m->w_head, w.x, logits, m->vocab, m->hidden);
}

}  // namespace kq
