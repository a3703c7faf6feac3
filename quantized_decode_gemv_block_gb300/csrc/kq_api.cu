// C-ABI boundary of libkq: argument checks, error reporting and kernel dispatch.
// The declarations, their sources and their contracts are in include/kq.h.
#include <cstdint>
#include <cstdio>
#include <mutex>
#include <algorithm>
#include <string>

#include "kq.h"
#include "kq_internal.h"

namespace {

thread_local std::string g_err;

int fail(int code, const std::string& msg) {
  g_err = msg;
  return code;
}
int ok() {
  g_err.clear();
  return KQ_OK;
}

bool fmt_known(int fmt) {
  return fmt == KQ_Q8_0 || fmt == KQ_Q4_K || fmt == KQ_AFFINE4_G32 || fmt == KQ_Q5_K || fmt == KQ_Q6_K;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int sm_count(std::string* err) {
  static int cached[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    *err = std::string("cudaGetDevice: ") + cudaGetErrorString(e);
    return -1;
  }
  if (dev < 64 && cached[dev] > 0) return cached[dev];
  int n = 0;
  e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess || n <= 0) {
    *err = std::string("cudaDeviceGetAttribute: ") + cudaGetErrorString(e);
    return -1;
  }
  if (dev < 64) cached[dev] = n;
  return n;
}

// Shared checks of kq_gemv / kq_gemm; returns KQ_OK or an error (already recorded).
int check_common(int fmt, const void* w, int x_dtype, const void* x, const float* y, int M, int N,
                 int K) {
  if (!fmt_known(fmt)) return fail(KQ_ERR_UNSUPPORTED, "unknown block format " + std::to_string(fmt));
  if (x_dtype != KQ_F32 && x_dtype != KQ_BF16)
    return fail(KQ_ERR_UNSUPPORTED, "unknown activation dtype " + std::to_string(x_dtype));
  if (M < 0 || N < 0 || K < 0) return fail(KQ_ERR_ARG, "M, N and K must be >= 0");
  if (K % 256 != 0) return fail(KQ_ERR_ARG, "K must be a multiple of 256, got " + std::to_string(K));
  if (M == 0 || N == 0) return KQ_OK;
  if (y == nullptr) return fail(KQ_ERR_ARG, "y is NULL");
  if (!aligned(y, 4)) return fail(KQ_ERR_ARG, "y must be 4-byte aligned");
  if (K > 0) {
    if (w == nullptr || x == nullptr) return fail(KQ_ERR_ARG, "w_blocks or x is NULL");
    if (!aligned(w, 16)) return fail(KQ_ERR_ARG, "w_blocks must be 16-byte aligned");
    if (!aligned(x, 16)) return fail(KQ_ERR_ARG, "x must be 16-byte aligned");
  }
  return KQ_OK;
}

int gemv_impl(int fmt, const void* w, int x_dtype, const void* x, float* y, int M, int N, int K,
              cudaStream_t s, unsigned flags = 0) {
  if (flags & ~static_cast<unsigned>(KQ_OVERLAP_PREVIOUS))
    return fail(KQ_ERR_ARG, "unknown flag bits " + std::to_string(flags));
  if (M > 16) return fail(KQ_ERR_ARG, "kq_gemv takes M <= 16 token rows, got " + std::to_string(M));
  int rc = check_common(fmt, w, x_dtype, x, y, M, N, K);
  if (rc != KQ_OK) return rc;
  if (M == 0 || N == 0) return ok();
  if (K == 0) {
    const cudaError_t e = cudaMemsetAsync(y, 0, sizeof(float) * (size_t)M * (size_t)N, s);
    if (e != cudaSuccess) return fail(KQ_ERR_CUDA, std::string("cudaMemsetAsync: ") + cudaGetErrorString(e));
    return ok();
  }
  std::string err;
  const long long row_bytes = (long long)kq_row_bytes(fmt, K);
  if (x_dtype == KQ_BF16) {
    const int sms = sm_count(&err);
    if (sms < 0) return fail(KQ_ERR_CUDA, err);
    if (kq::launch_gemv_mma(fmt, w, x, y, M, N, K, row_bytes, sms, s, (flags & KQ_OVERLAP_PREVIOUS) != 0,
                            &err) != 0)
      return fail(KQ_ERR_CUDA, err);
  } else {
    if (kq::launch_gemv_f32(fmt, w, static_cast<const float*>(x), y, M, N, K, row_bytes, s,
                            (flags & KQ_OVERLAP_PREVIOUS) != 0, &err) != 0)
      return fail(KQ_ERR_CUDA, err);
  }
  return ok();
}

}  // namespace

extern "C" {

size_t kq_block_bytes(int fmt) {
  switch (fmt) {
    case KQ_Q8_0: return 34;
    case KQ_Q4_K: return 144;
    case KQ_Q5_K: return 176;
    case KQ_Q6_K: return 210;
    case KQ_AFFINE4_G32: return 20;
  }
  return 0;
}

size_t kq_block_weights(int fmt) {
  switch (fmt) {
    case KQ_Q8_0: return 32;
    case KQ_Q4_K: return 256;
    case KQ_Q5_K: return 256;
    case KQ_Q6_K: return 256;
    case KQ_AFFINE4_G32: return 32;
  }
  return 0;
}

size_t kq_row_bytes(int fmt, int K) {
  const size_t bw = kq_block_weights(fmt);
  if (bw == 0 || K < 0 || (size_t)K % bw != 0) return 0;
  return (size_t)K / bw * kq_block_bytes(fmt);
}

const char* kq_last_error(void) { return g_err.c_str(); }

const char* kq_version(void) { return "kq 0.1.0 (sm_103a)"; }

int kq_device_errors(void) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail(KQ_ERR_CUDA, std::string("cudaDeviceSynchronize: ") + cudaGetErrorString(e));
  std::string err;
  unsigned int v = kq::take_device_errors(&err);
  if (v == 0xFFFFFFFFu) return fail(KQ_ERR_CUDA, err);
  const unsigned int vt = kq::take_tc_errors();
  if (vt == 0xFFFFFFFFu) return fail(KQ_ERR_CUDA, "reading the prefill error word");
  v |= vt;
  ok();
  return static_cast<int>(v & 0x7FFFFFFFu);
}

int kq_gemv(int fmt, const void* w_blocks, int x_dtype, const void* x, float* y, int M, int N,
            int K, void* stream) {
  return gemv_impl(fmt, w_blocks, x_dtype, x, y, M, N, K, static_cast<cudaStream_t>(stream));
}

int kq_gemv_ex(int fmt, const void* w_blocks, int x_dtype, const void* x, float* y, int M, int N,
               int K, unsigned flags, void* stream) {
  return gemv_impl(fmt, w_blocks, x_dtype, x, y, M, N, K, static_cast<cudaStream_t>(stream), flags);
}

// kq_gemm's routes for M > 16. The tensor-core product exists for Q4_K x bf16; up to
// kGemvPassMaxM rows the GEMV kernels in passes of 16 token rows are faster than it (its
// weight unpacking, not M, sets its time below a few hundred rows) and keep every row's
// bits those of kq_gemv. Pairs without a tensor-core product take the passes at any M.
constexpr int kGemvPassRows = 16;
constexpr int kGemvPassMaxM = 32;
bool gemm_by_passes(int fmt, int x_dtype, int M) {
  return M > kGemvPassRows && (!(fmt == KQ_Q4_K && x_dtype == KQ_BF16) || M <= kGemvPassMaxM);
}

size_t kq_gemm_workspace_size(int fmt, int x_dtype, int M, int N, int K) {
  if (M <= 16 || N <= 0 || fmt != KQ_Q4_K || x_dtype != KQ_BF16 || K <= 0 || K % 256 != 0) return 0;
  if (gemm_by_passes(fmt, x_dtype, M)) return 0;
  return kq::gemm_tc_workspace(M, N, K);
}

int kq_gemm(int fmt, const void* w_blocks, int x_dtype, const void* x, float* y, int M, int N,
            int K, void* workspace, size_t ws_bytes, void* stream) {
  if (M <= 16)
    return gemv_impl(fmt, w_blocks, x_dtype, x, y, M, N, K, static_cast<cudaStream_t>(stream));
  int rc = check_common(fmt, w_blocks, x_dtype, x, y, M, N, K);
  if (rc != KQ_OK) return rc;
  if (N == 0) return ok();
  if (K == 0) {
    const cudaError_t e = cudaMemsetAsync(y, 0, sizeof(float) * (size_t)M * (size_t)N, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(KQ_ERR_CUDA, std::string("cudaMemsetAsync: ") + cudaGetErrorString(e));
    return ok();
  }
  if (gemm_by_passes(fmt, x_dtype, M)) {
    // token rows c..c+15 per pass; a pass may stream its weights while the previous one
    // drains (it writes other rows of y and never w)
    const size_t xe = x_dtype == KQ_BF16 ? 2 : 4;
    for (int c = 0; c < M; c += kGemvPassRows) {
      rc = gemv_impl(fmt, w_blocks, x_dtype, static_cast<const char*>(x) + (size_t)c * K * xe, y + (size_t)c * N,
                     std::min(kGemvPassRows, M - c), N, K, static_cast<cudaStream_t>(stream),
                     c > 0 ? static_cast<unsigned>(KQ_OVERLAP_PREVIOUS) : 0u);
      if (rc != KQ_OK) return rc;
    }
    return ok();
  }
  const size_t need = kq::gemm_tc_workspace(M, N, K);
  if (!workspace || ws_bytes < need || !aligned(workspace, 256))
    return fail(KQ_ERR_WORKSPACE, "workspace must be >= " + std::to_string(need) + " bytes, 256-byte aligned");
  std::string err;
  const int sms = sm_count(&err);
  if (sms < 0) return fail(KQ_ERR_CUDA, err);
  if (kq::launch_gemm_tc(w_blocks, x, y, M, N, K, (long long)kq_row_bytes(fmt, K), workspace, sms,
                         static_cast<cudaStream_t>(stream), &err) != 0)
    return fail(KQ_ERR_CUDA, err);
  return ok();
}

size_t kq_decode_workspace_size(const kq_decode_model* model, int M) {
  std::string err;
  if (kq::decode_check(model, M, &err) != 0) return 0;
  return kq::decode_workspace_size(model, M);
}

static int decode_step_impl(const kq_decode_model* model, const void* x, float* logits, int M, void* workspace,
                            size_t ws_bytes, void* trace, size_t trace_bytes, void* stream);

int kq_decode_step(const kq_decode_model* model, const void* x, float* logits, int M, void* workspace,
                   size_t ws_bytes, void* stream) {
  return decode_step_impl(model, x, logits, M, workspace, ws_bytes, nullptr, 0, stream);
}

size_t kq_decode_trace_size(const kq_decode_model* model, int M) {
  std::string err;
  if (kq::decode_check(model, M, &err) != 0) return 0;
  return kq::decode_trace_size(model, M);
}

int kq_decode_step_trace(const kq_decode_model* model, const void* x, float* logits, int M, void* workspace,
                         size_t ws_bytes, void* trace, size_t trace_bytes, void* stream) {
  if (!trace) return fail(KQ_ERR_ARG, "trace is NULL");
  return decode_step_impl(model, x, logits, M, workspace, ws_bytes, trace, trace_bytes, stream);
}

static int decode_step_impl(const kq_decode_model* model, const void* x, float* logits, int M, void* workspace,
                            size_t ws_bytes, void* trace, size_t trace_bytes, void* stream) {
  std::string err;
  if (kq::decode_check(model, M, &err) != 0) return fail(KQ_ERR_ARG, err);
  if (!fmt_known(model->layer_fmt) || !fmt_known(model->head_fmt))
    return fail(KQ_ERR_UNSUPPORTED, "unknown weight format in the model");
  if (!x || !logits) return fail(KQ_ERR_ARG, "x or logits is NULL");
  if (!aligned(x, 16) || !aligned(logits, 4)) return fail(KQ_ERR_ARG, "misaligned x or logits");
  const size_t need = kq::decode_workspace_size(model, M);
  if (!workspace || ws_bytes < need || !aligned(workspace, 256))
    return fail(KQ_ERR_WORKSPACE, "workspace must be >= " + std::to_string(need) + " bytes, 256-byte aligned");
  for (int l = 0; l < model->n_layers; ++l) {
    const void* ps[4] = {model->w_qkv[l], model->w_o[l], model->w_gate_up[l], model->w_down[l]};
    for (const void* p : ps)
      if (!p || !aligned(p, 16)) return fail(KQ_ERR_ARG, "layer " + std::to_string(l) + ": NULL or misaligned weights");
  }
  if (!aligned(model->w_head, 16)) return fail(KQ_ERR_ARG, "misaligned w_head");
  if (trace) {
    const size_t tneed = kq::decode_trace_size(model, M);
    if (trace_bytes < tneed || !aligned(trace, 256))
      return fail(KQ_ERR_ARG, "trace must be >= " + std::to_string(tneed) + " bytes, 256-byte aligned");
  }
  const int sms = sm_count(&err);
  if (sms < 0) return fail(KQ_ERR_CUDA, err);
  if (kq::decode_step(model, static_cast<const uint16_t*>(x), logits, M, workspace, sms,
                      static_cast<cudaStream_t>(stream), &err, trace) != 0)
    return fail(KQ_ERR_CUDA, err);
  return ok();
}

static int attention_check(int M, int L, int n_q, int n_kv, int head_dim, std::string* err) {
  if (M < 1 || M > 32) { *err = "M must be in 1..32 (the window's tokens)"; return -1; }
  if (L < 0 || L > 65000) { *err = "L must be in 0..65000"; return -1; }
  if (n_q < 1 || n_kv < 1 || n_q % n_kv) { *err = "n_q must be a positive multiple of n_kv"; return -1; }
  if (head_dim != 64 && head_dim != 128) { *err = "head_dim must be 64 or 128"; return -1; }
  if ((n_q / n_kv) * M > 128) { *err = "(n_q / n_kv) * M must be <= 128"; return -1; }
  return 0;
}

size_t kq_attention_workspace_size(int M, int L, int n_q, int n_kv, int head_dim) {
  std::string err;
  if (attention_check(M, L, n_q, n_kv, head_dim, &err) != 0) return 0;
  return kq::attention_workspace(M, L, n_q, n_kv, head_dim);
}

int kq_attention(const float* q, const void* k_cache, const void* v_cache, float* o, int M, int L, int n_q,
                 int n_kv, int head_dim, const unsigned int* mask, float scale, void* workspace, size_t ws_bytes,
                 void* stream) {
  std::string err;
  if (attention_check(M, L, n_q, n_kv, head_dim, &err) != 0) return fail(KQ_ERR_ARG, err);
  if (!q || !k_cache || !v_cache || !o) return fail(KQ_ERR_ARG, "q, k_cache, v_cache or o is NULL");
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(o, 4) || (mask && !aligned(mask, 4)))
    return fail(KQ_ERR_ARG, "misaligned q, k_cache, v_cache, o or mask");
  const size_t need = kq::attention_workspace(M, L, n_q, n_kv, head_dim);
  if (!workspace || ws_bytes < need || !aligned(workspace, 256))
    return fail(KQ_ERR_WORKSPACE, "workspace must be >= " + std::to_string(need) + " bytes, 256-byte aligned");
  if (kq::launch_attention(q, n_q * head_dim, static_cast<const uint16_t*>(k_cache),
                           static_cast<const uint16_t*>(v_cache), o, nullptr, M, L, n_q, n_kv, head_dim,
                           reinterpret_cast<const uint32_t*>(mask), scale, workspace,
                           static_cast<cudaStream_t>(stream), true, &err) != 0)
    return fail(KQ_ERR_CUDA, err);
  return ok();
}

static int decode_attn_check(const kq_decode_model* model, const kq_kv_cache* cache, int M, std::string* err) {
  if (kq::decode_check(model, M, err) != 0) return -1;
  if (!cache) { *err = "cache is NULL"; return -1; }
  const int n_q = model->q_dim / model->head_dim, n_kv = model->kv_dim / model->head_dim;
  if (attention_check(M, cache->length, n_q, n_kv, model->head_dim, err) != 0) return -1;
  if ((long long)cache->length + M > cache->capacity) { *err = "cache capacity < length + M"; return -1; }
  if (model->n_layers > 0 && (!cache->k || !cache->v)) { *err = "cache pointer arrays are NULL"; return -1; }
  for (int l = 0; l < model->n_layers; ++l)
    if (!cache->k[l] || !cache->v[l] || !aligned(cache->k[l], 16) || !aligned(cache->v[l], 16)) {
      *err = "layer " + std::to_string(l) + ": NULL or misaligned cache";
      return -1;
    }
  return 0;
}

size_t kq_decode_attn_workspace_size(const kq_decode_model* model, int M, int L) {
  std::string err;
  if (kq::decode_check(model, M, &err) != 0 || L < 0) return 0;
  const int n_q = model->q_dim / model->head_dim, n_kv = model->kv_dim / model->head_dim;
  if (attention_check(M, L, n_q, n_kv, model->head_dim, &err) != 0) return 0;
  return kq::decode_attn_workspace_size(model, M, L);
}

int kq_decode_step_attn(const kq_decode_model* model, const kq_kv_cache* cache, const void* x, float* logits,
                        int M, const unsigned int* mask, void* workspace, size_t ws_bytes, void* stream) {
  std::string err;
  if (decode_attn_check(model, cache, M, &err) != 0) return fail(KQ_ERR_ARG, err);
  if (!fmt_known(model->layer_fmt) || !fmt_known(model->head_fmt))
    return fail(KQ_ERR_UNSUPPORTED, "unknown weight format in the model");
  if (!x || !logits) return fail(KQ_ERR_ARG, "x or logits is NULL");
  if (!aligned(x, 16) || !aligned(logits, 4) || (mask && !aligned(mask, 4)))
    return fail(KQ_ERR_ARG, "misaligned x, logits or mask");
  const size_t need = kq::decode_attn_workspace_size(model, M, cache->length);
  if (!workspace || ws_bytes < need || !aligned(workspace, 256))
    return fail(KQ_ERR_WORKSPACE, "workspace must be >= " + std::to_string(need) + " bytes, 256-byte aligned");
  for (int l = 0; l < model->n_layers; ++l) {
    const void* ps[4] = {model->w_qkv[l], model->w_o[l], model->w_gate_up[l], model->w_down[l]};
    for (const void* p : ps)
      if (!p || !aligned(p, 16)) return fail(KQ_ERR_ARG, "layer " + std::to_string(l) + ": NULL or misaligned weights");
  }
  if (!aligned(model->w_head, 16)) return fail(KQ_ERR_ARG, "misaligned w_head");
  const int sms = sm_count(&err);
  if (sms < 0) return fail(KQ_ERR_CUDA, err);
  if (kq::decode_step_attn(model, cache, static_cast<const uint16_t*>(x), logits, M,
                           reinterpret_cast<const uint32_t*>(mask), workspace, sms, static_cast<cudaStream_t>(stream),
                           &err) != 0)
    return fail(KQ_ERR_CUDA, err);
  return ok();
}

int kq_quantize(int fmt, const float* w, void* w_blocks, int N, int K, void* stream) {
  if (!fmt_known(fmt)) return fail(KQ_ERR_UNSUPPORTED, "unknown block format " + std::to_string(fmt));
  if (N < 0 || K < 0) return fail(KQ_ERR_ARG, "N and K must be >= 0");
  if (kq_row_bytes(fmt, K) == 0 && K != 0)
    return fail(KQ_ERR_ARG, "K must be a multiple of the block's weight count");
  if ((long long)N * K == 0) return ok();
  if (w == nullptr || w_blocks == nullptr) return fail(KQ_ERR_ARG, "w or w_blocks is NULL");
  if (!aligned(w, 4) || !aligned(w_blocks, 2)) return fail(KQ_ERR_ARG, "misaligned w or w_blocks");
  std::string err;
  if (kq::launch_quantize(fmt, w, w_blocks, N, K, static_cast<cudaStream_t>(stream), &err) != 0)
    return fail(KQ_ERR_CUDA, err);
  return ok();
}

// ---- Shortlist output head ----
static bool head_shape_ok(int N, int K) { return N >= 1 && K >= 256 && K % 256 == 0; }

size_t kq_shortlist_bytes(int N, int K) {
  if (!head_shape_ok(N, K)) return 0;
  return kq::shortlist_bytes(N, K);
}

int kq_shortlist_build(const void* w_q8, int N, int K, void* shortlist, size_t bytes, void* stream) {
  if (!head_shape_ok(N, K)) return fail(KQ_ERR_ARG, "N must be >= 1 and K a positive multiple of 256");
  if (!w_q8 || !shortlist) return fail(KQ_ERR_ARG, "w_q8 or shortlist is NULL");
  if (!aligned(w_q8, 16) || !aligned(shortlist, 256))
    return fail(KQ_ERR_ARG, "w_q8 must be 16-byte aligned and shortlist 256-byte aligned");
  const size_t need = kq::shortlist_bytes(N, K);
  if (bytes < need) return fail(KQ_ERR_ARG, "shortlist buffer must be >= " + std::to_string(need) + " bytes");
  float* bound = reinterpret_cast<float*>(static_cast<uint8_t*>(shortlist) + kq::shortlist_small_bytes(N, K));
  std::string err;
  if (kq::launch_shortlist_build(w_q8, shortlist, bound, N, K, static_cast<cudaStream_t>(stream), &err) != 0)
    return fail(KQ_ERR_CUDA, err);
  return ok();
}

size_t kq_head_argmax_workspace_size(int M, int N) {
  if (M < 1 || M > 16 || N < 1) return 0;
  return kq::head_argmax_workspace(M, N);
}

int kq_head_argmax(const void* w_q8, const void* shortlist, int x_dtype, const void* x, int M, int N, int K,
                   int* token, float* score, unsigned int* rows_scored, void* workspace, size_t ws_bytes,
                   unsigned flags, void* stream) {
  if (flags & ~static_cast<unsigned>(KQ_HEAD_ALL_ROWS))
    return fail(KQ_ERR_ARG, "unknown flag bits " + std::to_string(flags));
  const bool all = (flags & KQ_HEAD_ALL_ROWS) != 0;
  if (M < 1 || M > 16) return fail(KQ_ERR_ARG, "M must be in 1..16, got " + std::to_string(M));
  if (!head_shape_ok(N, K)) return fail(KQ_ERR_ARG, "N must be >= 1 and K a positive multiple of 256");
  if (x_dtype != KQ_F32 && x_dtype != KQ_BF16)
    return fail(KQ_ERR_UNSUPPORTED, "unknown activation dtype " + std::to_string(x_dtype));
  if (!w_q8 || !x || !token || !score || (!all && !shortlist))
    return fail(KQ_ERR_ARG, "w_q8, shortlist, x, token or score is NULL");
  if (!aligned(w_q8, 16) || !aligned(x, 16) || (!all && !aligned(shortlist, 256)) || !aligned(token, 4) ||
      !aligned(score, 4) || (rows_scored && !aligned(rows_scored, 4)))
    return fail(KQ_ERR_ARG, "misaligned w_q8, shortlist, x, token, score or rows_scored");
  const size_t need = kq::head_argmax_workspace(M, N);
  if (!workspace || ws_bytes < need || !aligned(workspace, 256))
    return fail(KQ_ERR_WORKSPACE, "workspace must be >= " + std::to_string(need) + " bytes, 256-byte aligned");
  std::string err;
  const int sms = sm_count(&err);
  if (sms < 0) return fail(KQ_ERR_CUDA, err);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (!all) {  // the small copy's scores into the workspace's first M*N floats
    const int rc = gemv_impl(KQ_Q4_K, shortlist, x_dtype, x, static_cast<float*>(workspace), M, N, K, s);
    if (rc != KQ_OK) return rc;
  }
  if (kq::launch_head_select(w_q8, shortlist, x_dtype == KQ_BF16, x, M, N, K, token, score, rows_scored, workspace,
                             all, sms, s, &err) != 0)
    return fail(KQ_ERR_CUDA, err);
  return ok();
}

// ---- Decode step with library-owned scratch (kq_decode_step_static) ----
// The scratch lives in one file-scope device array, so no call allocates. Host code may
// not use the array's name as a device address (on the host it names a stand-in object):
// the address comes from cudaGetSymbolAddress, looked up by the first call on a device
// (with that device current) and cached together with the context that was current. A
// context torn down and created again (cudaDeviceReset) loads the module afresh and the
// array may move, so a call that finds a different current context looks it up again.
static __device__ __align__(256) unsigned char g_decode_scratch[KQ_DECODE_STATIC_SCRATCH_BYTES];

namespace {
std::mutex g_scratch_mu;
void* g_scratch_ptr[64] = {nullptr};
void* g_scratch_ctx[64] = {nullptr};

// The driver's cuCtxGetCurrent, reached through the runtime (the library does not link
// libcuda directly); null if the entry point cannot be found.
using CtxGetCurrentFn = int (*)(void**);
CtxGetCurrentFn ctx_get_current_fn() {
  static CtxGetCurrentFn fn = nullptr;
  static bool looked = false;
  if (!looked) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
    looked = true;
  }
  return fn;
}
}  // namespace

int kq_decode_step_static(const kq_decode_model* model, const void* x, float* logits, int M, void* stream) {
  std::string err;
  if (kq::decode_check(model, M, &err) != 0) return fail(KQ_ERR_ARG, err);
  if (!fmt_known(model->layer_fmt) || !fmt_known(model->head_fmt))
    return fail(KQ_ERR_UNSUPPORTED, "unknown weight format in the model");
  if (!x || !logits) return fail(KQ_ERR_ARG, "x or logits is NULL");
  if (!aligned(x, 16) || !aligned(logits, 4)) return fail(KQ_ERR_ARG, "misaligned x or logits");
  const size_t need = kq::decode_workspace_size(model, M);
  if (need > (size_t)KQ_DECODE_STATIC_SCRATCH_BYTES)
    return fail(KQ_ERR_WORKSPACE, "this model needs " + std::to_string(need) + " bytes of scratch for M=" +
                                      std::to_string(M) + "; the static scratch holds " +
                                      std::to_string((size_t)KQ_DECODE_STATIC_SCRATCH_BYTES) +
                                      " bytes (use kq_decode_step with a caller workspace)");
  for (int l = 0; l < model->n_layers; ++l) {
    const void* ps[4] = {model->w_qkv[l], model->w_o[l], model->w_gate_up[l], model->w_down[l]};
    for (const void* p : ps)
      if (!p || !aligned(p, 16)) return fail(KQ_ERR_ARG, "layer " + std::to_string(l) + ": NULL or misaligned weights");
  }
  if (!aligned(model->w_head, 16)) return fail(KQ_ERR_ARG, "misaligned w_head");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(KQ_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return fail(KQ_ERR_UNSUPPORTED, "device index beyond 63");
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    void* ctx = nullptr;
    const CtxGetCurrentFn get_ctx = ctx_get_current_fn();
    if (get_ctx && get_ctx(&ctx) != 0) ctx = nullptr;
    if (!g_scratch_ptr[dev] || !ctx || ctx != g_scratch_ctx[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_decode_scratch);  // makes the primary context current if none is
      if (e != cudaSuccess || !p)
        return fail(KQ_ERR_CUDA, std::string("cudaGetSymbolAddress of the decode scratch: ") + cudaGetErrorString(e));
      if (get_ctx && get_ctx(&ctx) != 0) ctx = nullptr;
      g_scratch_ptr[dev] = p;
      g_scratch_ctx[dev] = ctx;  // null (context unknown): looked up again on every call
    }
    scratch = g_scratch_ptr[dev];
  }
  const int sms = sm_count(&err);
  if (sms < 0) return fail(KQ_ERR_CUDA, err);
  // Every buffer of the scratch is written before it is read within a step, so nothing
  // needs clearing between calls.
  if (kq::decode_step(model, static_cast<const uint16_t*>(x), logits, M, scratch, sms,
                      static_cast<cudaStream_t>(stream), &err) != 0)
    return fail(KQ_ERR_CUDA, err);
  return ok();
}

}  // extern "C"
