// Scalar fp64 oracle of one decode step of a dense transformer on block-quantized weights.
// TEST INFRASTRUCTURE ONLY (see oracle.cpp's header); no code shared with the CUDA path.
//
// The step composes the weight-streaming GEMV (Kinetic README, "What makes it fast": a
// decode step reads every weight once per token) with a dense layer:
//   x = bf16(RMSNorm(h));  qkv = x Wqkv^T;  o_in = bf16(v expanded over the query heads of
//   its group) -- the attention of a token over a context of one token (softmax weight 1
//   on its own value);  h = h + o_in Wo^T;  x = bf16(RMSNorm(h));  gu = x Wgu^T;
//   a = bf16(silu(g) * u);  h = h + a Wd^T;  ...;  logits = bf16(RMSNorm(h)) Whead^T.
// RMSNorm(h) = h / sqrt(mean(h^2) + eps) (unit weight), silu(g) = g / (1 + exp(-g)).
// Everything is fp64 here except the bf16 roundings (nearest, ties to even, from fp64),
// which sit where the model feeds a GEMV.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

extern "C" int orc_gemv(int fmt, const uint8_t* blocks, int x_dtype, const void* x, int64_t M, int64_t N,
                        int64_t K, double* y, double* absy, int nthreads);
extern "C" int orc_attention_bf16q(int M, int L, int n_q, int n_kv, int hd, const uint16_t* qb, const uint16_t* k,
                                   const uint16_t* v, const uint32_t* mask, float scale, double* out, double* base);

namespace {

// Correctly rounded binary64 -> bfloat16 (8 exponent bits, 7 fraction bits), ties to even.
uint16_t double_to_bf16_rn(double v) {
  if (std::isnan(v)) return 0x7FC0;
  const uint16_t sign = std::signbit(v) ? 0x8000 : 0;
  const double a = std::fabs(v);
  if (a == 0.0) return sign;
  const double max_bf = std::ldexp(255.0 / 128.0, 127);     // 0x7F7F
  const double half_ulp_top = std::ldexp(1.0, 127 - 8);     // half an ulp at the top binade
  if (a >= max_bf + half_ulp_top) return sign | 0x7F80;     // rounds to infinity
  int E;
  std::frexp(a, &E);
  E -= 1;                                                   // a in [2^E, 2^(E+1))
  if (E < -126) E = -126;                                   // subnormal range: quantum 2^-133
  const double n = std::ldexp(a, 7 - E);                    // significand in units of the quantum
  double f = std::floor(n);
  const double r = n - f;
  if (r > 0.5 || (r == 0.5 && std::fmod(f, 2.0) != 0.0)) f += 1.0;
  // reassemble through float (exact: f has at most 8 significant bits, E within range)
  const float out = (float)std::ldexp(f, E - 7);
  uint32_t u;
  std::memcpy(&u, &out, 4);
  return sign | (uint16_t)(u >> 16);
}

double bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return (double)f;
}

void rmsnorm_bf16(const std::vector<double>& h, int64_t M, int64_t D, double eps, std::vector<uint16_t>& out) {
  out.assign((size_t)(M * D), 0);
  for (int64_t j = 0; j < M; ++j) {
    double ss = 0.0;
    for (int64_t i = 0; i < D; ++i) ss += h[(size_t)(j * D + i)] * h[(size_t)(j * D + i)];
    const double inv = 1.0 / std::sqrt(ss / (double)D + eps);
    for (int64_t i = 0; i < D; ++i) out[(size_t)(j * D + i)] = double_to_bf16_rn(h[(size_t)(j * D + i)] * inv);
  }
}

// act[j][i] = bf16(silu(g) * u), g = gu[j][i], u = gu[j][F + i], silu(g) = g / (1 + exp(-g)):
// the gated activation that feeds the down projection.
void swiglu_bf16(const double* gu, int64_t M, int64_t F, uint16_t* act) {
  for (int64_t j = 0; j < M; ++j)
    for (int64_t i = 0; i < F; ++i) {
      const double g = gu[j * 2 * F + i], u = gu[j * 2 * F + F + i];
      act[j * F + i] = double_to_bf16_rn(g / (1.0 + std::exp(-g)) * u);
    }
}

}  // namespace

extern "C" {

uint16_t orc_double_to_bf16_rn(double v) { return double_to_bf16_rn(v); }

// out[i] = bf16(v[i]) (nearest, ties to even) for n values.
int orc_bf16_rn_n(const double* v, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = double_to_bf16_rn(v[i]);
  return 0;
}

// The SwiGLU of the decode step for M rows (gu: M x 2F, gate then up; act: M x F bf16 bits).
int orc_swiglu(const double* gu, int64_t M, int64_t F, uint16_t* act) {
  swiglu_bf16(gu, M, F, act);
  return 0;
}

// out = bf16(RMSNorm(h)) for M rows of D values.
int orc_rmsnorm(const double* h, uint16_t* out, int64_t M, int64_t D, double eps) {
  std::vector<double> hv(h, h + M * D);
  std::vector<uint16_t> o;
  rmsnorm_bf16(hv, M, D, eps, o);
  std::memcpy(out, o.data(), sizeof(uint16_t) * (size_t)(M * D));
  return 0;
}

// The step with attention over a KV cache (the step above with its attention stand-in
// replaced; attention.cpp defines the attention): per layer the window's k and v (rounded to
// bf16) are appended at positions L..L+M-1 of a copy of the layer's cache, q is rounded to
// bf16, and the attention output is rounded to bf16 as it feeds Wo. k_cache[l], v_cache[l]:
// L rows of kv_dim bf16 (read only). mask: NULL (causal) or M words. scale: the score
// multiplier (a float, as the kernels take it).
int orc_decode_step_attn(int n_layers, int hidden, int q_dim, int kv_dim, int head_dim, int ffn, int vocab,
                         int layer_fmt, int head_fmt, double eps, const uint8_t* const* w_qkv,
                         const uint8_t* const* w_o, const uint8_t* const* w_gu, const uint8_t* const* w_down,
                         const uint8_t* w_head, const uint16_t* const* k_cache, const uint16_t* const* v_cache,
                         int L, const uint32_t* mask, float scale, const uint16_t* x_bf16, int64_t M,
                         double* logits, int nthreads, uint16_t* x_final) {
  const int64_t D = hidden, QKV = q_dim + 2 * kv_dim, F = ffn;
  const int n_q = q_dim / head_dim, n_kv = kv_dim / head_dim;
  const int BF16 = 2;
  std::vector<double> h((size_t)(M * D));
  for (int64_t i = 0; i < M * D; ++i) h[(size_t)i] = bf16_to_double(x_bf16[i]);
  std::vector<uint16_t> xb;
  std::vector<double> qkv((size_t)(M * QKV)), y((size_t)(M * D)), gu((size_t)(M * 2 * F)), att((size_t)(M * q_dim));
  std::vector<uint16_t> oin((size_t)(M * q_dim)), act((size_t)(M * F)), qb((size_t)(M * q_dim));
  std::vector<uint16_t> kc((size_t)((L + M) * kv_dim)), vc((size_t)((L + M) * kv_dim));
  for (int l = 0; l < n_layers; ++l) {
    rmsnorm_bf16(h, M, D, eps, xb);
    if (orc_gemv(layer_fmt, w_qkv[l], BF16, xb.data(), M, QKV, D, qkv.data(), nullptr, nthreads)) return -1;
    if (L > 0) {
      std::memcpy(kc.data(), k_cache[l], sizeof(uint16_t) * (size_t)L * kv_dim);
      std::memcpy(vc.data(), v_cache[l], sizeof(uint16_t) * (size_t)L * kv_dim);
    }
    for (int64_t j = 0; j < M; ++j) {
      for (int c = 0; c < q_dim; ++c) qb[(size_t)(j * q_dim + c)] = double_to_bf16_rn(qkv[(size_t)(j * QKV + c)]);
      for (int c = 0; c < kv_dim; ++c) {
        kc[(size_t)((L + j) * kv_dim + c)] = double_to_bf16_rn(qkv[(size_t)(j * QKV + q_dim + c)]);
        vc[(size_t)((L + j) * kv_dim + c)] = double_to_bf16_rn(qkv[(size_t)(j * QKV + q_dim + kv_dim + c)]);
      }
    }
    if (orc_attention_bf16q((int)M, L, n_q, n_kv, head_dim, qb.data(), kc.data(), vc.data(), mask, scale,
                            att.data(), nullptr))
      return -1;
    for (int64_t e = 0; e < M * q_dim; ++e) oin[(size_t)e] = double_to_bf16_rn(att[(size_t)e]);
    if (orc_gemv(layer_fmt, w_o[l], BF16, oin.data(), M, D, q_dim, y.data(), nullptr, nthreads)) return -1;
    for (int64_t i = 0; i < M * D; ++i) h[(size_t)i] += y[(size_t)i];
    rmsnorm_bf16(h, M, D, eps, xb);
    if (orc_gemv(layer_fmt, w_gu[l], BF16, xb.data(), M, 2 * F, D, gu.data(), nullptr, nthreads)) return -1;
    swiglu_bf16(gu.data(), M, F, act.data());
    if (orc_gemv(layer_fmt, w_down[l], BF16, act.data(), M, D, F, y.data(), nullptr, nthreads)) return -1;
    for (int64_t i = 0; i < M * D; ++i) h[(size_t)i] += y[(size_t)i];
  }
  rmsnorm_bf16(h, M, D, eps, xb);
  if (x_final) std::memcpy(x_final, xb.data(), sizeof(uint16_t) * (size_t)(M * D));
  if (orc_gemv(head_fmt, w_head, BF16, xb.data(), M, vocab, D, logits, nullptr, nthreads)) return -1;
  return 0;
}

int orc_decode_step(int n_layers, int hidden, int q_dim, int kv_dim, int head_dim, int ffn, int vocab,
                    int layer_fmt, int head_fmt, double eps, const uint8_t* const* w_qkv,
                    const uint8_t* const* w_o, const uint8_t* const* w_gu, const uint8_t* const* w_down,
                    const uint8_t* w_head, const uint16_t* x_bf16, int64_t M, double* logits, int nthreads,
                    uint16_t* x_final) {
  const int64_t D = hidden, QKV = q_dim + 2 * kv_dim, F = ffn;
  const int group = (q_dim / head_dim) / (kv_dim / head_dim);
  const int BF16 = 2;
  std::vector<double> h((size_t)(M * D));
  for (int64_t i = 0; i < M * D; ++i) h[(size_t)i] = bf16_to_double(x_bf16[i]);
  std::vector<uint16_t> xb;
  std::vector<double> qkv((size_t)(M * QKV)), y((size_t)(M * D)), gu((size_t)(M * 2 * F));
  std::vector<uint16_t> oin((size_t)(M * q_dim)), act((size_t)(M * F));
  for (int l = 0; l < n_layers; ++l) {
    rmsnorm_bf16(h, M, D, eps, xb);
    if (orc_gemv(layer_fmt, w_qkv[l], BF16, xb.data(), M, QKV, D, qkv.data(), nullptr, nthreads)) return -1;
    for (int64_t j = 0; j < M; ++j)
      for (int c = 0; c < q_dim; ++c) {
        const int hq = c / head_dim, d = c % head_dim;
        oin[(size_t)(j * q_dim + c)] =
            double_to_bf16_rn(qkv[(size_t)(j * QKV + q_dim + kv_dim + (hq / group) * head_dim + d)]);
      }
    if (orc_gemv(layer_fmt, w_o[l], BF16, oin.data(), M, D, q_dim, y.data(), nullptr, nthreads)) return -1;
    for (int64_t i = 0; i < M * D; ++i) h[(size_t)i] += y[(size_t)i];
    rmsnorm_bf16(h, M, D, eps, xb);
    if (orc_gemv(layer_fmt, w_gu[l], BF16, xb.data(), M, 2 * F, D, gu.data(), nullptr, nthreads)) return -1;
    swiglu_bf16(gu.data(), M, F, act.data());
    if (orc_gemv(layer_fmt, w_down[l], BF16, act.data(), M, D, F, y.data(), nullptr, nthreads)) return -1;
    for (int64_t i = 0; i < M * D; ++i) h[(size_t)i] += y[(size_t)i];
  }
  rmsnorm_bf16(h, M, D, eps, xb);
  if (x_final) std::memcpy(x_final, xb.data(), sizeof(uint16_t) * (size_t)(M * D));  // the head's input
  if (orc_gemv(head_fmt, w_head, BF16, xb.data(), M, vocab, D, logits, nullptr, nthreads)) return -1;
  return 0;
}

}  // extern "C"
