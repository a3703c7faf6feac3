// Scalar fp64 oracle of decode attention over a KV cache for a window of M tokens (a
// speculative verify window). TEST INFRASTRUCTURE ONLY (see oracle.cpp's header); no code
// shared with the CUDA path.
//
// The pages check k guessed tokens in one pass (Kinetic README, "What makes it fast"; Kipp
// README, batched decode; Kapitsa README, the tree of guesses verified in one pass): every
// guess attends to the whole cached context and to the guesses before it in the window
// (causal), or to the guesses on its own branch (a tree mask). The reading used here:
//   positions 0..L-1 hold the cached context, positions L..L+M-1 the window's own keys and
//   values; window token i sees every cached position and window position L+j when
//   (mask == NULL ? j <= i : bit j of mask[i]);
//   query head hq reads kv head hq / (n_q / n_kv) (grouped-query attention);
//   q is rounded to bf16 (nearest, ties to even) first: activations between ops are bf16;
//   K and V are stored as bf16.
//   s_p = scale * sum_d q[d] k_p[d];  w_p = exp(s_p - max_p s_p);  o = sum_p w_p v_p / sum_p w_p.
// Everything after the bf16 inputs is fp64. A token that sees no position outputs zeros.
// base = sum_p (w_p / sum w) |v_p| per output element: the scale of the error contract.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

double bf16_bits_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return (double)f;
}

// fp32 -> bf16, round to nearest, ties to even (written out on the bit pattern; NaN kept
// quiet). Exact for every finite input: the discarded 16 bits decide the rounding.
uint16_t f32_to_bf16_rn(float x) {
  uint32_t u;
  std::memcpy(&u, &x, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x0040u);
  const uint32_t lower = u & 0xFFFFu, upper = u >> 16;
  if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) return (uint16_t)(upper + 1u);
  return (uint16_t)upper;
}

}  // namespace

extern "C" {

int orc_attention_bf16q(int M, int L, int n_q, int n_kv, int hd, const uint16_t* qb, const uint16_t* k,
                        const uint16_t* v, const uint32_t* mask, float scale, double* out, double* base);

// q: M x (n_q*hd) fp32; k, v: (L+M) x (n_kv*hd) bf16 bits; mask: M words or NULL.
// out, base: M x (n_q*hd) fp64. Returns 0, or -1 on bad arguments.
int orc_attention(int M, int L, int n_q, int n_kv, int hd, const float* q, const uint16_t* k, const uint16_t* v,
                  const uint32_t* mask, float scale, double* out, double* base) {
  if (M < 1 || M > 32 || n_q < 1 || hd < 1) return -1;
  std::vector<uint16_t> qb((size_t)M * n_q * hd);
  for (size_t e = 0; e < qb.size(); ++e) qb[e] = f32_to_bf16_rn(q[e]);
  return orc_attention_bf16q(M, L, n_q, n_kv, hd, qb.data(), k, v, mask, scale, out, base);
}

// The same with q given as bf16 bits (already rounded); base may be NULL.
int orc_attention_bf16q(int M, int L, int n_q, int n_kv, int hd, const uint16_t* qb, const uint16_t* k,
                        const uint16_t* v, const uint32_t* mask, float scale, double* out, double* base) {
  if (M < 1 || M > 32 || L < 0 || n_q < 1 || n_kv < 1 || hd < 1 || n_q % n_kv) return -1;
  const int group = n_q / n_kv, qw = n_q * hd, kw = n_kv * hd;
  std::vector<double> qv(hd), s;
  std::vector<int> pos;
  for (int i = 0; i < M; ++i) {
    pos.clear();
    for (int p = 0; p < L; ++p) pos.push_back(p);
    for (int j = 0; j < M; ++j) {
      const bool vis = mask ? ((mask[i] >> j) & 1u) != 0u : j <= i;
      if (vis) pos.push_back(L + j);
    }
    for (int hq = 0; hq < n_q; ++hq) {
      const int kvh = hq / group;
      double* o = out + (size_t)i * qw + (size_t)hq * hd;
      double* b = base ? base + (size_t)i * qw + (size_t)hq * hd : nullptr;
      for (int d = 0; d < hd; ++d) {
        o[d] = 0.0;
        if (b) b[d] = 0.0;
      }
      if (pos.empty()) continue;
      for (int d = 0; d < hd; ++d) qv[d] = bf16_bits_to_double(qb[(size_t)i * qw + (size_t)hq * hd + d]);
      s.assign(pos.size(), 0.0);
      double mx = -INFINITY;
      for (size_t t = 0; t < pos.size(); ++t) {
        const uint16_t* kp = k + (size_t)pos[t] * kw + (size_t)kvh * hd;
        double dot = 0.0;
        for (int d = 0; d < hd; ++d) dot += qv[d] * bf16_bits_to_double(kp[d]);
        s[t] = (double)scale * dot;
        if (s[t] > mx) mx = s[t];
      }
      double z = 0.0;
      for (size_t t = 0; t < pos.size(); ++t) {
        s[t] = std::exp(s[t] - mx);
        z += s[t];
      }
      for (size_t t = 0; t < pos.size(); ++t) {
        const uint16_t* vp = v + (size_t)pos[t] * kw + (size_t)kvh * hd;
        const double w = s[t] / z;
        for (int d = 0; d < hd; ++d) {
          const double vv = bf16_bits_to_double(vp[d]);
          o[d] += w * vv;
          if (b) b[d] += w * std::fabs(vv);
        }
      }
    }
  }
  return 0;
}

}  // extern "C"
