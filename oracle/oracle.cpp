// Scalar CPU oracle for block-quantized decode GEMV. TEST INFRASTRUCTURE ONLY.
//
// This file is the checker, not the product. Only the test suite, the smoke
// check and the benchmark's CPU-baseline leg may load it. It shares no code,
// header, table or constant generator with the CUDA path: everything here is
// written out from the definitions, in fp64, one weight at a time.
//
// What it computes (sources are the engine READMEs this library follows):
//  (Q5_K and Q6_K, the GGUF k-quants next to Q4_K, follow GGUF's published layouts for
//  the same reason as Q4_K: GGUF files are to work unchanged, and Q4_K_M files mix in
//  higher-precision k-quant tensors.)
//  * Kinetic README, "What makes it fast": a dense model reads all of its
//    weights once per token; a speculative check runs every guess through one
//    pass over the weights. The result of that pass is the plain product
//    y[j][n] = sum_k deq(W)[n][k] * x[j][k], which is what orc_gemv returns.
//  * Kinetic README, "Switching from llama.cpp": GGUF files work unchanged and
//    the quantizer writes llama.cpp's Q8_0 / Q4_K bytes, so the block layouts
//    are GGUF's published ones (Q8_0: fp16 d + 32 int8; Q4_K: fp16 d, fp16
//    dmin, 12 bytes of packed 6-bit sub-block scales and mins, 128 bytes of
//    4-bit codes).
//  * Kipp README, "How fast" (footnote): affine4 is scale + bias per group of
//    32. The pages give no byte layout; the reading used here is 20 bytes per
//    group: fp16 s, fp16 b, then 16 bytes of codes, weight 2i in the low
//    nibble of byte i and weight 2i+1 in the high nibble. w = s*q + b.
//
// The quantizers are test-data generators (the GPU path never quantizes in
// the timed region). They are deterministic covering schemes, not llama.cpp's
// search: each keeps |w - deq(q(w))| <= (step of its block)/2.
//
// Build: g++ -O2 -fopenmp -ffp-contract=off -fPIC -shared (no fast-math, no
// contraction, so every fp64 operation rounds once, as written).
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>
#include <algorithm>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

enum { ORC_Q8_0 = 1, ORC_Q4_K = 2, ORC_AFFINE4 = 3, ORC_Q5_K = 4, ORC_Q6_K = 5 };
enum { ORC_F32 = 1, ORC_BF16 = 2 };

// ---------------------------------------------------------------- fp16 ----
// IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits.
double half_to_double(uint16_t h) {
  const int sign = h >> 15;
  const int e = (h >> 10) & 31;
  const int f = h & 1023;
  double v;
  if (e == 0) {
    v = std::ldexp((double)f, -24);                 // subnormal: f * 2^-24
  } else if (e == 31) {
    v = f ? NAN : INFINITY;
  } else {
    v = std::ldexp((double)(1024 + f), e - 25);     // (1 + f/1024) * 2^(e-15)
  }
  return sign ? -v : v;
}

// Round a non-negative finite real n to an integer, ties to even.
double round_half_even(double n) {
  double f = std::floor(n);
  double r = n - f;                                  // exact for n < 2^52
  if (r > 0.5 || (r == 0.5 && std::fmod(f, 2.0) != 0.0)) f += 1.0;
  return f;
}

// Correctly rounded (nearest, ties to even) binary64 -> binary16, in one step.
uint16_t double_to_half_rn(double v) {
  if (std::isnan(v)) return 0x7E00;
  const uint16_t sign = std::signbit(v) ? 0x8000 : 0;
  const double a = std::fabs(v);
  if (a == 0.0) return sign;
  if (a >= 65520.0) return sign | 0x7C00;            // 65504 + half an ulp and up
  if (a < std::ldexp(1.0, -14)) {                     // subnormal range, quantum 2^-24
    const double n = round_half_even(std::ldexp(a, 24));
    return sign | (uint16_t)n;                        // n == 1024 is the smallest normal
  }
  int ex;
  std::frexp(a, &ex);                                 // a = fr * 2^ex, fr in [0.5, 1)
  int E = ex - 1;                                     // a in [2^E, 2^(E+1))
  double n = round_half_even(std::ldexp(a, 10 - E));  // in [1024, 2048]
  if (n == 2048.0) { n = 1024.0; E += 1; }
  if (E > 15) return sign | 0x7C00;
  return sign | (uint16_t)((E + 15) << 10) | (uint16_t)(n - 1024.0);
}

uint16_t half_next_up(uint16_t h) {
  if (h == 0x8000) return 0x0001;
  if (h & 0x8000) return h - 1;
  return h + 1;
}
uint16_t half_next_down(uint16_t h) {
  if (h == 0x0000) return 0x8001;
  if (h & 0x8000) return h + 1;
  return h - 1;
}
// Smallest binary16 >= t (t finite).
uint16_t double_to_half_up(double t) {
  uint16_t h = double_to_half_rn(t);
  if (half_to_double(h) < t) h = half_next_up(h);
  return h;
}
// Largest binary16 <= t (t finite).
uint16_t double_to_half_down(double t) {
  uint16_t h = double_to_half_rn(t);
  if (half_to_double(h) > t) h = half_next_down(h);
  return h;
}

double bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return (double)f;
}

uint16_t rd16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }
void wr16(uint8_t* p, uint16_t v) { p[0] = (uint8_t)(v & 0xFF); p[1] = (uint8_t)(v >> 8); }

int block_bytes(int fmt) {
  switch (fmt) { case ORC_Q8_0: return 34; case ORC_Q4_K: return 144; case ORC_AFFINE4: return 20; case ORC_Q5_K: return 176; case ORC_Q6_K: return 210; }
  return 0;
}
int block_weights(int fmt) {
  switch (fmt) { case ORC_Q8_0: return 32; case ORC_Q4_K: return 256; case ORC_AFFINE4: return 32; case ORC_Q5_K: return 256; case ORC_Q6_K: return 256; }
  return 0;
}

// ---------------------------------------------------------------- Q8_0 ----
// 34 bytes: d (fp16 LE) then q[32] (int8). w_i = d * q_i.
// Quantizer: d = fp16_rn(max|w| / 127); q_i = clamp(round_half_away(w_i / d), -127, 127),
// computed against the stored fp16 d so that |w_i - d q_i| <= d/2.
void quant_q8_0(const float* w, uint8_t* blk) {
  double amax = 0.0;
  for (int i = 0; i < 32; ++i) amax = std::max(amax, std::fabs((double)w[i]));
  const uint16_t d16 = double_to_half_rn(amax / 127.0);
  const double d = half_to_double(d16);
  wr16(blk, d16);
  for (int i = 0; i < 32; ++i) {
    double q = 0.0;
    if (d != 0.0) q = std::min(127.0, std::max(-127.0, std::round((double)w[i] / d)));
    blk[2 + i] = (uint8_t)(int8_t)(int)q;
  }
}
void deq_q8_0(const uint8_t* blk, double* out) {
  const double d = half_to_double(rd16(blk));
  for (int i = 0; i < 32; ++i) out[i] = d * (double)(int8_t)blk[2 + i];
}

// ---------------------------------------------------------------- Q4_K ----
// 144 bytes: d (fp16), dmin (fp16), scales[12], qs[128].
// Sub-block j (0..7) holds weights 32j .. 32j+31 and has a 6-bit scale sc_j and
// a 6-bit min m_j, packed GGUF-style into the 12 scale bytes:
//   j < 4 : sc_j = scales[j] & 63,  m_j = scales[j+4] & 63
//   j >= 4: sc_j = (scales[j+4] & 15) | ((scales[j-4] >> 6) << 4)
//           m_j  = (scales[j+4] >> 4) | ((scales[j]   >> 6) << 4)
// Codes: for chunk c = 0..3 and l = 0..31, byte qs[32c + l] holds weight 64c + l
// in its low nibble and weight 64c + 32 + l in its high nibble.
// w = d * sc_j * q - dmin * m_j.
void unpack_scale_min(const uint8_t* sc12, int j, int* sc, int* m) {
  if (j < 4) {
    *sc = sc12[j] & 63;
    *m = sc12[j + 4] & 63;
  } else {
    *sc = (sc12[j + 4] & 15) | ((sc12[j - 4] >> 6) << 4);
    *m = (sc12[j + 4] >> 4) | ((sc12[j] >> 6) << 4);
  }
}
void pack_scale_min(const int* sc, const int* m, uint8_t* sc12) {
  std::memset(sc12, 0, 12);
  for (int j = 0; j < 4; ++j) {
    sc12[j] |= (uint8_t)(sc[j] & 63);
    sc12[j + 4] |= (uint8_t)(m[j] & 63);
  }
  for (int j = 4; j < 8; ++j) {
    sc12[j + 4] = (uint8_t)((sc[j] & 15) | ((m[j] & 15) << 4));
    sc12[j - 4] |= (uint8_t)((sc[j] >> 4) << 6);
    sc12[j] |= (uint8_t)((m[j] >> 4) << 6);
  }
}
int code_q4_k(const uint8_t* qs, int i) {            // weight index i in 0..255
  const int c = i / 64, r = i % 64;
  const uint8_t byte = qs[32 * c + (r % 32)];
  return r < 32 ? (byte & 15) : (byte >> 4);
}
// Quantizer (a covering scheme, not llama.cpp's search):
//  per sub-block: lo = min(0, min w), hi = max(0, max w), mraw = -lo
//  dmin = smallest fp16 >= max(mraw)/63,  m_j = ceil(mraw_j / dmin)
//  t_j  = hi_j + dmin*m_j,  d = smallest fp16 >= max(t)/945,  sc_j = ceil(t_j / (15 d))
//  q    = round_half_away((w + dmin*m_j) / (d*sc_j)), which lies in [0, 15].
// If a rounding step ever pushed m_j or sc_j past 63, the fp16 step is raised by
// one code and the step repeated (never observed; kept so 6 bits always hold).
void quant_q4_k(const float* w, uint8_t* blk) {
  double lo[8], hi[8], mraw[8];
  for (int j = 0; j < 8; ++j) {
    lo[j] = 0.0; hi[j] = 0.0;
    for (int i = 0; i < 32; ++i) {
      const double v = (double)w[32 * j + i];
      lo[j] = std::min(lo[j], v);
      hi[j] = std::max(hi[j], v);
    }
    mraw[j] = -lo[j];
  }
  double maxm = 0.0;
  for (int j = 0; j < 8; ++j) maxm = std::max(maxm, mraw[j]);
  uint16_t dmin16 = 0;
  int m[8] = {0};
  if (maxm > 0.0) {
    dmin16 = double_to_half_up(maxm / 63.0);
    for (;;) {
      const double dmin = half_to_double(dmin16);
      bool ok = true;
      for (int j = 0; j < 8; ++j) {
        m[j] = (int)std::ceil(mraw[j] / dmin);
        if (m[j] > 63) ok = false;
      }
      if (ok) break;
      dmin16 = half_next_up(dmin16);
    }
  }
  const double dmin = half_to_double(dmin16);
  double t[8], maxt = 0.0;
  for (int j = 0; j < 8; ++j) {
    t[j] = hi[j] + dmin * (double)m[j];
    maxt = std::max(maxt, t[j]);
  }
  uint16_t d16 = 0;
  int sc[8] = {0};
  if (maxt > 0.0) {
    d16 = double_to_half_up(maxt / 945.0);
    for (;;) {
      const double d = half_to_double(d16);
      bool ok = true;
      for (int j = 0; j < 8; ++j) {
        sc[j] = (int)std::ceil(t[j] / (15.0 * d));
        if (sc[j] > 63) ok = false;
      }
      if (ok) break;
      d16 = half_next_up(d16);
    }
  }
  const double d = half_to_double(d16);
  wr16(blk + 0, d16);
  wr16(blk + 2, dmin16);
  pack_scale_min(sc, m, blk + 4);
  uint8_t* qs = blk + 16;
  std::memset(qs, 0, 128);
  for (int i = 0; i < 256; ++i) {
    const int j = i / 32;
    const double step = d * (double)sc[j];
    int q = 0;
    if (step != 0.0) {
      const double r = std::round(((double)w[i] + dmin * (double)m[j]) / step);
      q = (int)std::min(15.0, std::max(0.0, r));
    }
    const int c = i / 64, r = i % 64;
    if (r < 32) qs[32 * c + r] |= (uint8_t)q;
    else qs[32 * c + (r - 32)] |= (uint8_t)(q << 4);
  }
}
void deq_q4_k(const uint8_t* blk, double* out) {
  const double d = half_to_double(rd16(blk + 0));
  const double dmin = half_to_double(rd16(blk + 2));
  for (int i = 0; i < 256; ++i) {
    int sc, m;
    unpack_scale_min(blk + 4, i / 32, &sc, &m);
    out[i] = d * (double)sc * (double)code_q4_k(blk + 16, i) - dmin * (double)m;
  }
}

// ---------------------------------------------------------------- Q5_K ----
// 176 bytes: d (fp16), dmin (fp16), scales[12] (packed exactly as in Q4_K), qh[32],
// qs[128]. The low four bits of weight i sit where Q4_K keeps its code (chunk c = i/64,
// l = i%32: low nibble of qs[32c + l] for i%64 < 32, high nibble otherwise); the fifth
// bit is bit (2c + (i%64 >= 32)) of qh[l]. q = low4 + 16*bit5 in 0..31.
// w = d * sc_j * q - dmin * m_j, sub-block j = i/32 as in Q4_K.
int code_q5_k(const uint8_t* blk, int i) {
  const int c = i / 64, r = i % 64, l = r % 32;
  const int low4 = code_q4_k(blk + 48, i);
  const int bit5 = (blk[16 + l] >> (2 * c + (r >= 32 ? 1 : 0))) & 1;
  return low4 + 16 * bit5;
}
// Quantizer: the Q4_K covering scheme with 31 levels per step:
//  dmin = smallest fp16 >= max(mraw)/63, m_j = ceil(mraw_j / dmin), t_j = hi_j + dmin*m_j,
//  d = smallest fp16 >= max(t)/(63*31), sc_j = ceil(t_j / (31 d)),
//  q = round_half_away((w + dmin*m_j) / (d*sc_j)), which lies in [0, 31].
void quant_q5_k(const float* w, uint8_t* blk) {
  double lo[8], hi[8], mraw[8];
  for (int j = 0; j < 8; ++j) {
    lo[j] = 0.0; hi[j] = 0.0;
    for (int i = 0; i < 32; ++i) {
      const double v = (double)w[32 * j + i];
      lo[j] = std::min(lo[j], v);
      hi[j] = std::max(hi[j], v);
    }
    mraw[j] = -lo[j];
  }
  double maxm = 0.0;
  for (int j = 0; j < 8; ++j) maxm = std::max(maxm, mraw[j]);
  uint16_t dmin16 = 0;
  int m[8] = {0};
  if (maxm > 0.0) {
    dmin16 = double_to_half_up(maxm / 63.0);
    for (;;) {
      const double dmin = half_to_double(dmin16);
      bool ok = true;
      for (int j = 0; j < 8; ++j) {
        m[j] = (int)std::ceil(mraw[j] / dmin);
        if (m[j] > 63) ok = false;
      }
      if (ok) break;
      dmin16 = half_next_up(dmin16);
    }
  }
  const double dmin = half_to_double(dmin16);
  double t[8], maxt = 0.0;
  for (int j = 0; j < 8; ++j) {
    t[j] = hi[j] + dmin * (double)m[j];
    maxt = std::max(maxt, t[j]);
  }
  uint16_t d16 = 0;
  int sc[8] = {0};
  if (maxt > 0.0) {
    d16 = double_to_half_up(maxt / (63.0 * 31.0));
    for (;;) {
      const double d = half_to_double(d16);
      bool ok = true;
      for (int j = 0; j < 8; ++j) {
        sc[j] = (int)std::ceil(t[j] / (31.0 * d));
        if (sc[j] > 63) ok = false;
      }
      if (ok) break;
      d16 = half_next_up(d16);
    }
  }
  const double d = half_to_double(d16);
  wr16(blk + 0, d16);
  wr16(blk + 2, dmin16);
  pack_scale_min(sc, m, blk + 4);
  uint8_t* qh = blk + 16;
  uint8_t* qs = blk + 48;
  std::memset(qh, 0, 32);
  std::memset(qs, 0, 128);
  for (int i = 0; i < 256; ++i) {
    const int j = i / 32;
    const double step = d * (double)sc[j];
    int q = 0;
    if (step != 0.0) {
      const double r = std::round(((double)w[i] + dmin * (double)m[j]) / step);
      q = (int)std::min(31.0, std::max(0.0, r));
    }
    const int c = i / 64, r = i % 64, l = r % 32;
    if (r < 32) qs[32 * c + l] |= (uint8_t)(q & 15);
    else qs[32 * c + l] |= (uint8_t)((q & 15) << 4);
    if (q & 16) qh[l] |= (uint8_t)(1u << (2 * c + (r >= 32 ? 1 : 0)));
  }
}
void deq_q5_k(const uint8_t* blk, double* out) {
  const double d = half_to_double(rd16(blk + 0));
  const double dmin = half_to_double(rd16(blk + 2));
  for (int i = 0; i < 256; ++i) {
    int sc, m;
    unpack_scale_min(blk + 4, i / 32, &sc, &m);
    out[i] = d * (double)sc * (double)code_q5_k(blk, i) - dmin * (double)m;
  }
}

// ---------------------------------------------------------------- Q6_K ----
// 210 bytes: ql[128], qh[64], scales[16] (int8), d (fp16) at byte 208 (GGUF's Q6_K).
// Weight i = 128n + 32k + l (half n = 0..1, quarter k = 0..3, l = 0..31) has the 6-bit code
//   q = low4 | (high2 << 4), low4 = nibble (k < 2 ? low : high) of ql[64n + 32*(k%2) + l],
//   high2 = bits 2k..2k+1 of qh[32n + l],
// and sub-block b = i/16 with int8 scale scales[b]: w = d * scales[b] * (q - 32).
int code_q6_k(const uint8_t* blk, int i) {
  const int n = i / 128, k = (i % 128) / 32, l = i % 32;
  const uint8_t qlb = blk[64 * n + 32 * (k % 2) + l];
  const int low4 = k < 2 ? (qlb & 15) : (qlb >> 4);
  const int high2 = (blk[128 + 32 * n + l] >> (2 * k)) & 3;
  return low4 | (high2 << 4);
}
// Quantizer (covering): a_b = max |w| over sub-block b (16 weights); d = smallest fp16 >=
// max(a)/(127*31); sc_b = ceil(a_b / (31 d)) <= 127; q = 32 + round_half_away(w / (d sc_b)),
// so q - 32 lies in [-31, 31] and |w - deq| <= d*sc_b/2.
void quant_q6_k(const float* w, uint8_t* blk) {
  double a[16], amax = 0.0;
  for (int b = 0; b < 16; ++b) {
    a[b] = 0.0;
    for (int i = 0; i < 16; ++i) a[b] = std::max(a[b], std::fabs((double)w[16 * b + i]));
    amax = std::max(amax, a[b]);
  }
  uint16_t d16 = 0;
  int sc[16] = {0};
  if (amax > 0.0) {
    d16 = double_to_half_up(amax / (127.0 * 31.0));
    for (;;) {
      const double d = half_to_double(d16);
      bool ok = true;
      for (int b = 0; b < 16; ++b) {
        sc[b] = (int)std::ceil(a[b] / (31.0 * d));
        if (sc[b] > 127) ok = false;
      }
      if (ok) break;
      d16 = half_next_up(d16);
    }
  }
  const double d = half_to_double(d16);
  std::memset(blk, 0, 210);
  for (int b = 0; b < 16; ++b) blk[192 + b] = (uint8_t)(int8_t)sc[b];
  wr16(blk + 208, d16);
  for (int i = 0; i < 256; ++i) {
    const double step = d * (double)sc[i / 16];
    int q = 32;
    if (step != 0.0) q = 32 + (int)std::min(31.0, std::max(-31.0, std::round((double)w[i] / step)));
    const int n = i / 128, k = (i % 128) / 32, l = i % 32;
    uint8_t& qlb = blk[64 * n + 32 * (k % 2) + l];
    qlb |= (uint8_t)(k < 2 ? (q & 15) : ((q & 15) << 4));
    blk[128 + 32 * n + l] |= (uint8_t)(((q >> 4) & 3) << (2 * k));
  }
}
void deq_q6_k(const uint8_t* blk, double* out) {
  const double d = half_to_double(rd16(blk + 208));
  for (int i = 0; i < 256; ++i) {
    const int sc = (int)(int8_t)blk[192 + i / 16];
    out[i] = d * (double)sc * (double)(code_q6_k(blk, i) - 32);
  }
}

// ------------------------------------------------------------- affine4 ----
// 20 bytes: s (fp16), b (fp16), codes[16]; weight 2i = low nibble of codes[i],
// weight 2i+1 = high nibble. w = s * q + b.
// Quantizer: b = largest fp16 <= min w; s = smallest fp16 >= (max w - b)/15;
// q = clamp(round_half_away((w - b)/s), 0, 15).
void quant_affine4(const float* w, uint8_t* blk) {
  double mn = (double)w[0], mx = (double)w[0];
  for (int i = 1; i < 32; ++i) { mn = std::min(mn, (double)w[i]); mx = std::max(mx, (double)w[i]); }
  const uint16_t b16 = double_to_half_down(mn);
  const double b = half_to_double(b16);
  const double span = mx - b;
  const uint16_t s16 = span > 0.0 ? double_to_half_up(span / 15.0) : 0;
  const double s = half_to_double(s16);
  wr16(blk + 0, s16);
  wr16(blk + 2, b16);
  for (int i = 0; i < 16; ++i) blk[4 + i] = 0;
  for (int i = 0; i < 32; ++i) {
    int q = 0;
    if (s != 0.0) q = (int)std::min(15.0, std::max(0.0, std::round(((double)w[i] - b) / s)));
    blk[4 + i / 2] |= (uint8_t)((i & 1) ? (q << 4) : q);
  }
}
void deq_affine4(const uint8_t* blk, double* out) {
  const double s = half_to_double(rd16(blk + 0));
  const double b = half_to_double(rd16(blk + 2));
  for (int i = 0; i < 32; ++i) {
    const int q = (i & 1) ? (blk[4 + i / 2] >> 4) : (blk[4 + i / 2] & 15);
    out[i] = s * (double)q + b;
  }
}

void deq_block(int fmt, const uint8_t* blk, double* out) {
  if (fmt == ORC_Q8_0) deq_q8_0(blk, out);
  else if (fmt == ORC_Q4_K) deq_q4_k(blk, out);
  else if (fmt == ORC_Q5_K) deq_q5_k(blk, out);
  else if (fmt == ORC_Q6_K) deq_q6_k(blk, out);
  else deq_affine4(blk, out);
}
void deq_row(int fmt, const uint8_t* row, int64_t K, double* out) {
  const int bw = block_weights(fmt), bb = block_bytes(fmt);
  for (int64_t b = 0; b < K / bw; ++b) deq_block(fmt, row + b * bb, out + b * bw);
}
double x_at(int x_dtype, const void* x, int64_t idx) {
  if (x_dtype == ORC_F32) return (double)((const float*)x)[idx];
  return bf16_to_double(((const uint16_t*)x)[idx]);
}

}  // namespace

extern "C" {

int orc_block_bytes(int fmt) { return block_bytes(fmt); }
int orc_block_weights(int fmt) { return block_weights(fmt); }
double orc_half_to_double(uint16_t h) { return half_to_double(h); }
uint16_t orc_double_to_half_rn(double v) { return double_to_half_rn(v); }
uint16_t orc_double_to_half_up(double v) { return double_to_half_up(v); }
uint16_t orc_double_to_half_down(double v) { return double_to_half_down(v); }
void orc_unpack_scale_min(const uint8_t* sc12, int j, int* sc, int* m) { unpack_scale_min(sc12, j, sc, m); }

// Quantize an N x K fp32 matrix (row-major) into N rows of K/bw blocks each.
// Returns 0, or -1 for an unknown format or K not a multiple of the block size.
int orc_quantize(int fmt, const float* w, int64_t N, int64_t K, uint8_t* blocks, int nthreads) {
  const int bw = block_weights(fmt), bb = block_bytes(fmt);
  if (bw == 0 || K % bw != 0) return -1;
  const int64_t nb = K / bw;
#pragma omp parallel for schedule(static) num_threads(nthreads > 0 ? nthreads : 1)
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t b = 0; b < nb; ++b) {
      const float* src = w + n * K + b * bw;
      uint8_t* dst = blocks + (n * nb + b) * bb;
      if (fmt == ORC_Q8_0) quant_q8_0(src, dst);
      else if (fmt == ORC_Q4_K) quant_q4_k(src, dst);
      else if (fmt == ORC_Q5_K) quant_q5_k(src, dst);
      else if (fmt == ORC_Q6_K) quant_q6_k(src, dst);
      else quant_affine4(src, dst);
    }
  }
  return 0;
}

// Dequantize N rows into an N x K fp64 matrix.
int orc_dequant(int fmt, const uint8_t* blocks, int64_t N, int64_t K, double* out) {
  const int bw = block_weights(fmt), bb = block_bytes(fmt);
  if (bw == 0 || K % bw != 0) return -1;
  for (int64_t n = 0; n < N; ++n) deq_row(fmt, blocks + n * (K / bw) * bb, K, out + n * K);
  return 0;
}

// y[j*N + n] = sum_k deq(W)[n][k] * x[j*K + k]   (fp64, k ascending)
// absy[j*N + n] = sum_k |deq(W)[n][k] * x[j*K + k]|  (the tolerance base)
// OpenMP over output rows n only; the result does not depend on nthreads.
int orc_gemv(int fmt, const uint8_t* blocks, int x_dtype, const void* x, int64_t M, int64_t N,
             int64_t K, double* y, double* absy, int nthreads) {
  const int bw = block_weights(fmt), bb = block_bytes(fmt);
  if (bw == 0 || K % bw != 0 || (x_dtype != ORC_F32 && x_dtype != ORC_BF16)) return -1;
  const int64_t row_bytes = (K / bw) * bb;
#pragma omp parallel num_threads(nthreads > 0 ? nthreads : 1)
  {
    std::vector<double> wrow((size_t)K);
    std::vector<double> xd((size_t)(M * K));
    for (int64_t i = 0; i < M * K; ++i) xd[(size_t)i] = x_at(x_dtype, x, i);
#pragma omp for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
      deq_row(fmt, blocks + n * row_bytes, K, wrow.data());
      for (int64_t j = 0; j < M; ++j) {
        double acc = 0.0, aacc = 0.0;
        const double* xj = xd.data() + j * K;
        for (int64_t k = 0; k < K; ++k) {
          const double p = wrow[(size_t)k] * xj[k];
          acc += p;
          aacc += std::fabs(p);
        }
        y[j * N + n] = acc;
        if (absy) absy[j * N + n] = aacc;
      }
    }
  }
  return 0;
}

// The same sum for a list of (j, n) output coordinates only.
int orc_gemv_sampled(int fmt, const uint8_t* blocks, int x_dtype, const void* x, int64_t M,
                     int64_t N, int64_t K, int64_t npairs, const int64_t* js, const int64_t* ns,
                     double* y, double* absy, int nthreads) {
  const int bw = block_weights(fmt), bb = block_bytes(fmt);
  if (bw == 0 || K % bw != 0 || (x_dtype != ORC_F32 && x_dtype != ORC_BF16)) return -1;
  const int64_t row_bytes = (K / bw) * bb;
  for (int64_t p = 0; p < npairs; ++p)
    if (js[p] < 0 || js[p] >= M || ns[p] < 0 || ns[p] >= N) return -2;
#pragma omp parallel num_threads(nthreads > 0 ? nthreads : 1)
  {
    std::vector<double> wrow((size_t)K);
#pragma omp for schedule(static)
    for (int64_t p = 0; p < npairs; ++p) {
      deq_row(fmt, blocks + ns[p] * row_bytes, K, wrow.data());
      double acc = 0.0, aacc = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        const double prod = wrow[(size_t)k] * x_at(x_dtype, x, js[p] * K + k);
        acc += prod;
        aacc += std::fabs(prod);
      }
      y[p] = acc;
      if (absy) absy[p] = aacc;
    }
  }
  return 0;
}

}  // extern "C"
