// Scalar fp64 oracle of the shortlist output head's small copy and score bounds.
// TEST INFRASTRUCTURE ONLY (see oracle.cpp's header); no code shared with the CUDA path.
//
// The method (Kinetic README, "What makes it fast", the paragraph on choosing the next
// token): an output layer of up to a quarter of a million rows is read for every token;
// each row's score is first bounded from a small copy of the layer, and exact scores are
// computed only for the rows whose bound still lets them win. The pages name neither the
// copy nor the bound; the reading used here:
//   * the head is Q8_0; the small copy is its Q4_K quantization (each 256-weight super-block
//     of deq(W), exact in fp32, through the Q4_K covering quantizer: 144 bytes per 256
//     weights against 272, i.e. 53 % of the bytes, in the cheapest format to stream);
//   * the per-row bound of |score - approximate score| is, by Cauchy-Schwarz,
//     r_n * ||x||_2 with r_n = ||w_n - w'_n||_2 (w' = the small copy's values), plus a
//     floating-point allowance c_K * (||w_n||_2 + A_n) * ||x||_2 that covers the fp32
//     rounding of both the exact and the approximate GPU products:
//       c_K = K * 2^-22 (four times K units of fp32 roundoff),
//       A_n = sqrt(32 * sum_g (15 d sc_g + dmin m_g)^2), the Cauchy-Schwarz scale of the
//             Q4_K product's scale and min terms (sub-block g, 32 weights);
//   * B_n = r_n + c_K * (||w_n|| + A_n), times (1 + 2^-32) for this fp64 evaluation's own
//     rounding, then rounded up to fp32. A row n can hold the maximum only if
//     approx_n + B_n ||x|| >= max_m (approx_m - B_m ||x||).
// This file writes the small copy's bytes and B_n; the argmax itself is the plain
// definition (the largest exact score, ties to the lowest row), taken from orc_gemv.
#include <cmath>
#include <cstdint>
#include <vector>

extern "C" int orc_quantize(int fmt, const float* w, int64_t N, int64_t K, uint8_t* blocks, int nthreads);
extern "C" int orc_dequant(int fmt, const uint8_t* blocks, int64_t N, int64_t K, double* out);
extern "C" double orc_half_to_double(uint16_t h);
extern "C" void orc_unpack_scale_min(const uint8_t* sc12, int j, int* sc, int* m);

namespace {

constexpr int kQ8_0 = 1, kQ4_K = 2;

// The smallest fp32 value >= v (v finite, non-negative here).
float f32_round_up(double v) {
  float f = static_cast<float>(v);
  if (static_cast<double>(f) < v) f = std::nextafter(f, INFINITY);
  return f;
}

}  // namespace

extern "C" {

// w_q8: N rows of K/32 Q8_0 blocks (34 bytes). small: N rows of K/256 Q4_K blocks
// (144 bytes). bound: N floats (B_n above). Returns 0, or -1 on bad arguments.
int orc_shortlist_build(const uint8_t* w_q8, int64_t N, int64_t K, uint8_t* small, float* bound, int nthreads) {
  if (N < 0 || K <= 0 || K % 256 != 0) return -1;
  const int64_t nb = K / 32, qrow = nb * 34, srow = (K / 256) * 144;
  const double cK = static_cast<double>(K) * std::ldexp(1.0, -22);
#pragma omp parallel num_threads(nthreads > 0 ? nthreads : 1)
  {
    std::vector<double> w((size_t)K), ws((size_t)K);
    std::vector<float> wf((size_t)K);
#pragma omp for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
      orc_dequant(kQ8_0, w_q8 + n * qrow, 1, K, w.data());
      for (int64_t k = 0; k < K; ++k) wf[(size_t)k] = static_cast<float>(w[(size_t)k]);  // exact
      uint8_t* srow_p = small + n * srow;
      orc_quantize(kQ4_K, wf.data(), 1, K, srow_p, 1);
      orc_dequant(kQ4_K, srow_p, 1, K, ws.data());
      double rr = 0.0, ww = 0.0, aa = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        const double e = w[(size_t)k] - ws[(size_t)k];
        rr += e * e;
        ww += w[(size_t)k] * w[(size_t)k];
      }
      for (int64_t g = 0; g < nb; ++g) {
        const uint8_t* blk = srow_p + (g / 8) * 144;  // fp16 d, dmin little-endian, then the scales
        const double d = orc_half_to_double(static_cast<uint16_t>(blk[0] | (blk[1] << 8)));
        const double dmin = orc_half_to_double(static_cast<uint16_t>(blk[2] | (blk[3] << 8)));
        int sc = 0, m = 0;
        orc_unpack_scale_min(blk + 4, static_cast<int>(g % 8), &sc, &m);
        const double t = 15.0 * d * sc + dmin * m;
        aa += t * t;
      }
      const double B = std::sqrt(rr) + cK * (std::sqrt(ww) + std::sqrt(32.0 * aa));
      bound[n] = f32_round_up(B * (1.0 + std::ldexp(1.0, -32)));
    }
  }
  return 0;
}

}  // extern "C"
