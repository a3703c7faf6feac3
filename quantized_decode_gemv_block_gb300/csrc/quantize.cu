// GPU quantizers: fp32 weights -> Q8_0 / Q4_K / affine4 blocks, in fp64.
//
// They make synthetic test and benchmark data (the GEMV itself never quantizes).
// Block layouts follow GGUF (Kinetic README, "Switching from llama.cpp": GGUF files
// and llama.cpp's Q8_0/Q4_K bytes unchanged) and, for affine4, the scale + bias per
// 32 weights of the Kipp README ("How fast"). The scales are chosen by a covering
// scheme with a provable bound |w - deq(q(w))| <= step/2 (not llama.cpp's search):
//   Q8_0    d = fp16_rn(max|w| / 127); q = clamp(round_half_away(w / d), -127, 127)
//   Q4_K    per sub-block lo = min(0, min w), hi = max(0, max w), mraw = -lo;
//           dmin = smallest fp16 >= max(mraw) / 63, m = ceil(mraw / dmin);
//           t = hi + dmin*m; d = smallest fp16 >= max(t) / 945; sc = ceil(t / (15 d));
//           q = round_half_away((w + dmin*m) / (d*sc)), which lies in [0, 15]
//   affine4 b = largest fp16 <= min w; s = smallest fp16 >= (max w - b) / 15;
//           q = clamp(round_half_away((w - b) / s), 0, 15)
// Every fp64 operation is an explicitly rounded intrinsic so that no contraction
// changes a rounding decision. If a rounding step ever pushed a 6-bit scale or
// min past 63, its fp16 step is raised by one code and the step repeated.
#include "kq_device.cuh"
#include "kq_internal.h"

namespace kq {
namespace {

__device__ __forceinline__ double h2d(uint16_t h) {
  return static_cast<double>(__half2float(__ushort_as_half(h)));
}
__device__ __forceinline__ uint16_t d2h_rn(double v) {
  return __half_as_ushort(__double2half(v));
}
__device__ __forceinline__ uint16_t h_next_up(uint16_t h) {
  if (h == 0x8000u) return 0x0001u;
  return (h & 0x8000u) ? static_cast<uint16_t>(h - 1) : static_cast<uint16_t>(h + 1);
}
__device__ __forceinline__ uint16_t h_next_down(uint16_t h) {
  if (h == 0x0000u) return 0x8001u;
  return (h & 0x8000u) ? static_cast<uint16_t>(h + 1) : static_cast<uint16_t>(h - 1);
}
__device__ __forceinline__ uint16_t d2h_up(double t) {
  uint16_t h = d2h_rn(t);
  if (h2d(h) < t) h = h_next_up(h);
  return h;
}
__device__ __forceinline__ uint16_t d2h_down(double t) {
  uint16_t h = d2h_rn(t);
  if (h2d(h) > t) h = h_next_down(h);
  return h;
}
__device__ __forceinline__ double dmin_of(double a, double b) { return (b < a) ? b : a; }
__device__ __forceinline__ double dmax_of(double a, double b) { return (a < b) ? b : a; }
// fp16 codes are written with one aligned 16-bit store (every block offset is even and
// kq_quantize requires a 2-byte aligned destination). Writing the two bytes of a code
// taken straight from cvt.rn.f16.f64 separately was measured to drop its low byte.
__device__ __forceinline__ void put16(uint8_t* p, uint16_t v) {
  *reinterpret_cast<uint16_t*>(p) = v;
}

__global__ void quant_q8_0_kernel(const float* __restrict__ w, uint8_t* __restrict__ out,
                                  long long nblk) {
  const long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (b >= nblk) return;
  const float* src = w + b * 32;
  double amax = 0.0;
  for (int i = 0; i < 32; ++i) amax = dmax_of(amax, fabs(static_cast<double>(src[i])));
  const uint16_t d16 = d2h_rn(__ddiv_rn(amax, 127.0));
  const double d = h2d(d16);
  uint8_t* dst = out + b * 34;
  put16(dst, d16);
  for (int i = 0; i < 32; ++i) {
    double qv = 0.0;
    if (d != 0.0) qv = fmin(127.0, fmax(-127.0, round(__ddiv_rn(static_cast<double>(src[i]), d))));
    dst[2 + i] = static_cast<uint8_t>(static_cast<int8_t>(static_cast<int>(qv)));
  }
}

// Q4_K (LEVELS = 15, 144-byte blocks) and Q5_K (LEVELS = 31, 176-byte blocks: the fifth
// code bit of weight i goes to bit 2c + h of qh[l], c = i/64, h = (i%64 >= 32), l = i%32).
// One super-block of 256 fp32 weights into dst; the chosen 6-bit scales and mins and the
// fp16 d and dmin are also returned (sc, m, d16, dmin16).
template <int LEVELS>
__device__ void qk_block(const float* src, uint8_t* dst, int (&sc)[8], int (&m)[8], uint16_t& d16_out,
                         uint16_t& dmin16_out) {
  constexpr int kCodes = LEVELS == 15 ? 16 : 48;  // offset of the low-nibble bytes
  double hi[8], mraw[8];
  double maxm = 0.0;
  for (int j = 0; j < 8; ++j) {
    double l = 0.0, h = 0.0;
    for (int i = 0; i < 32; ++i) {
      const double v = static_cast<double>(src[32 * j + i]);
      l = dmin_of(l, v);
      h = dmax_of(h, v);
    }
    hi[j] = h;
    mraw[j] = -l;
    maxm = dmax_of(maxm, mraw[j]);
  }
  uint16_t dmin16 = 0;
  for (int j = 0; j < 8; ++j) m[j] = 0;
  if (maxm > 0.0) {
    dmin16 = d2h_up(__ddiv_rn(maxm, 63.0));
    for (int guard = 0; guard < 64; ++guard) {
      const double dm = h2d(dmin16);
      bool ok = true;
      for (int j = 0; j < 8; ++j) {
        m[j] = static_cast<int>(ceil(__ddiv_rn(mraw[j], dm)));
        if (m[j] > 63) ok = false;
      }
      if (ok) break;
      dmin16 = h_next_up(dmin16);
    }
  }
  const double dmin = h2d(dmin16);
  double t[8], maxt = 0.0;
  for (int j = 0; j < 8; ++j) {
    t[j] = __dadd_rn(hi[j], __dmul_rn(dmin, static_cast<double>(m[j])));
    maxt = dmax_of(maxt, t[j]);
  }
  uint16_t d16 = 0;
  for (int j = 0; j < 8; ++j) sc[j] = 0;
  if (maxt > 0.0) {
    d16 = d2h_up(__ddiv_rn(maxt, 63.0 * LEVELS));
    for (int guard = 0; guard < 64; ++guard) {
      const double dd = h2d(d16);
      bool ok = true;
      for (int j = 0; j < 8; ++j) {
        sc[j] = static_cast<int>(ceil(__ddiv_rn(t[j], __dmul_rn(static_cast<double>(LEVELS), dd))));
        if (sc[j] > 63) ok = false;
      }
      if (ok) break;
      d16 = h_next_up(d16);
    }
  }
  const double d = h2d(d16);
  d16_out = d16;
  dmin16_out = dmin16;
  put16(dst, d16);
  put16(dst + 2, dmin16);
  uint8_t scales[12];
  for (int i = 0; i < 12; ++i) scales[i] = 0;
  for (int j = 0; j < 4; ++j) {
    scales[j] = static_cast<uint8_t>(scales[j] | (sc[j] & 63));
    scales[j + 4] = static_cast<uint8_t>(scales[j + 4] | (m[j] & 63));
  }
  for (int j = 4; j < 8; ++j) {
    scales[j + 4] = static_cast<uint8_t>((sc[j] & 15) | ((m[j] & 15) << 4));
    scales[j - 4] = static_cast<uint8_t>(scales[j - 4] | ((sc[j] >> 4) << 6));
    scales[j] = static_cast<uint8_t>(scales[j] | ((m[j] >> 4) << 6));
  }
  for (int i = 0; i < 12; ++i) dst[4 + i] = scales[i];
  uint8_t qh[32];
  for (int l = 0; l < 32; ++l) qh[l] = 0;
  for (int c = 0; c < 4; ++c) {
    for (int l = 0; l < 32; ++l) {
      int qq[2];
      for (int hsel = 0; hsel < 2; ++hsel) {
        const int i = 64 * c + 32 * hsel + l, j = i >> 5;
        const double step = __dmul_rn(d, static_cast<double>(sc[j]));
        int qv = 0;
        if (step != 0.0) {
          const double r = round(__ddiv_rn(
              __dadd_rn(static_cast<double>(src[i]), __dmul_rn(dmin, static_cast<double>(m[j]))),
              step));
          qv = static_cast<int>(fmin(static_cast<double>(LEVELS), fmax(0.0, r)));
        }
        qq[hsel] = qv;
        if (qv & 16) qh[l] = static_cast<uint8_t>(qh[l] | (1u << (2 * c + hsel)));
      }
      dst[kCodes + 32 * c + l] = static_cast<uint8_t>((qq[0] & 15) | ((qq[1] & 15) << 4));
    }
  }
  if (LEVELS == 31)
    for (int l = 0; l < 32; ++l) dst[16 + l] = qh[l];
}

template <int LEVELS>
__global__ void quant_qk_kernel(const float* __restrict__ w, uint8_t* __restrict__ out, long long nblk) {
  constexpr int kBytes = LEVELS == 15 ? 144 : 176;
  const long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (b >= nblk) return;
  int sc[8], m[8];
  uint16_t d16, dmin16;
  qk_block<LEVELS>(w + b * 256, out + b * kBytes, sc, m, d16, dmin16);
}

// Q6_K (GGUF): per 16-weight sub-block a = max |w|; d = smallest fp16 >= max(a)/(127*31);
// sc = ceil(a / (31 d)) <= 127; q = 32 + round_half_away(w / (d sc)) in [1, 63]. Same fp64
// operations, in the same order, as the oracle's quantizer.
__global__ void quant_q6_k_kernel(const float* __restrict__ w, uint8_t* __restrict__ out, long long nblk) {
  const long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (b >= nblk) return;
  const float* src = w + b * 256;
  double a[16];
  double amax = 0.0;
  for (int s = 0; s < 16; ++s) {
    double m = 0.0;
    for (int i = 0; i < 16; ++i) m = dmax_of(m, fabs(static_cast<double>(src[16 * s + i])));
    a[s] = m;
    amax = dmax_of(amax, m);
  }
  uint16_t d16 = 0;
  int sc[16];
  for (int s = 0; s < 16; ++s) sc[s] = 0;
  if (amax > 0.0) {
    d16 = d2h_up(__ddiv_rn(amax, 127.0 * 31.0));
    for (int guard = 0; guard < 64; ++guard) {
      const double dd = h2d(d16);
      bool ok = true;
      for (int s = 0; s < 16; ++s) {
        sc[s] = static_cast<int>(ceil(__ddiv_rn(a[s], __dmul_rn(31.0, dd))));
        if (sc[s] > 127) ok = false;
      }
      if (ok) break;
      d16 = h_next_up(d16);
    }
  }
  const double d = h2d(d16);
  uint8_t* dst = out + b * 210;
  uint8_t ql[128], qh[64];
  for (int i = 0; i < 128; ++i) ql[i] = 0;
  for (int i = 0; i < 64; ++i) qh[i] = 0;
  for (int i = 0; i < 256; ++i) {
    const double step = __dmul_rn(d, static_cast<double>(sc[i / 16]));
    int qv = 32;
    if (step != 0.0) qv = 32 + static_cast<int>(fmin(31.0, fmax(-31.0, round(__ddiv_rn(static_cast<double>(src[i]), step)))));
    const int n = i / 128, k = (i % 128) / 32, l = i % 32;
    const int qi = 64 * n + 32 * (k % 2) + l;
    ql[qi] = static_cast<uint8_t>(ql[qi] | (k < 2 ? (qv & 15) : ((qv & 15) << 4)));
    qh[32 * n + l] = static_cast<uint8_t>(qh[32 * n + l] | (((qv >> 4) & 3) << (2 * k)));
  }
  for (int i = 0; i < 128; ++i) dst[i] = ql[i];
  for (int i = 0; i < 64; ++i) dst[128 + i] = qh[i];
  for (int s = 0; s < 16; ++s) dst[192 + s] = static_cast<uint8_t>(static_cast<int8_t>(sc[s]));
  dst[208] = static_cast<uint8_t>(d16 & 0xFFu);
  dst[209] = static_cast<uint8_t>(d16 >> 8);
}

// One affine4 block of 32 fp32 weights: b, s by the covering rule, then the codes.
__device__ void affine4_block(const float* src, uint8_t* dst) {
  double mn = static_cast<double>(src[0]), mx = mn;
  for (int i = 1; i < 32; ++i) {
    const double v = static_cast<double>(src[i]);
    mn = dmin_of(mn, v);
    mx = dmax_of(mx, v);
  }
  const uint16_t b16 = d2h_down(mn);
  const double bias = h2d(b16);
  const double span = __dadd_rn(mx, -bias);
  const uint16_t s16 = span > 0.0 ? d2h_up(__ddiv_rn(span, 15.0)) : 0;
  const double s = h2d(s16);
  put16(dst, s16);
  put16(dst + 2, b16);
  for (int k = 0; k < 16; ++k) {
    int qq[2];
    for (int e = 0; e < 2; ++e) {
      int qv = 0;
      if (s != 0.0)
        qv = static_cast<int>(
            fmin(15.0, fmax(0.0, round(__ddiv_rn(__dadd_rn(static_cast<double>(src[2 * k + e]), -bias), s)))));
      qq[e] = qv;
    }
    dst[4 + k] = static_cast<uint8_t>(qq[0] | (qq[1] << 4));
  }
}

__global__ void quant_affine4_kernel(const float* __restrict__ w, uint8_t* __restrict__ out,
                                     long long nblk) {
  const long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (b >= nblk) return;
  affine4_block(w + b * 32, out + b * 20);
}

// Small copy of a Q8_0 output head for the shortlist (Kinetic README, "What makes it fast":
// every row's score is bounded from a small copy): each 256-weight super-block of deq(W)
// (d * q, exact in fp32) through the Q4_K quantizer, and per row the bound
//   B_n = ||w_n - w'_n|| + K 2^-22 (||w_n|| + sqrt(32 sum_g (15 d sc_g + dmin m_g)^2)),
// times (1 + 2^-32) for the fp64 evaluation, rounded up to fp32. The first term bounds the
// copy's error of a score per unit ||x|| (Cauchy-Schwarz); the second covers the fp32
// rounding of the exact and the approximate products (at most 4K units of roundoff each,
// against sum |w x| <= ||w|| ||x|| and the Q4_K terms' scale). One warp per row; each lane
// sums its super-blocks in fp64 and the lanes meet in a fixed butterfly.
__global__ void shortlist_build_kernel(const uint8_t* __restrict__ wq, uint8_t* __restrict__ small,
                                       float* __restrict__ bound, int N, int K) {
  const int lane = threadIdx.x & 31;
  const long long n = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  if (n >= N) return;
  const int nsb = K / 256;
  const uint8_t* qrow = wq + n * (long long)(K / 32) * 34;
  uint8_t* srow = small + n * (long long)nsb * 144;
  double rr = 0.0, ww = 0.0, aa = 0.0;
  float w[256];
  for (int g = lane; g < nsb; g += 32) {
    for (int b8 = 0; b8 < 8; ++b8) {
      const uint8_t* blk = qrow + (g * 8 + b8) * 34;
      const float d = __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t*>(blk)));
      for (int i = 0; i < 32; ++i) w[32 * b8 + i] = d * static_cast<float>(static_cast<int8_t>(blk[2 + i]));  // exact
    }
    uint8_t* dst = srow + g * 144;
    int sc[8], m[8];
    uint16_t d16, dmin16;
    qk_block<15>(w, dst, sc, m, d16, dmin16);
    const double d = h2d(d16), dmin = h2d(dmin16);
    for (int i = 0; i < 256; ++i) {
      const int j = i >> 5, c = i >> 6, l = i & 31;
      const int q = (dst[16 + 32 * c + l] >> (4 * (j & 1))) & 15;
      // exact in fp64: products of fp16 values and small integers, and their difference
      const double wc = __dadd_rn(__dmul_rn(__dmul_rn(d, static_cast<double>(sc[j])), static_cast<double>(q)),
                                  -__dmul_rn(dmin, static_cast<double>(m[j])));
      const double e = __dadd_rn(static_cast<double>(w[i]), -wc);
      rr = __dadd_rn(rr, __dmul_rn(e, e));
      ww = __dadd_rn(ww, __dmul_rn(static_cast<double>(w[i]), static_cast<double>(w[i])));
    }
    for (int j = 0; j < 8; ++j) {
      const double t = __dadd_rn(__dmul_rn(__dmul_rn(15.0, d), static_cast<double>(sc[j])),
                                 __dmul_rn(dmin, static_cast<double>(m[j])));
      aa = __dadd_rn(aa, __dmul_rn(t, t));
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    rr = __dadd_rn(rr, __shfl_xor_sync(0xffffffffu, rr, off));
    ww = __dadd_rn(ww, __shfl_xor_sync(0xffffffffu, ww, off));
    aa = __dadd_rn(aa, __shfl_xor_sync(0xffffffffu, aa, off));
  }
  if (lane == 0) {
    const double cK = static_cast<double>(K) * 0x1p-22;
    const double B = __dadd_rn(sqrt(rr), __dmul_rn(cK, __dadd_rn(sqrt(ww), sqrt(__dmul_rn(32.0, aa)))));
    bound[n] = __double2float_ru(__dmul_rn(B, 1.0 + 0x1p-32));
  }
}

}  // namespace

int launch_quantize(int fmt, const float* w, void* blocks, int N, int K, cudaStream_t stream,
                    std::string* err) {
  uint8_t* out = static_cast<uint8_t*>(blocks);
  const int bw = (fmt == FMT_Q4_K || fmt == FMT_Q5_K || fmt == FMT_Q6_K) ? 256 : 32;
  const long long nblk = (long long)N * (K / bw);
  if (nblk == 0) return 0;
  const int threads = 128;
  const long long grid = (nblk + threads - 1) / threads;
  if (fmt == FMT_Q8_0) quant_q8_0_kernel<<<(unsigned)grid, threads, 0, stream>>>(w, out, nblk);
  else if (fmt == FMT_Q4_K) quant_qk_kernel<15><<<(unsigned)grid, threads, 0, stream>>>(w, out, nblk);
  else if (fmt == FMT_Q5_K) quant_qk_kernel<31><<<(unsigned)grid, threads, 0, stream>>>(w, out, nblk);
  else if (fmt == FMT_Q6_K) quant_q6_k_kernel<<<(unsigned)grid, threads, 0, stream>>>(w, out, nblk);
  else quant_affine4_kernel<<<(unsigned)grid, threads, 0, stream>>>(w, out, nblk);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    *err = std::string("quantize launch: ") + cudaGetErrorString(e);
    return -1;
  }
  return 0;
}

int launch_shortlist_build(const void* wq, void* small, float* bound, int N, int K, cudaStream_t stream,
                           std::string* err) {
  if (N == 0) return 0;
  const int threads = 128;
  const long long grid = ((long long)N * 32 + threads - 1) / threads;
  shortlist_build_kernel<<<(unsigned)grid, threads, 0, stream>>>(static_cast<const uint8_t*>(wq),
                                                                 static_cast<uint8_t*>(small), bound, N, K);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    *err = std::string("shortlist build launch: ") + cudaGetErrorString(e);
    return -1;
  }
  return 0;
}

}  // namespace kq
