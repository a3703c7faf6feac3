// Per-format pieces of the tensor-core GEMV: how a warp reads one 256-weight unit of
// 16 rows (rows g and g+8 per thread), turns the codes into exact bf16 MMA A fragments,
// and promotes each 32-weight group's fp32 MMA result by its scale and min/bias.
// Included by gemv_mma.cu only.
#pragma once
#include "kq_device.cuh"

namespace kq {
namespace gemv {

constexpr uint32_t kBf16Magic = 0x43434343u;  // bf16 0x43nn = 128 + nn for nn < 128
constexpr uint32_t kBf16x2_128 = 0x43004300u;

struct LdGlobal {
  __device__ static uint4 v128(const void* p) { return ldg128(p); }
  __device__ static uint2 v64(const void* p) { return ldg64(p); }
  __device__ static uint32_t v32(const void* p) { return ldg32(p); }
};
struct LdShared {  // plain loads: the compiler may combine and schedule them (the stage's
                  // mbarrier wait carries a memory clobber, so none moves above it)
  __device__ static uint4 v128(const void* p) { return *static_cast<const uint4*>(p); }
  __device__ static uint2 v64(const void* p) { return *static_cast<const uint2*>(p); }
  __device__ static uint32_t v32(const void* p) { return *static_cast<const uint32_t*>(p); }
};
// ------------------------------------------------------------------ Q4_K --
// One unit = one 144-byte super-block. Thread (g, q) of a warp handles rows g and
// g+8 of the warp's 16 rows; for each 32-byte chunk c of codes it loads the 8 bytes
// 8q..8q+7, i.e. weights 8q..8q+7 of sub-block 2c (low nibbles) and of sub-block
// 2c+1 (high nibbles).
struct FmtQ4K {
  static constexpr bool kHalfX = false;
  static constexpr int kUnitBytes = 144;
  static constexpr bool kPerm0213 = false;
  static constexpr bool kNeedsSum = true;
  struct Raw {
    uint4 h[2];
    uint2 qs[2][4];
  };
  template <class Ld>
  __device__ static void load(Raw& r, const uint8_t* pa, const uint8_t* pb, int q) {
    r.h[0] = Ld::v128(pa);
    r.h[1] = Ld::v128(pb);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      r.qs[0][c] = Ld::v64(pa + 16 + 32 * c + 8 * q);
      r.qs[1][c] = Ld::v64(pb + 16 + 32 * c + 8 * q);
    }
  }
  // 4-bit codes -> bf16 pairs: slots (2q, 2q+1) <- bytes (0,1), (2q+8, 2q+9) <- bytes (2,3).
  template <int NT>
  __device__ static void compute(const Raw& r, float (&acc)[NT][4], const uint16_t* xs_unit,
                                 int xstride, const float* s_unit, int lane, int M) {
    constexpr int T = 8 * NT;
    const int g = lane >> 2, q = lane & 3;
    uint32_t sc_lo[2], sc_hi[2], m_lo[2], m_hi[2];
    float d[2], nd[2], dmin[2], pdmin[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint32_t s0 = r.h[i].y, s1 = r.h[i].z, s2 = r.h[i].w;
      sc_lo[i] = s0 & 0x3F3F3F3Fu;
      m_lo[i] = s1 & 0x3F3F3F3Fu;
      sc_hi[i] = (s2 & 0x0F0F0F0Fu) | ((s0 >> 2) & 0x30303030u);
      m_hi[i] = ((s2 >> 4) & 0x0F0F0F0Fu) | ((s1 >> 2) & 0x30303030u);
      d[i] = half_bits_to_float(r.h[i].x);
      dmin[i] = half_bits_to_float(r.h[i].x >> 16);
      nd[i] = -8388608.f * d[i];
      pdmin[i] = 8388608.f * dmin[i];
    }
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const int c = b >> 1;
      uint32_t a0[4], a1[4];
      float ds[2], ndm[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint32_t w0 = r.qs[i][c].x, w1 = r.qs[i][c].y;
        const uint32_t n0 = (b & 1) ? ((w0 >> 4) & 0x0F0F0F0Fu) : (w0 & 0x0F0F0F0Fu);
        const uint32_t n1 = (b & 1) ? ((w1 >> 4) & 0x0F0F0F0Fu) : (w1 & 0x0F0F0F0Fu);
        a0[i] = bf16x2_sub(prmt(n0, kBf16Magic, 0x4140u), kBf16x2_128);
        a0[i + 2] = bf16x2_sub(prmt(n0, kBf16Magic, 0x4342u), kBf16x2_128);
        a1[i] = bf16x2_sub(prmt(n1, kBf16Magic, 0x4140u), kBf16x2_128);
        a1[i + 2] = bf16x2_sub(prmt(n1, kBf16Magic, 0x4342u), kBf16x2_128);
        const uint32_t scw = (b < 4) ? sc_lo[i] : sc_hi[i];
        const uint32_t mw = (b < 4) ? m_lo[i] : m_hi[i];
        ds[i] = scaled_byte(scw, b & 3, d[i], nd[i]);          //  d * sc_b (exact)
        ndm[i] = scaled_byte(mw, b & 3, -dmin[i], pdmin[i]);   // -dmin * m_b (exact)
      }
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const int tok = 8 * t + g;
        uint4 xb = make_uint4(0u, 0u, 0u, 0u);
        if (tok < M) xb = lds128(xs_unit + tok * xstride + 32 * b + 8 * q);
        const float z[4] = {0.f, 0.f, 0.f, 0.f};
        float p[4];
        mma_bf16_16816(p, a0, xb.x, xb.y, z);
        mma_bf16_16816(p, a1, xb.z, xb.w, p);
        const float2 sv = lds_f2(s_unit + b * T + 8 * t + 2 * q);
        acc[t][0] = __fmaf_rn(ndm[0], sv.x, __fmaf_rn(ds[0], p[0], acc[t][0]));
        acc[t][1] = __fmaf_rn(ndm[0], sv.y, __fmaf_rn(ds[0], p[1], acc[t][1]));
        acc[t][2] = __fmaf_rn(ndm[1], sv.x, __fmaf_rn(ds[1], p[2], acc[t][2]));
        acc[t][3] = __fmaf_rn(ndm[1], sv.y, __fmaf_rn(ds[1], p[3], acc[t][3]));
      }
    }
  }
};

// ------------------------------------------------------------------ Q5_K --
// One unit = one 176-byte super-block: Q4_K's 16-byte header (d, dmin, packed 6-bit
// scales and mins), qh[32] (the fifth code bit of weight i is bit 2c + h of qh[i % 32],
// c = i/64, h = 1 for the high-nibble half; i.e. bit b for sub-block b), then Q4_K's 128
// bytes of low nibbles. Codes 0..31, w = d*sc*q - dmin*m.
struct FmtQ5K {
  static constexpr bool kHalfX = false;
  static constexpr int kUnitBytes = 176;
  static constexpr bool kPerm0213 = false;
  static constexpr bool kNeedsSum = true;
  struct Raw {
    uint4 h[2];
    uint2 qs[2][4];
    uint2 qh[2];  // fifth bits of weights 8q..8q+7 of every sub-block (bit b for sub-block b)
  };
  template <class Ld>
  __device__ static void load(Raw& r, const uint8_t* pa, const uint8_t* pb, int q) {
    r.h[0] = Ld::v128(pa);
    r.h[1] = Ld::v128(pb);
    r.qh[0] = Ld::v64(pa + 16 + 8 * q);
    r.qh[1] = Ld::v64(pb + 16 + 8 * q);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      r.qs[0][c] = Ld::v64(pa + 48 + 32 * c + 8 * q);
      r.qs[1][c] = Ld::v64(pb + 48 + 32 * c + 8 * q);
    }
  }
  // 4-bit codes -> bf16 pairs: slots (2q, 2q+1) <- bytes (0,1), (2q+8, 2q+9) <- bytes (2,3).
  template <int NT>
  __device__ static void compute(const Raw& r, float (&acc)[NT][4], const uint16_t* xs_unit,
                                 int xstride, const float* s_unit, int lane, int M) {
    constexpr int T = 8 * NT;
    const int g = lane >> 2, q = lane & 3;
    uint32_t sc_lo[2], sc_hi[2], m_lo[2], m_hi[2];
    float d[2], nd[2], dmin[2], pdmin[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint32_t s0 = r.h[i].y, s1 = r.h[i].z, s2 = r.h[i].w;
      sc_lo[i] = s0 & 0x3F3F3F3Fu;
      m_lo[i] = s1 & 0x3F3F3F3Fu;
      sc_hi[i] = (s2 & 0x0F0F0F0Fu) | ((s0 >> 2) & 0x30303030u);
      m_hi[i] = ((s2 >> 4) & 0x0F0F0F0Fu) | ((s1 >> 2) & 0x30303030u);
      d[i] = half_bits_to_float(r.h[i].x);
      dmin[i] = half_bits_to_float(r.h[i].x >> 16);
      nd[i] = -8388608.f * d[i];
      pdmin[i] = 8388608.f * dmin[i];
    }
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const int c = b >> 1;
      uint32_t a0[4], a1[4];
      float ds[2], ndm[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint32_t w0 = r.qs[i][c].x, w1 = r.qs[i][c].y;
        // 5-bit codes: the nibble plus 16 * (bit b of the weight's qh byte), each < 32
        const uint32_t n0 = ((b & 1) ? ((w0 >> 4) & 0x0F0F0F0Fu) : (w0 & 0x0F0F0F0Fu)) |
                            (((r.qh[i].x >> b) & 0x01010101u) << 4);
        const uint32_t n1 = ((b & 1) ? ((w1 >> 4) & 0x0F0F0F0Fu) : (w1 & 0x0F0F0F0Fu)) |
                            (((r.qh[i].y >> b) & 0x01010101u) << 4);
        a0[i] = bf16x2_sub(prmt(n0, kBf16Magic, 0x4140u), kBf16x2_128);
        a0[i + 2] = bf16x2_sub(prmt(n0, kBf16Magic, 0x4342u), kBf16x2_128);
        a1[i] = bf16x2_sub(prmt(n1, kBf16Magic, 0x4140u), kBf16x2_128);
        a1[i + 2] = bf16x2_sub(prmt(n1, kBf16Magic, 0x4342u), kBf16x2_128);
        const uint32_t scw = (b < 4) ? sc_lo[i] : sc_hi[i];
        const uint32_t mw = (b < 4) ? m_lo[i] : m_hi[i];
        ds[i] = scaled_byte(scw, b & 3, d[i], nd[i]);          //  d * sc_b (exact)
        ndm[i] = scaled_byte(mw, b & 3, -dmin[i], pdmin[i]);   // -dmin * m_b (exact)
      }
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const int tok = 8 * t + g;
        uint4 xb = make_uint4(0u, 0u, 0u, 0u);
        if (tok < M) xb = lds128(xs_unit + tok * xstride + 32 * b + 8 * q);
        const float z[4] = {0.f, 0.f, 0.f, 0.f};
        float p[4];
        mma_bf16_16816(p, a0, xb.x, xb.y, z);
        mma_bf16_16816(p, a1, xb.z, xb.w, p);
        const float2 sv = lds_f2(s_unit + b * T + 8 * t + 2 * q);
        acc[t][0] = __fmaf_rn(ndm[0], sv.x, __fmaf_rn(ds[0], p[0], acc[t][0]));
        acc[t][1] = __fmaf_rn(ndm[0], sv.y, __fmaf_rn(ds[0], p[1], acc[t][1]));
        acc[t][2] = __fmaf_rn(ndm[1], sv.x, __fmaf_rn(ds[1], p[2], acc[t][2]));
        acc[t][3] = __fmaf_rn(ndm[1], sv.y, __fmaf_rn(ds[1], p[3], acc[t][3]));
      }
    }
  }
};

// ------------------------------------------------------------------ Q8_0 --
// One unit = 8 blocks of 34 bytes = 272 bytes, read as 4 pairs of 68 bytes. The
// even block of a pair starts on a 4-byte boundary (its codes 2 bytes after it),
// the odd block's codes start on one. Thread q takes codes 8q..8q+7 of each block.
// The fp16 scale of the even block sits in the first word of thread 0's window
// and that of the odd block in the last word of thread 3's; they are broadcast in
// the quad with shuffles.
struct FmtQ8_0 {
  static constexpr bool kHalfX = false;
  static constexpr bool kRowCopies = false;
  static constexpr int kUnitBytes = 272;
  static constexpr bool kPerm0213 = true;
  static constexpr bool kNeedsSum = false;
  struct Raw {
    uint32_t w[2][4][5];
  };
  template <class Ld>
  __device__ static void load(Raw& r, const uint8_t* pa, const uint8_t* pb, int q) {
#pragma unroll
    for (int p = 0; p < 4; ++p) {
#pragma unroll
      for (int k = 0; k < 3; ++k) {
        r.w[0][p][k] = Ld::v32(pa + 68 * p + 8 * q + 4 * k);
        r.w[1][p][k] = Ld::v32(pb + 68 * p + 8 * q + 4 * k);
      }
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        r.w[0][p][3 + k] = Ld::v32(pa + 68 * p + 36 + 8 * q + 4 * k);
        r.w[1][p][3 + k] = Ld::v32(pb + 68 * p + 36 + 8 * q + 4 * k);
      }
    }
  }
  // int8 pair (bytes 0 and 2, or 1 and 3) -> exact bf16 pair: (128 + (q & 127)) - (128 or 256).
  __device__ static uint32_t i8pair(uint32_t v) {
    return bf16x2_sub(and_or(v, 0x007F007Fu, kBf16x2_128), and_or(v, 0x00800080u, kBf16x2_128));
  }
  template <int NT>
  __device__ static void compute(const Raw& r, float (&acc)[NT][4], const uint16_t* xs_unit,
                                 int xstride, const float* /*s_unit*/, int lane, int M) {
    const int g = lane >> 2, q = lane & 3;
    const int quad = lane & ~3;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
#pragma unroll
      for (int odd = 0; odd < 2; ++odd) {
        const int b = 2 * p + odd;
        uint32_t a0[4], a1[4];
        float dsc[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          uint32_t c0, c1;
          if (!odd) {
            c0 = prmt(r.w[i][p][0], r.w[i][p][1], 0x5432u);
            c1 = prmt(r.w[i][p][1], r.w[i][p][2], 0x5432u);
          } else {
            c0 = r.w[i][p][3];
            c1 = r.w[i][p][4];
          }
          const uint32_t dw = __shfl_sync(0xFFFFFFFFu, odd ? r.w[i][p][2] : r.w[i][p][0],
                                          quad | (odd ? 3 : 0));
          dsc[i] = half_bits_to_float(odd ? (dw >> 16) : dw);
          a0[i] = i8pair(c0);
          a0[i + 2] = i8pair(c0 >> 8);
          a1[i] = i8pair(c1);
          a1[i + 2] = i8pair(c1 >> 8);
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const int tok = 8 * t + g;
          uint4 xb = make_uint4(0u, 0u, 0u, 0u);
          if (tok < M) xb = lds128(xs_unit + tok * xstride + 32 * b + 8 * q);
          const float z[4] = {0.f, 0.f, 0.f, 0.f};
          float pr[4];
          mma_bf16_16816(pr, a0, xb.x, xb.y, z);
          mma_bf16_16816(pr, a1, xb.z, xb.w, pr);
          acc[t][0] = __fmaf_rn(dsc[0], pr[0], acc[t][0]);
          acc[t][1] = __fmaf_rn(dsc[0], pr[1], acc[t][1]);
          acc[t][2] = __fmaf_rn(dsc[1], pr[2], acc[t][2]);
          acc[t][3] = __fmaf_rn(dsc[1], pr[3], acc[t][3]);
        }
      }
    }
  }
};

// --------------------------------------------------------------- affine4 --
// One unit = 8 groups of 20 bytes = 160 bytes. Group g: word 0 = (s, b) fp16, then
// 16 code bytes; thread q takes code bytes 4q..4q+3 (weights 8q..8q+7; even weight in
// the low nibble).
struct FmtAffine4 {
  static constexpr bool kHalfX = false;
  static constexpr bool kRowCopies = false;
  static constexpr int kUnitBytes = 160;
  static constexpr bool kPerm0213 = true;
  static constexpr bool kNeedsSum = true;
  struct Raw {
    uint32_t sb[2][8];
    uint32_t cw[2][8];
  };
  template <class Ld>
  __device__ static void load(Raw& r, const uint8_t* pa, const uint8_t* pb, int q) {
#pragma unroll
    for (int gi = 0; gi < 8; ++gi) {
      r.sb[0][gi] = Ld::v32(pa + 20 * gi);
      r.sb[1][gi] = Ld::v32(pb + 20 * gi);
      r.cw[0][gi] = Ld::v32(pa + 20 * gi + 4 + 4 * q);
      r.cw[1][gi] = Ld::v32(pb + 20 * gi + 4 + 4 * q);
    }
  }
  template <int NT>
  __device__ static void compute(const Raw& r, float (&acc)[NT][4], const uint16_t* xs_unit,
                                 int xstride, const float* s_unit, int lane, int M) {
    constexpr int T = 8 * NT;
    const int g = lane >> 2, q = lane & 3;
#pragma unroll
    for (int gi = 0; gi < 8; ++gi) {
      uint32_t a0[4], a1[4];
      float s[2], bias[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint32_t cw = r.cw[i][gi];
        const uint32_t lo = cw & 0x0F0F0F0Fu, hi = (cw >> 4) & 0x0F0F0F0Fu;
        a0[i] = bf16x2_sub(prmt(lo, kBf16Magic, 0x4140u), kBf16x2_128);      // w0, w2
        a0[i + 2] = bf16x2_sub(prmt(hi, kBf16Magic, 0x4140u), kBf16x2_128);  // w1, w3
        a1[i] = bf16x2_sub(prmt(lo, kBf16Magic, 0x4342u), kBf16x2_128);      // w4, w6
        a1[i + 2] = bf16x2_sub(prmt(hi, kBf16Magic, 0x4342u), kBf16x2_128);  // w5, w7
        s[i] = half_bits_to_float(r.sb[i][gi]);
        bias[i] = half_bits_to_float(r.sb[i][gi] >> 16);
      }
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const int tok = 8 * t + g;
        uint4 xb = make_uint4(0u, 0u, 0u, 0u);
        if (tok < M) xb = lds128(xs_unit + tok * xstride + 32 * gi + 8 * q);
        const float z[4] = {0.f, 0.f, 0.f, 0.f};
        float p[4];
        mma_bf16_16816(p, a0, xb.x, xb.y, z);
        mma_bf16_16816(p, a1, xb.z, xb.w, p);
        const float2 sv = lds_f2(s_unit + gi * T + 8 * t + 2 * q);
        acc[t][0] = __fmaf_rn(bias[0], sv.x, __fmaf_rn(s[0], p[0], acc[t][0]));
        acc[t][1] = __fmaf_rn(bias[0], sv.y, __fmaf_rn(s[0], p[1], acc[t][1]));
        acc[t][2] = __fmaf_rn(bias[1], sv.x, __fmaf_rn(s[1], p[2], acc[t][2]));
        acc[t][3] = __fmaf_rn(bias[1], sv.y, __fmaf_rn(s[1], p[3], acc[t][3]));
      }
    }
  }
};

template <int FMT> struct FmtOf;
template <> struct FmtOf<FMT_Q4_K> { using type = FmtQ4K; };
template <> struct FmtOf<FMT_Q8_0> { using type = FmtQ8_0; };
template <> struct FmtOf<FMT_AFFINE4> { using type = FmtAffine4; };
template <> struct FmtOf<FMT_Q5_K> { using type = FmtQ5K; };

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }


// ------------------------------------------------------- Q4_K, fp16 path --
// The streaming kernel's Q4_K variant. Each thread of a quad owns whole sub-blocks:
// thread q reads the 32 code bytes 32q..32q+31 of its two rows' super-block, i.e. all
// of sub-block 2q (low nibbles) and sub-block 2q+1 (high nibbles). The 6-bit scale is
// folded into the fp16 A operand (sc*q <= 945 is exact in fp16), so one MMA may mix
// the four threads' sub-blocks and the fp32 result needs one promotion by d per
// super-block. The min term sum_b dmin*m_b*S_b(x) is one more MMA per super-block with
// A = m_b (exact) and B = S_b/64 split into an fp16 high and low part.
//
// The activations are staged as fp16 after an exact per-token power-of-two scale
// 2^e (max |x| of the CTA's slice lands in [2^14, 2^15)); every bf16 value within a
// factor 2^28 of that maximum converts exactly. The scale is removed when a partial
// is emitted (exact power-of-two multiply).
//
// MMA m (0..15) of a super-block takes, for thread q, weights 64q + 4m + {0,2 | 1,3}
// (m < 8, low nibbles of code word m) or 64q + 32 + 4(m-8) + {0,2 | 1,3} (m >= 8,
// high nibbles of word m-8): slots (2q, 2q+1) get the pair (+0, +2), slots (2q+8,
// 2q+9) the pair (+1, +3). The staged x of each thread's 64 positions is permuted the
// same way within groups of four, so B fragments are plain 16-byte loads.
// Scales and mins of one K-quant super-block row (Q4_K and Q5_K share the 12-byte packing:
// s0 = scales[0..3], s1 = scales[4..7], s2 = scales[8..11]) for thread q, which owns
// sub-blocks a = 2q and b = 2q + 1. For j < 4: sc_j = scales[j] & 63, m_j = scales[j+4] & 63;
// for j >= 4: sc_j = (scales[j+4] & 15) | (scales[j-4] >> 6) << 4 and
// m_j = (scales[j+4] >> 4) | (scales[j] >> 6) << 4. Threads 0, 1 take the first form and
// threads 2, 3 the second; both are one masked formula over the same two permutes, with
// per-thread masks, so no lane computes a form it then discards.
struct KqHeadConst {
  uint32_t sel_p, sel_l, m_p, m_h, m_l, m_l4;
};
__device__ __forceinline__ KqHeadConst kq_head_const(int q) {
  const uint32_t ja = static_cast<uint32_t>((2 * q) & 3);
  KqHeadConst c;
  c.sel_p = ja | ((ja + 1) << 4) | ((ja + 4) << 8) | ((ja + 5) << 12);  // s0.ja, s0.ja+1, s1.ja, s1.ja+1
  c.sel_l = ja | ((ja + 1) << 4) | (ja << 8) | ((ja + 1) << 12);        // s2.ja, s2.ja+1, s2.ja, s2.ja+1
  const bool lo_form = q < 2;
  c.m_p = lo_form ? 0x3F3F3F3Fu : 0u;          // the 6-bit values themselves
  c.m_h = lo_form ? 0u : 0x30303030u;          // bits 6, 7 of s0 / s1 bytes, as bits 4, 5
  c.m_l = lo_form ? 0u : 0x00000F0Fu;          // sc: low nibble of the s2 byte
  c.m_l4 = lo_form ? 0u : 0x0F0F0000u;         // m: high nibble of the s2 byte
  return c;
}
// From the row's 16-byte header h (d | dmin, s0, s1, s2): sa = (sc_a, sc_a), nsa = -1024 sc_a,
// sb16 = (sc_b / 16, sc_b / 16), nsb64 = -64 sc_b, mm = (m_a, m_b) as exact fp16 pairs, and
// d, dmin in fp32. 1024 + v and 64 + v/16 (v < 64) are exact fp16 values, so each pair is one
// permute (v under the exponent byte 0x64 or 0x54) and one subtraction.
__device__ __forceinline__ void kq_head(const uint4& h, const KqHeadConst& c, uint32_t& sa, uint32_t& nsa,
                                        uint32_t& sb16, uint32_t& nsb64, uint32_t& mm, float& d, float& dmin) {
  const uint32_t P = prmt(h.y, h.z, c.sel_p);
  const uint32_t L = prmt(h.w, h.w, c.sel_l);
  // bytes (sc_a, sc_b, m_a, m_b)
  const uint32_t v = (P & c.m_p) | ((P >> 2) & c.m_h) | (L & c.m_l) | ((L >> 4) & c.m_l4);
  sa = h2_sub(prmt(v, 0x64646464u, 0x4040u), 0x64006400u);
  nsa = h2_mul(sa, 0xE400E400u);
  sb16 = h2_sub(prmt(v, 0x54545454u, 0x4141u), 0x54005400u);
  nsb64 = h2_mul(sb16, 0xE400E400u);
  mm = h2_sub(prmt(v, 0x64646464u, 0x4342u), 0x64006400u);
  d = half_bits_to_float(h.x);
  dmin = half_bits_to_float(h.x >> 16);
}

struct FmtQ4KH {
  static constexpr bool kHalfX = true;
  static constexpr bool kRowCopies = false;
  static constexpr bool kPerm0213 = false;
  static constexpr bool kNeedsSum = false;
  static constexpr int kXq = 16;  // bytes between threads q of a token's staged super-block
  static constexpr int kUnitBytes = 144;
  struct Raw {
    uint4 h[2];
    uint4 c[2][2];
  };
  template <class Ld>
  __device__ static void load(Raw& r, const uint8_t* pa, const uint8_t* pb, int q) {
    r.h[0] = Ld::v128(pa);
    r.h[1] = Ld::v128(pb);
    r.c[0][0] = Ld::v128(pa + 16 + 32 * q);
    r.c[0][1] = Ld::v128(pa + 32 + 32 * q);
    r.c[1][0] = Ld::v128(pb + 16 + 32 * q);
    r.c[1][1] = Ld::v128(pb + 32 + 32 * q);
  }
  // Byte offset, within one token's 512-byte super-block slot, of the 16-byte chunk i
  // (0..7) of thread q: the quad's four chunks i sit side by side (64 bytes), and tokens
  // are 64 bytes apart modulo 128, so a quarter-warp's loads hit 32 distinct banks.
  __device__ static int chunk_off(int q, int i) { return 64 * i + 16 * q; }
  // Byte offset, within a token's 512-byte super-block slot, of the staged 16-byte chunk holding
  // values 32j + 8v .. +7 (pairs (0,2) (1,3) (4,6) (5,7)): sub-block j belongs to thread j / 2.
  __device__ static int stage_chunk(int j, int v) { return chunk_off(j >> 1, 4 * (j & 1) + v); }

  // xh_unit: token 0's slot of this super-block; xts: token stride (bytes).
  // s2_unit: token 0's min-term operands of this super-block; s2ts: their token stride.
  // The fp32 sums of one super-block: ps = sum (sc*q)*x per (row, token) and mn = sum m*S/64.
  // xo[t] / so[t]: byte offsets of this thread's token row in tile t within the staged x
  // and min-term operands (absent tokens point at the zero row), 16q / 8q included.
  template <int NT>
  __device__ static void sums(const Raw& r, const uint8_t* xh_unit, const int (&xo)[NT],
                              const uint8_t* s2_unit, const int (&so)[NT], int lane,
                              float (&ps)[NT][4], float (&mnv)[NT][4], float (&d)[2], float (&dmin)[2]) {
    const uint32_t kMagic = 0x64006400u;   // fp16 1024 in both halves
    uint32_t sa[2], nsa[2], sb16[2], nsb64[2], mm[2];
    const KqHeadConst hc = kq_head_const(lane & 3);
#pragma unroll
    for (int i = 0; i < 2; ++i) kq_head(r.h[i], hc, sa[i], nsa[i], sb16[i], nsb64[i], mm[i], d[i], dmin[i]);
    // two accumulation chains (low and high nibbles), added at the end; the first MMA of
    // each starts from zero
    float p[NT][2][4];
    const float z0[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k = 0; k < 8; ++k) {  // code word k: MMA k (low nibbles) and MMA 8+k (high nibbles)
      uint32_t alo[4], ahi[4];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint4 cv = r.c[i][k >> 2];
        const uint32_t w = (k & 3) == 0 ? cv.x : (k & 3) == 1 ? cv.y : (k & 3) == 2 ? cv.z : cv.w;
        const uint32_t w8 = w >> 8;
        alo[i] = h2_fma(and_or(w, 0x000F000Fu, kMagic), sa[i], nsa[i]);
        alo[i + 2] = h2_fma(and_or(w8, 0x000F000Fu, kMagic), sa[i], nsa[i]);
        ahi[i] = h2_fma(and_or(w, 0x00F000F0u, kMagic), sb16[i], nsb64[i]);
        ahi[i + 2] = h2_fma(and_or(w8, 0x00F000F0u, kMagic), sb16[i], nsb64[i]);
      }
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        // chunk i = k/2 holds MMAs 2i, 2i+1 of the low half; chunk 4 + k/2 of the high half
        const uint8_t* base = xh_unit + xo[t];
        const uint4 xlo = *reinterpret_cast<const uint4*>(base + 64 * (k >> 1));
        const uint4 xhi = *reinterpret_cast<const uint4*>(base + 64 * (4 + (k >> 1)));
        const uint32_t bl0 = (k & 1) ? xlo.z : xlo.x, bl1 = (k & 1) ? xlo.w : xlo.y;
        const uint32_t bh0 = (k & 1) ? xhi.z : xhi.x, bh1 = (k & 1) ? xhi.w : xhi.y;
        if (k == 0) {
          mma_f16_16816(p[t][0], alo, bl0, bl1, z0);
          mma_f16_16816(p[t][1], ahi, bh0, bh1, z0);
        } else {
          mma_f16_16816(p[t][0], alo, bl0, bl1, p[t][0]);
          mma_f16_16816(p[t][1], ahi, bh0, bh1, p[t][1]);
        }
      }
    }
    // min term: A2 slots (2q, 2q+1) and (2q+8, 2q+9) both = (m_2q, m_2q+1); B2 = the high
    // parts (S_2q, S_2q+1)/64, then the low parts
    const uint32_t a2[4] = {mm[0], mm[1], mm[0], mm[1]};
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const uint2 b2 = *reinterpret_cast<const uint2*>(s2_unit + so[t]);
      mma_f16_16816(mnv[t], a2, b2.x, b2.y, z0);
#pragma unroll
      for (int e = 0; e < 4; ++e) ps[t][e] = p[t][0][e] + p[t][1][e];
    }
  }

  // acc += (d*ps - 64*dmin*mn) * 2^-e, rows g (elements 0, 1) and g+8 (elements 2, 3); iv[t]
  // holds 2^-e of this super-block's activations for the thread's tokens 8t+2q and 8t+2q+1
  // (the products above are in units of 2^e; removing it is exact unless the result is
  // subnormal)
  template <int NT>
  __device__ static void promote(float (&acc)[NT][4], const float (&ps)[NT][4], const float (&mnv)[NT][4],
                                 const float (&d)[2], const float (&dmin)[2], const float2 (&iv)[NT]) {
    const float nd0 = -64.f * dmin[0], nd1 = -64.f * dmin[1];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      acc[t][0] = __fmaf_rn(__fmaf_rn(d[0], ps[t][0], nd0 * mnv[t][0]), iv[t].x, acc[t][0]);
      acc[t][1] = __fmaf_rn(__fmaf_rn(d[0], ps[t][1], nd0 * mnv[t][1]), iv[t].y, acc[t][1]);
      acc[t][2] = __fmaf_rn(__fmaf_rn(d[1], ps[t][2], nd1 * mnv[t][2]), iv[t].x, acc[t][2]);
      acc[t][3] = __fmaf_rn(__fmaf_rn(d[1], ps[t][3], nd1 * mnv[t][3]), iv[t].y, acc[t][3]);
    }
  }

  // iv_unit: 2^-e of token 0 for this super-block (16 tokens per super-block, 16 floats apart);
  // io[t]: this thread's first token of tile t within it (8t + 2q)
  template <int NT>
  __device__ static void compute(const Raw& r, float (&acc)[NT][4], const uint8_t* xh_unit,
                                 const int (&xo)[NT], const uint8_t* s2_unit, const int (&so)[NT],
                                 const float* iv_unit, const int (&io)[NT], int lane) {
    float ps[NT][4], mnv[NT][4], d[2], dmin[2];
    float2 iv[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) iv[t] = lds_f2(iv_unit + io[t]);
    sums<NT>(r, xh_unit, xo, s2_unit, so, lane, ps, mnv, d, dmin);
    promote<NT>(acc, ps, mnv, d, dmin, iv);
  }

};

// ------------------------------------------------------- Q5_K, fp16 path --
// FmtQ4KH's arithmetic with 5-bit codes: the fifth bit joins the code inside the fp16
// magic word before the fma that forms sc*q (<= 63*31 = 1953, still an exact fp16
// integer; the fused fma rounds once, so (1024 + 31)*63 never has to fit fp16).
struct FmtQ5KH {
  static constexpr bool kHalfX = true;
  static constexpr bool kRowCopies = false;
  static constexpr bool kPerm0213 = false;
  static constexpr bool kNeedsSum = false;
  static constexpr int kXq = 16;  // bytes between threads q of a token's staged super-block
  static constexpr int kUnitBytes = 176;
  struct Raw {
    uint4 h[2];
    uint4 c[2][2];
    uint4 qh[2][2];  // all 32 fifth-bit bytes of each row (thread q needs bits 2q, 2q+1)
  };
  template <class Ld>
  __device__ static void load(Raw& r, const uint8_t* pa, const uint8_t* pb, int q) {
    r.h[0] = Ld::v128(pa);
    r.h[1] = Ld::v128(pb);
    r.qh[0][0] = Ld::v128(pa + 16);
    r.qh[0][1] = Ld::v128(pa + 32);
    r.qh[1][0] = Ld::v128(pb + 16);
    r.qh[1][1] = Ld::v128(pb + 32);
    r.c[0][0] = Ld::v128(pa + 48 + 32 * q);
    r.c[0][1] = Ld::v128(pa + 64 + 32 * q);
    r.c[1][0] = Ld::v128(pb + 48 + 32 * q);
    r.c[1][1] = Ld::v128(pb + 64 + 32 * q);
  }
  // Byte offset, within one token's 512-byte super-block slot, of the 16-byte chunk i
  // (0..7) of thread q: the quad's four chunks i sit side by side (64 bytes), and tokens
  // are 64 bytes apart modulo 128, so a quarter-warp's loads hit 32 distinct banks.
  __device__ static int chunk_off(int q, int i) { return 64 * i + 16 * q; }
  // Byte offset, within a token's 512-byte super-block slot, of the staged 16-byte chunk holding
  // values 32j + 8v .. +7 (pairs (0,2) (1,3) (4,6) (5,7)): sub-block j belongs to thread j / 2.
  __device__ static int stage_chunk(int j, int v) { return chunk_off(j >> 1, 4 * (j & 1) + v); }

  // xh_unit: token 0's slot of this super-block; xts: token stride (bytes).
  // s2_unit: token 0's min-term operands of this super-block; s2ts: their token stride.
  // The fp32 sums of one super-block: ps = sum (sc*q)*x per (row, token) and mn = sum m*S/64.
  // xo[t] / so[t]: byte offsets of this thread's token row in tile t within the staged x
  // and min-term operands (absent tokens point at the zero row), 16q / 8q included.
  template <int NT>
  __device__ static void sums(const Raw& r, const uint8_t* xh_unit, const int (&xo)[NT],
                              const uint8_t* s2_unit, const int (&so)[NT], int lane,
                              float (&ps)[NT][4], float (&mnv)[NT][4], float (&d)[2], float (&dmin)[2]) {
    const int q = lane & 3;
    const uint32_t kMagic = 0x64006400u;   // fp16 1024 in both halves
    uint32_t sa[2], nsa[2], sb16[2], nsb64[2], mm[2];
    const KqHeadConst hc = kq_head_const(lane & 3);
#pragma unroll
    for (int i = 0; i < 2; ++i) kq_head(r.h[i], hc, sa[i], nsa[i], sb16[i], nsb64[i], mm[i], d[i], dmin[i]);
    // two accumulation chains (low and high nibbles), added at the end; the first MMA of
    // each starts from zero
    float p[NT][2][4];
    const float z0[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k = 0; k < 8; ++k) {  // code word k: MMA k (low nibbles) and MMA 8+k (high nibbles)
      uint32_t alo[4], ahi[4];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint4 cv = r.c[i][k >> 2];
        const uint32_t w = (k & 3) == 0 ? cv.x : (k & 3) == 1 ? cv.y : (k & 3) == 2 ? cv.z : cv.w;
        const uint32_t w8 = w >> 8;
        // fifth bits of the same four weights l = 4k..4k+3: bit 2q (low nibbles) and bit
        // 2q+1 (high nibbles) of qh[l]; as fp16 they add 16 to 1024 + q (bit 4 of the
        // word) or 256 to 1024 + 16q (bit 8)
        const uint4 hv = r.qh[i][k >> 2];
        const uint32_t hw = ((k & 3) == 0 ? hv.x : (k & 3) == 1 ? hv.y : (k & 3) == 2 ? hv.z : hv.w) >> (2 * q);
        alo[i] = h2_fma(and_or(w, 0x000F000Fu, and_or(hw << 4, 0x00100010u, kMagic)), sa[i], nsa[i]);
        alo[i + 2] = h2_fma(and_or(w8, 0x000F000Fu, and_or(hw >> 4, 0x00100010u, kMagic)), sa[i], nsa[i]);
        ahi[i] = h2_fma(and_or(w, 0x00F000F0u, and_or(hw << 7, 0x01000100u, kMagic)), sb16[i], nsb64[i]);
        ahi[i + 2] = h2_fma(and_or(w8, 0x00F000F0u, and_or(hw >> 1, 0x01000100u, kMagic)), sb16[i], nsb64[i]);
      }
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        // chunk i = k/2 holds MMAs 2i, 2i+1 of the low half; chunk 4 + k/2 of the high half
        const uint8_t* base = xh_unit + xo[t];
        const uint4 xlo = *reinterpret_cast<const uint4*>(base + 64 * (k >> 1));
        const uint4 xhi = *reinterpret_cast<const uint4*>(base + 64 * (4 + (k >> 1)));
        const uint32_t bl0 = (k & 1) ? xlo.z : xlo.x, bl1 = (k & 1) ? xlo.w : xlo.y;
        const uint32_t bh0 = (k & 1) ? xhi.z : xhi.x, bh1 = (k & 1) ? xhi.w : xhi.y;
        if (k == 0) {
          mma_f16_16816(p[t][0], alo, bl0, bl1, z0);
          mma_f16_16816(p[t][1], ahi, bh0, bh1, z0);
        } else {
          mma_f16_16816(p[t][0], alo, bl0, bl1, p[t][0]);
          mma_f16_16816(p[t][1], ahi, bh0, bh1, p[t][1]);
        }
      }
    }
    // min term: A2 slots (2q, 2q+1) and (2q+8, 2q+9) both = (m_2q, m_2q+1); B2 = the high
    // parts (S_2q, S_2q+1)/64, then the low parts
    const uint32_t a2[4] = {mm[0], mm[1], mm[0], mm[1]};
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const uint2 b2 = *reinterpret_cast<const uint2*>(s2_unit + so[t]);
      mma_f16_16816(mnv[t], a2, b2.x, b2.y, z0);
#pragma unroll
      for (int e = 0; e < 4; ++e) ps[t][e] = p[t][0][e] + p[t][1][e];
    }
  }

  // acc += (d*ps - 64*dmin*mn) * 2^-e, rows g (elements 0, 1) and g+8 (elements 2, 3); iv[t]
  // holds 2^-e of this super-block's activations for the thread's tokens 8t+2q and 8t+2q+1
  // (the products above are in units of 2^e; removing it is exact unless the result is
  // subnormal)
  template <int NT>
  __device__ static void promote(float (&acc)[NT][4], const float (&ps)[NT][4], const float (&mnv)[NT][4],
                                 const float (&d)[2], const float (&dmin)[2], const float2 (&iv)[NT]) {
    const float nd0 = -64.f * dmin[0], nd1 = -64.f * dmin[1];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      acc[t][0] = __fmaf_rn(__fmaf_rn(d[0], ps[t][0], nd0 * mnv[t][0]), iv[t].x, acc[t][0]);
      acc[t][1] = __fmaf_rn(__fmaf_rn(d[0], ps[t][1], nd0 * mnv[t][1]), iv[t].y, acc[t][1]);
      acc[t][2] = __fmaf_rn(__fmaf_rn(d[1], ps[t][2], nd1 * mnv[t][2]), iv[t].x, acc[t][2]);
      acc[t][3] = __fmaf_rn(__fmaf_rn(d[1], ps[t][3], nd1 * mnv[t][3]), iv[t].y, acc[t][3]);
    }
  }

  // iv_unit: 2^-e of token 0 for this super-block (16 tokens per super-block, 16 floats apart);
  // io[t]: this thread's first token of tile t within it (8t + 2q)
  template <int NT>
  __device__ static void compute(const Raw& r, float (&acc)[NT][4], const uint8_t* xh_unit,
                                 const int (&xo)[NT], const uint8_t* s2_unit, const int (&so)[NT],
                                 const float* iv_unit, const int (&io)[NT], int lane) {
    float ps[NT][4], mnv[NT][4], d[2], dmin[2];
    float2 iv[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) iv[t] = lds_f2(iv_unit + io[t]);
    sums<NT>(r, xh_unit, xo, s2_unit, so, lane, ps, mnv, d, dmin);
    promote<NT>(acc, ps, mnv, d, dmin, iv);
  }

};


// ------------------------------------------------------- Q8_0, fp16 path --
// The Q8_0 unit (eight 34-byte blocks) against fp16 activations under the staging's exact
// per-(token, super-block) 2^e (shared with FmtQ4KH): an int8 pair becomes an exact fp16 pair
// with one LOP3 and one subtraction. LOP3 with table 0x6A computes mask ? (v ^ c) : c; with
// mask = the low byte of each half and c = 0x6480 per half it keeps bits 0..6 of the code,
// flips bit 7 (q + 128 as an unsigned byte) and puts fp16 1024 above them: 1024 + 128 + q,
// and subtracting 1152 leaves q (integers below 2048 are exact in fp16). Thread q takes codes
// 8q..8q+7 of every block, the pairs (0, 2) and (1, 3) of each four as FmtQ8_0 does, so the
// staged x of each block is in natural chunk order (the staging's pair packing gives 0213).
__device__ __forceinline__ uint32_t i8pair_h(uint32_t v) {  // bytes 0 and 2 -> fp16 pair, exact
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(v), "r"(0x00FF00FFu), "r"(0x64806480u));
  return h2_sub(d, 0x64806480u);
}

struct FmtQ8_0H {
  static constexpr bool kHalfX = true;
  static constexpr bool kRowCopies = false;
  static constexpr int kXq = 16;  // bytes between threads q of a token's staged super-block
  static constexpr int kUnitBytes = 272;
  using Raw = FmtQ8_0::Raw;
  // FmtQ8_0's words, with 8-byte loads where the offset allows (units and stage rows are
  // 8-byte aligned): block pair p starts at 68p, so words 8q.. are 8-aligned for even p and
  // words 36 + 8q.. for odd p; 10 loads per row instead of 20.
  template <class Ld>
  __device__ static void load(Raw& r, const uint8_t* pa, const uint8_t* pb, int q) {
    const uint8_t* rows[2] = {pa, pb};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const uint8_t* b = rows[i] + 68 * p + 8 * q;
        if ((p & 1) == 0) {
          const uint2 v = Ld::v64(b);
          r.w[i][p][0] = v.x;
          r.w[i][p][1] = v.y;
          r.w[i][p][2] = Ld::v32(b + 8);
          r.w[i][p][3] = Ld::v32(b + 36);
          r.w[i][p][4] = Ld::v32(b + 40);
        } else {
          r.w[i][p][0] = Ld::v32(b);
          const uint2 v = Ld::v64(b + 4);
          r.w[i][p][1] = v.x;
          r.w[i][p][2] = v.y;
          const uint2 u = Ld::v64(b + 36);
          r.w[i][p][3] = u.x;
          r.w[i][p][4] = u.y;
        }
      }
    }
  }
  // Byte offset, within a token's 512-byte super-block slot, of the staged 16-byte chunk
  // holding values 32j + 8v .. +7: block j, thread v.
  __device__ static int stage_chunk(int j, int v) { return 64 * j + 16 * v; }

  template <int NT>
  __device__ static void compute(const Raw& r, float (&acc)[NT][4], const uint8_t* xh_unit, const int (&xo)[NT],
                                 const uint8_t* /*s2_unit*/, const int (&/*so*/)[NT], const float* iv_unit,
                                 const int (&io)[NT], int lane) {
    const int quad = lane & ~3;
    float u[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t) u[t][0] = u[t][1] = u[t][2] = u[t][3] = 0.f;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
#pragma unroll
      for (int odd = 0; odd < 2; ++odd) {
        const int b = 2 * p + odd;
        uint32_t a0[4], a1[4];
        float dsc[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          uint32_t c0, c1;
          if (!odd) {
            c0 = prmt(r.w[i][p][0], r.w[i][p][1], 0x5432u);
            c1 = prmt(r.w[i][p][1], r.w[i][p][2], 0x5432u);
          } else {
            c0 = r.w[i][p][3];
            c1 = r.w[i][p][4];
          }
          const uint32_t dw = __shfl_sync(0xFFFFFFFFu, odd ? r.w[i][p][2] : r.w[i][p][0], quad | (odd ? 3 : 0));
          dsc[i] = half_bits_to_float(odd ? (dw >> 16) : dw);
          a0[i] = i8pair_h(c0);
          a0[i + 2] = i8pair_h(c0 >> 8);
          a1[i] = i8pair_h(c1);
          a1[i + 2] = i8pair_h(c1 >> 8);
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const uint4 xb = *reinterpret_cast<const uint4*>(xh_unit + xo[t] + 64 * b);
          const float z[4] = {0.f, 0.f, 0.f, 0.f};
          float pr[4];
          mma_f16_16816(pr, a0, xb.x, xb.y, z);
          mma_f16_16816(pr, a1, xb.z, xb.w, pr);
          u[t][0] = __fmaf_rn(dsc[0], pr[0], u[t][0]);
          u[t][1] = __fmaf_rn(dsc[0], pr[1], u[t][1]);
          u[t][2] = __fmaf_rn(dsc[1], pr[2], u[t][2]);
          u[t][3] = __fmaf_rn(dsc[1], pr[3], u[t][3]);
        }
      }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const float2 iv = lds_f2(iv_unit + io[t]);
      acc[t][0] = __fmaf_rn(u[t][0], iv.x, acc[t][0]);
      acc[t][1] = __fmaf_rn(u[t][1], iv.y, acc[t][1]);
      acc[t][2] = __fmaf_rn(u[t][2], iv.x, acc[t][2]);
      acc[t][3] = __fmaf_rn(u[t][3], iv.y, acc[t][3]);
    }
  }
};

// ------------------------------------------------------- Q6_K, fp16 path --
// One unit = one 210-byte super-block: ql[128], qh[64], int8 scales[16], fp16 d. Weight w:
// half n = w / 128, quarter kq = (w % 128) / 32, l = w % 32; code q = (ql[64n + 32(kq % 2) + l]
// >> 4 (kq >= 2)) & 15 | ((qh[32n + l] >> 2kq) & 3) << 4; w = d * scales[w / 16] * (q - 32).
// Rows are only 2-byte aligned (210-byte blocks), so the streaming kernel copies each row's
// 16-byte-aligned covering span into its stage row (kRowCopies) and a unit starts at an even
// offset there; a 4-byte word is read as the two aligned words around it joined by a permute.
// MMA s (0..15) is sub-block s (16 weights, one scale): n = s / 8, kq = (s / 2) % 4, l = 16 (s % 2)
// + 4q + {0..3} for thread q, whose slots (2q, 2q+1) take the weights (+0, +2) and (2q+8, 2q+9)
// the weights (+1, +3); the staged x of every group of four is in the order (0 2 1 3) (what the
// staging's pair packing gives in natural chunk order), so a B fragment is one 8-byte load.
// A = q - 32 is exact in fp16; sc * (q - 32) is not (up to 127 * 32), so each sub-block's fp32
// MMA result is promoted by its scale, and d and 2^-e once per super-block.
__device__ __forceinline__ uint32_t lds_u32_a2(uint32_t a) {  // a: 2-byte aligned shared address
  uint32_t w0, w1;
  asm("ld.shared.u32 %0, [%1];" : "=r"(w0) : "r"(a & ~3u));
  asm("ld.shared.u32 %0, [%1];" : "=r"(w1) : "r"((a & ~3u) + 4u));
  return prmt(w0, w1, (a & 2u) ? 0x5432u : 0x3210u);
}

struct FmtQ6KH {
  static constexpr bool kHalfX = true;
  static constexpr bool kRowCopies = true;
  static constexpr int kUnitBytes = 210;
  static constexpr int kXq = 8;  // bytes between threads q of a token's staged super-block
  struct Raw {
    uint32_t ql[2][8];  // [row][4n + 2(kq % 2) + s % 2]: ql bytes 64n + 32(kq % 2) + 16(s % 2) + 4q .. +3
    uint32_t qh[2][4];  // [row][2n + s % 2]: qh bytes 32n + 16(s % 2) + 4q .. +3
    uint32_t sc[2][4];  // [row][i]: scales 4i .. 4i+3
    uint32_t d[2];      // [row]: fp16 d in the low half
  };
  // pa / pb: the unit of rows g / g+8 in shared memory (2-byte aligned)
  template <class Ld>
  __device__ static void load(Raw& r, const uint8_t* pa, const uint8_t* pb, int q) {
    const uint32_t a[2] = {smem_addr(pa), smem_addr(pb)};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
#pragma unroll
      for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int k2 = 0; k2 < 2; ++k2) r.ql[i][4 * n + 2 * k2 + h] = lds_u32_a2(a[i] + 64 * n + 32 * k2 + 16 * h + 4 * q);
          r.qh[i][2 * n + h] = lds_u32_a2(a[i] + 128 + 32 * n + 16 * h + 4 * q);
        }
#pragma unroll
      for (int k = 0; k < 4; ++k) r.sc[i][k] = lds_u32_a2(a[i] + 192 + 4 * k);
      r.d[i] = lds_u32_a2(a[i] + 208);
    }
  }
  __device__ static int stage_chunk(int j, int v) { return 64 * j + 16 * v; }

  template <int NT>
  __device__ static void compute(const Raw& r, float (&acc)[NT][4], const uint8_t* xh_unit, const int (&xo)[NT],
                                 const uint8_t* /*s2_unit*/, const int (&/*so*/)[NT], const float* iv_unit,
                                 const int (&io)[NT], int /*lane*/) {
    float u[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t) u[t][0] = u[t][1] = u[t][2] = u[t][3] = 0.f;
#pragma unroll
    for (int sb = 0; sb < 16; ++sb) {
      const int n = sb >> 3, kq = (sb >> 1) & 3, h = sb & 1;
      uint32_t a[4];
      float scf[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint32_t ql = r.ql[i][4 * n + 2 * (kq & 1) + h], qh = r.qh[i][2 * n + h];
        const uint32_t nib = (kq >= 2 ? ql >> 4 : ql) & 0x0F0F0F0Fu;
        const uint32_t hb = kq == 0 ? (qh << 4) : kq == 1 ? (qh << 2) : kq == 2 ? qh : (qh >> 2);
        const uint32_t qw = nib | (hb & 0x30303030u);  // the four 6-bit codes, one per byte
        // (1024 + q) per half from bytes 0, 2 and 1, 3, minus 1056: q - 32, exact
        a[i] = h2_sub(and_or(qw, 0x003F003Fu, 0x64006400u), 0x64206420u);
        a[i + 2] = h2_sub(and_or(qw >> 8, 0x003F003Fu, 0x64006400u), 0x64206420u);
        // the sub-block's int8 scale as fp32: (b ^ 0x80) in the mantissa of 2^23, minus 2^23 + 128
        const uint32_t sbyte = prmt(r.sc[i][sb >> 2] ^ 0x80808080u, 0x4B000000u, 0x7650u | (sb & 3));
        scf[i] = __fsub_rn(__uint_as_float(sbyte), 8388736.f);
      }
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const uint2 b = *reinterpret_cast<const uint2*>(xh_unit + xo[t] + 32 * sb);
        const float z[4] = {0.f, 0.f, 0.f, 0.f};
        float p[4];
        mma_f16_16816(p, a, b.x, b.y, z);
        u[t][0] = __fmaf_rn(scf[0], p[0], u[t][0]);
        u[t][1] = __fmaf_rn(scf[0], p[1], u[t][1]);
        u[t][2] = __fmaf_rn(scf[1], p[2], u[t][2]);
        u[t][3] = __fmaf_rn(scf[1], p[3], u[t][3]);
      }
    }
    const float d0 = half_bits_to_float(r.d[0]), d1 = half_bits_to_float(r.d[1]);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const float2 iv = lds_f2(iv_unit + io[t]);
      acc[t][0] = __fmaf_rn(d0 * u[t][0], iv.x, acc[t][0]);
      acc[t][1] = __fmaf_rn(d0 * u[t][1], iv.y, acc[t][1]);
      acc[t][2] = __fmaf_rn(d1 * u[t][2], iv.x, acc[t][2]);
      acc[t][3] = __fmaf_rn(d1 * u[t][3], iv.y, acc[t][3]);
    }
  }
};

// Staging of one CTA's K-slice of the activations for FmtQ4KH / FmtQ5KH (all threads of the
// CTA take part). x: M x K bf16. Slice = super-blocks [k0, k0+S).
// Every (token, super-block) gets its own power-of-two scale 2^e with max|x| * 2^e in
// [2^14, 2^15) over its 256 values (from the bits of max|x|, an fp32 pattern; zero, Inf and
// NaN keep 2^0): every bf16 value within a factor 2^28 of that maximum converts to fp16
// exactly, and the scale depends on the token's own values only (never on M).
__device__ __forceinline__ float token_scale(uint32_t mb) {
  const int E = static_cast<int>(mb >> 23);
  int e = 0;
  if (mb != 0u && E < 255) {
    e = 14 - (E == 0 ? -126 : E - 127);
    e = max(-126, min(127, e));
  }
  return __int_as_float((e + 127) << 23);
}

// Two phases, so the loads of x leave before any conversion work: load() reads this thread's
// items into registers (and clears the zero row and the scales of absent tokens); finish()
// takes each (token, super-block) maximum across the eight lanes that hold its 256 values
// (no shared-memory atomics, no barrier), converts, stores, and writes the min-term operands
// and 2^-e. The caller places one __syncthreads after finish().
// Rows 0..M-1 of the staged x hold the tokens, row M zeros (absent token slots read it).
// iv: 2^-e per (super-block, token), 16 floats per super-block.
template <int NTHREADS, class F>
struct StageQ4KH {
  static_assert(NTHREADS % 32 == 0, "an item's eight lanes must share a warp");
  static constexpr int kItems = 5;  // 16 tokens x 10 super-blocks x 8 groups / 256 threads
  uint4 u[kItems][4];

  __device__ void load(const uint16_t* x, int M, int K, int k0, int S, uint8_t* xh, int xts, uint8_t* s2,
                       int s2ts, float* iv) {
    const int items = M * S * 8;
#pragma unroll
    for (int it = 0; it < kItems; ++it) {
      const int idx = threadIdx.x + it * NTHREADS;
      if (idx < items) {
        const int tok = idx / (S * 8), grp = idx - tok * (S * 8);
        const uint16_t* src = x + (long long)tok * K + (long long)k0 * 256 + grp * 32;
#pragma unroll
        for (int v = 0; v < 4; ++v) u[it][v] = ldg128(src + 8 * v);
      }
    }
    for (int i = threadIdx.x; i < S * 32; i += NTHREADS)
      *reinterpret_cast<uint4*>(xh + M * xts + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
    for (int i = threadIdx.x; i < S * 4; i += NTHREADS)
      *reinterpret_cast<uint2*>(s2 + M * s2ts + 8 * i) = make_uint2(0u, 0u);
    for (int i = threadIdx.x; i < S * 16; i += NTHREADS)
      if ((i & 15) >= M) iv[i] = 0.f;
  }

  __device__ void finish(int M, int S, uint8_t* xh, int xts, uint8_t* s2, int s2ts, float* iv) {
    const int items = M * S * 8;
#pragma unroll
    for (int it = 0; it < kItems; ++it) {
      if (it * NTHREADS >= items) break;  // uniform over the CTA
      const int idx = threadIdx.x + it * NTHREADS;
      const bool act = idx < items;
      uint32_t best = 0u;
      if (act) {
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const uint32_t w4[4] = {u[it][v].x, u[it][v].y, u[it][v].z, u[it][v].w};
#pragma unroll
          for (int k = 0; k < 4; ++k) best = max(best, max((w4[k] & 0x7FFFu) << 16, w4[k] & 0x7FFF0000u));
        }
      }
      // lanes 8a..8a+7 hold groups 0..7 of one (token, super-block): S * 8 items per token
      best = max(best, __shfl_xor_sync(0xFFFFFFFFu, best, 1));
      best = max(best, __shfl_xor_sync(0xFFFFFFFFu, best, 2));
      best = max(best, __shfl_xor_sync(0xFFFFFFFFu, best, 4));
      if (act) {
        const int tok = idx / (S * 8), grp = idx - tok * (S * 8);
        const int ul = grp >> 3, j = grp & 7, q = j >> 1, half = j & 1;
        const float sc = token_scale(best);
        if (j == 0) iv[ul * 16 + tok] = 1.0f / sc;  // exact: a power of two
        float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const uint4 w = u[it][v];
          const float f0 = __uint_as_float(w.x << 16) * sc, f1 = __uint_as_float(w.x & 0xFFFF0000u) * sc;
          const float f2 = __uint_as_float(w.y << 16) * sc, f3 = __uint_as_float(w.y & 0xFFFF0000u) * sc;
          const float f4 = __uint_as_float(w.z << 16) * sc, f5 = __uint_as_float(w.z & 0xFFFF0000u) * sc;
          const float f6 = __uint_as_float(w.w << 16) * sc, f7 = __uint_as_float(w.w & 0xFFFF0000u) * sc;
          const uint4 o = make_uint4(f2_to_h2(f0, f2), f2_to_h2(f1, f3), f2_to_h2(f4, f6), f2_to_h2(f5, f7));
          *reinterpret_cast<uint4*>(xh + tok * xts + ul * 512 + F::stage_chunk(j, v)) = o;
          // the sum of what the MMA will see (the fp16 values), four partial sums in a fixed order
          const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            a[k] += half_bits_to_float(ow[k]);
            a[k] += half_bits_to_float(ow[k] >> 16);
          }
        }
        const float hs = ((a[0] + a[1]) + (a[2] + a[3])) * 0.015625f;  // S / 64
        const uint32_t hh = f2_to_h2(hs, 0.f) & 0xFFFFu;
        const uint32_t hl = f2_to_h2(hs - h_lo_to_f(hh), 0.f) & 0xFFFFu;
        uint16_t* s2h = reinterpret_cast<uint16_t*>(s2 + tok * s2ts + ul * 32 + 8 * q);
        s2h[half] = static_cast<uint16_t>(hh);      // (S_2q, S_2q+1) / 64, high parts
        s2h[2 + half] = static_cast<uint16_t>(hl);  // then the low parts
      }
    }
  }
};

}  // namespace gemv
}  // namespace kq
