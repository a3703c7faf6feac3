// Tensor-core GEMV / speculative-verify kernels for bf16 activations, M = 1..16.
//
// Computes Y[j][n] = sum_k deq(W)[n][k] * X[j][k] for block-quantized W (Kinetic
// README, "What makes it fast": a decode step reads every weight once per token, a
// speculative check runs all guesses through one pass over the weights).
//
// Layout of the work:
//  * A CTA owns 128 consecutive rows of W (8 warps x 16 rows) and one K-slice.
//    When N alone gives too few CTAs to keep the HBM busy, K is split across the
//    CTAs of a thread-block cluster (2, 4 or 8); their partial sums meet in
//    distributed shared memory and are added in rank order. The split depends on
//    (N, K, SM count) only, never on M.
//  * Each warp streams its 16 rows with 8- and 16-byte read-only loads, two
//    256-weight units ahead, and dequantizes in registers to exact bf16 codes
//    (4-bit codes and int8 codes are exact in bf16).
//  * mma.sync m16n8k16 (bf16 in, fp32 accumulate) multiplies 16 weight rows by
//    8 token columns per instruction; tokens 8..15 take a second column tile.
//    The activations of the CTA's K-slice are staged once in shared memory, in
//    the order the B fragments need, together with the per-32 sums of x used by
//    the min/bias terms.
//  * Per 32-weight group the fp32 MMA result is promoted by its scale with one
//    FMA, and the min/bias term is added with a second FMA against the staged
//    sum of x: acc += (d*sc)*P - (dmin*m)*S (Q4_K), acc += d*P (Q8_0),
//    acc += s*P + b*S (affine4).
//
// Batch invariance (Kinetic README, "What makes it fast", last paragraph: every row
// of a batch is summed in the same order as that token alone): a token column's
// arithmetic is the same instruction sequence for every M. M only predicates the
// activation loads (absent tokens read as zero) and the stores, and the column
// tile count (1 or 2) leaves tile 0 unchanged.
#include <cooperative_groups.h>

#include "kq_device.cuh"
#include "kq_internal.h"

namespace cg = cooperative_groups;

namespace kq {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRowsPerCta = 16 * kWarps;
constexpr int kUnit = 256;       // weights per K-unit (one Q4_K super-block, 8 Q8_0 / affine4 blocks)
constexpr int kChunkUnits = 8;   // K-units of activations staged in shared memory at a time
constexpr int kDepth = 2;        // K-units each warp keeps in flight
constexpr uint32_t kBf16Magic = 0x43434343u;  // bf16 0x43nn = 128 + nn for nn < 128
constexpr uint32_t kBf16x2_128 = 0x43004300u;

struct Params {
  const uint8_t* w;
  const uint16_t* x;
  float* y;
  int M, N, K;
  int units;        // K / 256
  int ks;           // K-split (cluster size)
  int chunk_units;  // staging granularity
  int xstride;      // staged row stride, in bf16 elements
  long long row_bytes;
};

// ------------------------------------------------------------------ Q4_K --
// One unit = one 144-byte super-block. Thread (g, q) of a warp handles rows g and
// g+8 of the warp's 16 rows; for each 32-byte chunk c of codes it loads the 8 bytes
// 8q..8q+7, i.e. weights 8q..8q+7 of sub-block 2c (low nibbles) and of sub-block
// 2c+1 (high nibbles).
struct FmtQ4K {
  static constexpr int kUnitBytes = 144;
  static constexpr bool kPerm0213 = false;
  static constexpr bool kNeedsSum = true;
  struct Raw {
    uint4 h[2];
    uint2 qs[2][4];
  };
  __device__ static void load(Raw& r, const uint8_t* pa, const uint8_t* pb, int q) {
    r.h[0] = ldg128(pa);
    r.h[1] = ldg128(pb);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      r.qs[0][c] = ldg64(pa + 16 + 32 * c + 8 * q);
      r.qs[1][c] = ldg64(pb + 16 + 32 * c + 8 * q);
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

// ------------------------------------------------------------------ Q8_0 --
// One unit = 8 blocks of 34 bytes = 272 bytes, read as 4 pairs of 68 bytes. The
// even block of a pair starts on a 4-byte boundary (its codes 2 bytes after it),
// the odd block's codes start on one. Thread q takes codes 8q..8q+7 of each block.
// The fp16 scale of the even block sits in the first word of thread 0's window
// and that of the odd block in the last word of thread 3's; they are broadcast in
// the quad with shuffles.
struct FmtQ8_0 {
  static constexpr int kUnitBytes = 272;
  static constexpr bool kPerm0213 = true;
  static constexpr bool kNeedsSum = false;
  struct Raw {
    uint32_t w[2][4][5];
  };
  __device__ static void load(Raw& r, const uint8_t* pa, const uint8_t* pb, int q) {
#pragma unroll
    for (int p = 0; p < 4; ++p) {
#pragma unroll
      for (int k = 0; k < 3; ++k) {
        r.w[0][p][k] = ldg32(pa + 68 * p + 8 * q + 4 * k);
        r.w[1][p][k] = ldg32(pb + 68 * p + 8 * q + 4 * k);
      }
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        r.w[0][p][3 + k] = ldg32(pa + 68 * p + 36 + 8 * q + 4 * k);
        r.w[1][p][3 + k] = ldg32(pb + 68 * p + 36 + 8 * q + 4 * k);
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
  static constexpr int kUnitBytes = 160;
  static constexpr bool kPerm0213 = true;
  static constexpr bool kNeedsSum = true;
  struct Raw {
    uint32_t sb[2][8];
    uint32_t cw[2][8];
  };
  __device__ static void load(Raw& r, const uint8_t* pa, const uint8_t* pb, int q) {
#pragma unroll
    for (int gi = 0; gi < 8; ++gi) {
      r.sb[0][gi] = ldg32(pa + 20 * gi);
      r.sb[1][gi] = ldg32(pb + 20 * gi);
      r.cw[0][gi] = ldg32(pa + 20 * gi + 4 + 4 * q);
      r.cw[1][gi] = ldg32(pb + 20 * gi + 4 + 4 * q);
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

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Stage X[0:M][uc*256 : (uc+nun)*256] into shared memory (B-fragment order) and, when the
// format has a min or bias term, the fp32 sum of each 32-group of every token.
template <class F, int T>
__device__ void stage_x(const Params& p, uint16_t* xs, float* ss, int uc, int nun) {
  const int per_tok = nun * 32;  // 16-byte vectors per token
  for (int idx = threadIdx.x; idx < p.M * per_tok; idx += kThreads) {
    const int tok = idx / per_tok, v = idx - tok * per_tok;
    uint4 val = ldg128(p.x + (long long)tok * p.K + (long long)uc * kUnit + v * 8);
    if (F::kPerm0213) {  // (e0 e1 e2 e3) -> (e0 e2 e1 e3) within each group of four
      const uint4 o = val;
      val.x = prmt(o.x, o.y, 0x5410u);
      val.y = prmt(o.x, o.y, 0x7632u);
      val.z = prmt(o.z, o.w, 0x5410u);
      val.w = prmt(o.z, o.w, 0x7632u);
    }
    *reinterpret_cast<uint4*>(xs + tok * p.xstride + v * 8) = val;
  }
  if (F::kNeedsSum) {
    for (int idx = threadIdx.x; idx < T * nun * 8; idx += kThreads) {
      const int grp = idx / T, tok = idx - grp * T;
      float s = 0.f;
      if (tok < p.M) {
        const uint16_t* src = p.x + (long long)tok * p.K + (long long)uc * kUnit + grp * 32;
        float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const uint4 u = ldg128(src + 8 * v);
          a[0] += bf16_lo(u.x); a[1] += bf16_hi(u.x); a[2] += bf16_lo(u.y); a[3] += bf16_hi(u.y);
          a[0] += bf16_lo(u.z); a[1] += bf16_hi(u.z); a[2] += bf16_lo(u.w); a[3] += bf16_hi(u.w);
        }
        s = (a[0] + a[1]) + (a[2] + a[3]);
      }
      ss[grp * T + tok] = s;
    }
  }
}

template <int FMT, int NT>
__global__ void __launch_bounds__(kThreads, 2) gemv_mma_kernel(const Params p) {
  using F = typename FmtOf<FMT>::type;
  constexpr int T = 8 * NT;
  extern __shared__ __align__(16) uint8_t smem[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);
  float* ss = reinterpret_cast<float*>(smem + (size_t)T * p.xstride * 2);
  float* red = ss + p.chunk_units * 8 * T;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  int rank = 0, rowblk = blockIdx.x;
  if (p.ks > 1) {
    rank = static_cast<int>(cg::this_cluster().block_rank());
    rowblk = blockIdx.x / p.ks;
  }
  const int u0 = static_cast<int>((long long)rank * p.units / p.ks);
  const int u1 = static_cast<int>((long long)(rank + 1) * p.units / p.ks);
  const int n0 = rowblk * kRowsPerCta + warp * 16;
  const int ra = min(n0 + g, p.N - 1), rb = min(n0 + g + 8, p.N - 1);
  const uint8_t* wa = p.w + (long long)ra * p.row_bytes;
  const uint8_t* wb = p.w + (long long)rb * p.row_bytes;

  float acc[NT][4];
#pragma unroll
  for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;

  typename F::Raw raw[kDepth];
#pragma unroll
  for (int i = 0; i < kDepth; ++i)
    if (u0 + i < u1)
      F::load(raw[i], wa + (long long)(u0 + i) * F::kUnitBytes,
              wb + (long long)(u0 + i) * F::kUnitBytes, q);

  int chunk0 = u0;
  for (int u = u0; u < u1; u += kDepth) {
#pragma unroll
    for (int i = 0; i < kDepth; ++i) {
      const int uu = u + i;
      if (uu < u1) {
        if ((uu - u0) % p.chunk_units == 0) {  // uniform over the CTA
          chunk0 = uu;
          __syncthreads();
          stage_x<F, T>(p, xs, ss, uu, min(p.chunk_units, u1 - uu));
          __syncthreads();
        }
        const int ul = uu - chunk0;
        F::template compute<NT>(raw[i], acc, xs + ul * kUnit, p.xstride, ss + ul * 8 * T, lane,
                                p.M);
        if (uu + kDepth < u1)
          F::load(raw[i], wa + (long long)(uu + kDepth) * F::kUnitBytes,
                  wb + (long long)(uu + kDepth) * F::kUnitBytes, q);
      }
    }
  }

  if (p.ks == 1) {
    const int na = n0 + g, nb = n0 + g + 8;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int j0 = 8 * t + 2 * q;
      if (j0 < p.M) {
        if (na < p.N) p.y[(long long)j0 * p.N + na] = acc[t][0];
        if (nb < p.N) p.y[(long long)j0 * p.N + nb] = acc[t][2];
      }
      if (j0 + 1 < p.M) {
        if (na < p.N) p.y[(long long)(j0 + 1) * p.N + na] = acc[t][1];
        if (nb < p.N) p.y[(long long)(j0 + 1) * p.N + nb] = acc[t][3];
      }
    }
    return;
  }

  // K-split: partials of this CTA's 128 rows into its shared memory, then each rank
  // adds a slice of the rows over all ranks, rank 0 first.
  const int rl = warp * 16 + g;
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const int j0 = 8 * t + 2 * q;
    red[rl * T + j0] = acc[t][0];
    red[rl * T + j0 + 1] = acc[t][1];
    red[(rl + 8) * T + j0] = acc[t][2];
    red[(rl + 8) * T + j0 + 1] = acc[t][3];
  }
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();
  const int rpr = kRowsPerCta / p.ks;
  for (int idx = threadIdx.x; idx < rpr * p.M; idx += kThreads) {
    const int row = rank * rpr + idx / p.M, tok = idx % p.M;
    float v = 0.f;
    for (int r = 0; r < p.ks; ++r) v += cluster.map_shared_rank(red, r)[row * T + tok];
    const int n = rowblk * kRowsPerCta + row;
    if (n < p.N) p.y[(long long)tok * p.N + n] = v;
  }
  cluster.sync();
}

template <int FMT, int NT>
int launch_one(const Params& prm, size_t smem, cudaStream_t stream, std::string* err) {
  auto kern = gemv_mma_kernel<FMT, NT>;
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kMaxGemvSmem);
    if (e != cudaSuccess) {
      *err = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e);
      return -1;
    }
    attr_done[dev] = true;
  }
  const int rowblks = (prm.N + kRowsPerCta - 1) / kRowsPerCta;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(rowblks * prm.ks, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  cfg.numAttrs = 0;
  if (prm.ks > 1) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = prm.ks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, prm);
  if (e != cudaSuccess) {
    *err = std::string("gemv launch: ") + cudaGetErrorString(e);
    return -1;
  }
  return 0;
}

}  // namespace

GemvPlan plan_gemv_mma(int N, int K, int num_sms) {
  GemvPlan pl;
  pl.units = K / kUnit;
  const int rowblks = (N + kRowsPerCta - 1) / kRowsPerCta;
  int ks = 1;
  while (ks < 8 && rowblks * ks < 2 * num_sms && ks * 2 <= pl.units) ks *= 2;
  pl.ks = ks;
  const int slice = (pl.units + ks - 1) / ks;
  pl.chunk_units = slice < kChunkUnits ? (slice > 0 ? slice : 1) : kChunkUnits;
  pl.grid = rowblks * ks;
  return pl;
}

size_t gemv_mma_smem(const GemvPlan& pl, int M) {
  const int T = M > 8 ? 16 : 8;
  const size_t xstride = (size_t)pl.chunk_units * kUnit + 32;
  size_t s = (size_t)T * xstride * 2 + (size_t)pl.chunk_units * 8 * T * 4;
  if (pl.ks > 1) s += (size_t)kRowsPerCta * T * 4;
  return s;
}

int launch_gemv_mma(int fmt, const void* w, const void* x, float* y, int M, int N, int K,
                    long long row_bytes, int num_sms, cudaStream_t stream, std::string* err) {
  const GemvPlan pl = plan_gemv_mma(N, K, num_sms);
  Params prm;
  prm.w = static_cast<const uint8_t*>(w);
  prm.x = static_cast<const uint16_t*>(x);
  prm.y = y;
  prm.M = M;
  prm.N = N;
  prm.K = K;
  prm.units = pl.units;
  prm.ks = pl.ks;
  prm.chunk_units = pl.chunk_units;
  prm.xstride = pl.chunk_units * kUnit + 32;
  prm.row_bytes = row_bytes;
  const size_t smem = gemv_mma_smem(pl, M);
  const bool two = M > 8;
  switch (fmt) {
    case FMT_Q4_K:
      return two ? launch_one<FMT_Q4_K, 2>(prm, smem, stream, err)
                 : launch_one<FMT_Q4_K, 1>(prm, smem, stream, err);
    case FMT_Q8_0:
      return two ? launch_one<FMT_Q8_0, 2>(prm, smem, stream, err)
                 : launch_one<FMT_Q8_0, 1>(prm, smem, stream, err);
    case FMT_AFFINE4:
      return two ? launch_one<FMT_AFFINE4, 2>(prm, smem, stream, err)
                 : launch_one<FMT_AFFINE4, 1>(prm, smem, stream, err);
  }
  *err = "unsupported format";
  return -1;
}

}  // namespace kq
