// Decode attention of a verify window over a KV cache (grouped-query heads).
//
// A speculative step checks its M guesses in one pass (Kinetic README, "What makes it
// fast"; the tree of guesses of Kapitsa README): window token i attends to every cached
// position 0..L-1 and to the window positions L+j it may see (j <= i, or bit j of its tree
// mask). Query head hq reads kv head hq / group. q (fp32) is rounded to bf16, K and V are
// bf16, scores and sums are fp32.
//
// Work split (by absolute position, never by M): positions 0..L+M-1 of the cache arrays (the
// cached ones, then the window's own at L..L+M-1) are cut into chunks of 128. One CTA per
// (chunk, kv head) holds the chunk's K and V rows and the Q rows of its head group in shared
// memory; row r = i*group + g is query head kvh*group + g of token i, so a token's row sits
// in the same MMA slot whatever M is. A position a token may not see adds exact zeros to its
// chunk's sums and to the combine, so a token's output depends on its own position and what
// it sees only: verified in a window of M at cache length L, or decoded alone at cache length
// L + i with the earlier window rows cached, it gets the same bits (tested).
// Each warp owns 16 rows: S = Q K^T on mma.sync (bf16 in, fp32 out), the chunk's
// row maximum m and p = exp(s - m), l = sum p, and o = P V on mma.sync with P split into
// bf16 hi + lo parts (P = hi + lo to 2^-16 relative), so o carries fp32 rounding only.
// A second kernel adds the chunks in index order, each weighted by exp(m_c - max m).
#include <cuda_bf16.h>

#include <cmath>

#include "kq.h"
#include "kq_device.cuh"
#include "kq_internal.h"

namespace kq {
namespace {

constexpr int kChunk = 128;
constexpr int kAttnThreads = 256;  // 8 warps x 16 query rows
constexpr int kAttnMaxRows = 128;
// from this many 16-row blocks on, each warp takes whole row blocks (same arithmetic)
constexpr int kRowSplitBlocks = 4;

struct AttnParams {
  const float* q;      // M rows of n_q*hd, q_stride apart
  const uint16_t* k;   // (L+M) x (n_kv*hd) bf16
  const uint16_t* v;
  const uint32_t* mask;  // M words or null (causal)
  float* part;         // [n_kv][nchunks][R][hd + 2]: unnormalised o, m, l
  float* o;            // M x (n_q*hd) fp32, or null
  uint16_t* o16;       // M x (n_q*hd) bf16 (nearest even), or null
  int q_stride;        // elements between q rows
  int M, L, n_q, n_kv, group, R, nchunks;
  float scale;
};

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_addr(p)));
}
__device__ __forceinline__ void ldsm_x2(uint32_t& r0, uint32_t& r1, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(smem_addr(p)));
}
__device__ __forceinline__ void ldsm_x2_t(uint32_t& r0, uint32_t& r1, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(smem_addr(p)));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
         ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
}
__device__ __forceinline__ float bf16_rn_f(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

// 16-byte asynchronous copy global -> shared; src_bytes = 0 writes zeros.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// o = P V for one warp's NP pieces: row block rb, dimension groups dg0 + j*dstride (j < NP),
// each summed over the chunk's 128 positions in order (hi part, then lo part, per 16).
template <int HD, int NP>
__device__ __forceinline__ void pv_pieces(const uint16_t* Ph, const uint16_t* Pl, const uint16_t* Vs, int rb, int dg0,
                                          int dstride, int lane, float* base, int R) {
  constexpr int LD = HD + 8, PLD = kChunk + 8, DW = HD / (kAttnThreads / 32), NDT = DW / 8;
  float acc[NP][NDT][4];
#pragma unroll
  for (int j = 0; j < NP; ++j)
#pragma unroll
    for (int dt = 0; dt < NDT; ++dt) acc[j][dt][0] = acc[j][dt][1] = acc[j][dt][2] = acc[j][dt][3] = 0.f;
#pragma unroll
  for (int kk = 0; kk < kChunk / 16; ++kk) {
    uint32_t ah[4], al[4];
    ldsm_x4(ah, Ph + (16 * rb + (lane & 15)) * PLD + kk * 16 + (lane >> 4) * 8);
    ldsm_x4(al, Pl + (16 * rb + (lane & 15)) * PLD + kk * 16 + (lane >> 4) * 8);
#pragma unroll
    for (int j = 0; j < NP; ++j)
#pragma unroll
      for (int dt = 0; dt < NDT; ++dt) {
        uint32_t b0, b1;
        ldsm_x2_t(b0, b1, Vs + (kk * 16 + (lane & 15)) * LD + (dg0 + j * dstride) * DW + dt * 8);
        mma_bf16_16816(acc[j][dt], ah, b0, b1, acc[j][dt]);
        mma_bf16_16816(acc[j][dt], al, b0, b1, acc[j][dt]);
      }
  }
  const int g = lane >> 2, q4 = lane & 3, ra = 16 * rb + g, rbb = ra + 8;
#pragma unroll
  for (int j = 0; j < NP; ++j)
#pragma unroll
    for (int dt = 0; dt < NDT; ++dt) {
      const int d = (dg0 + j * dstride) * DW + dt * 8 + 2 * q4;
      if (ra < R) *reinterpret_cast<float2*>(base + (long long)ra * (HD + 2) + d) = make_float2(acc[j][dt][0], acc[j][dt][1]);
      if (rbb < R) *reinterpret_cast<float2*>(base + (long long)rbb * (HD + 2) + d) = make_float2(acc[j][dt][2], acc[j][dt][3]);
    }
}

// One CTA per (chunk, kv head); all eight warps take part at any M. Warp w copies chunk rows
// 16w..16w+15 of K and V asynchronously (V lands behind the K work). For each 16-row block of
// query rows, warp w forms S = Q K^T for its 16 positions; the chunk's row maxima meet in
// shared memory, and each warp writes p = exp(s - m) for its positions (bf16 hi / lo parts)
// and its partial row sums. The warps then share o = P V by pieces of 16 rows x HD/8
// dimensions, the row blocks padded to a power of two so that a warp keeps one row block
// (padding rows are never stored; MMA rows are independent). Every sum runs in an order fixed
// by positions (never by M), and which warp takes a piece changes nothing in its arithmetic.
template <int HD>
__global__ void __launch_bounds__(kAttnThreads, 1) attn_chunk_kernel(const AttnParams p) {
  constexpr int LD = HD + 8;       // shared row stride (elements): 16-byte pad, conflict-free ldmatrix
  constexpr int PLD = kChunk + 8;  // the same for P
  constexpr int NW = kAttnThreads / 32;
  static_assert(kChunk == 16 * NW, "16 positions per warp");
  static_assert((HD / NW) % 8 == 0, "whole 8-wide MMA tiles per warp");
  extern __shared__ __align__(16) uint16_t asmem[];
  uint16_t* Qs = asmem;                       // [128][LD]
  uint16_t* Ks = Qs + kAttnMaxRows * LD;      // [kChunk][LD]
  uint16_t* Vs = Ks + kChunk * LD;            // [kChunk][LD]
  uint16_t* Ph = Vs + kChunk * LD;            // [128][PLD]: P rounded to bf16
  uint16_t* Pl = Ph + kAttnMaxRows * PLD;     // [128][PLD]: P - hi, rounded to bf16
  float* red_m = reinterpret_cast<float*>(Pl + kAttnMaxRows * PLD);  // [NW][128]: per-warp row maxima
  float* red_l = red_m + NW * kAttnMaxRows;                          // [NW][128]: per-warp row sums
  // the combine kernel may be launched now; it waits for this grid before reading anything
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // when this grid was itself launched early (programmatic dependent launch), wait for the
  // previous one before the first read or write (a no-op otherwise)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int c = blockIdx.x, kvh = blockIdx.y;
  const int pos0 = c * kChunk;
  const int npos = min(kChunk, p.L + p.M - pos0);
  const int wcol = p.L - pos0;  // column of window position 0: columns before it are cached positions
  const int kvw = p.n_kv * HD, qw = p.q_stride;
  const int rows16 = (p.R + 15) & ~15, nrb = rows16 / 16;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q4 = lane & 3;

  // the Q rows of the head group (fp32), loads first; rows R..rows16-1 as zeros
  constexpr int Q_PER_T = kAttnMaxRows * (HD / 4) / kAttnThreads;  // float4 pieces per thread
  float4 qf[Q_PER_T];
#pragma unroll
  for (int t = 0; t < Q_PER_T; ++t) {
    const int e = threadIdx.x + t * kAttnThreads, r = e / (HD / 4), c4 = e - r * (HD / 4);
    qf[t] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r < p.R) {
      const int i = r / p.group, hq = kvh * p.group + (r - i * p.group);
      qf[t] = __ldg(reinterpret_cast<const float4*>(p.q + (long long)i * qw + hq * HD + c4 * 4));
    }
  }
  // this warp's 16 K rows (group 0) and 16 V rows (group 1); rows past the chunk read zeros
  constexpr int PIECES = 16 * (HD / 8) / 32;  // 16-byte pieces per lane per matrix
#pragma unroll
  for (int t = 0; t < PIECES; ++t) {
    const int e = lane + 32 * t, r = 16 * warp + e / (HD / 8), c8 = e % (HD / 8);
    const bool in = r < npos;
    const long long off = in ? (long long)(pos0 + r) * kvw + kvh * HD + c8 * 8 : 0;
    cp_async16(Ks + r * LD + c8 * 8, p.k + off, in ? 16u : 0u);
  }
  cp_async_commit();
#pragma unroll
  for (int t = 0; t < PIECES; ++t) {
    const int e = lane + 32 * t, r = 16 * warp + e / (HD / 8), c8 = e % (HD / 8);
    const bool in = r < npos;
    const long long off = in ? (long long)(pos0 + r) * kvw + kvh * HD + c8 * 8 : 0;
    cp_async16(Vs + r * LD + c8 * 8, p.v + off, in ? 16u : 0u);
  }
  cp_async_commit();
#pragma unroll
  for (int t = 0; t < Q_PER_T; ++t) {
    const int e = threadIdx.x + t * kAttnThreads, r = e / (HD / 4), c4 = e - r * (HD / 4);
    if (r < rows16)
      *reinterpret_cast<uint2*>(Qs + r * LD + c4 * 4) =
          make_uint2(pack_bf16(qf[t].x, qf[t].y), pack_bf16(qf[t].z, qf[t].w));
  }
  __syncthreads();
  float* base = p.part + ((long long)kvh * p.nchunks + c) * p.R * (HD + 2);

  if (nrb >= kRowSplitBlocks) {
    // Many rows: warp w takes row block w over all 128 positions (S, p and P V in registers),
    // with the same arithmetic as the position split below: the same MMAs, an exact maximum,
    // and each row sum formed per 16 positions (4 values per thread, then the quad butterfly)
    // and added in position-group order.
    cp_async_wait<0>();
    __syncthreads();  // all K and V rows
    if (warp < nrb) {
      const int r0 = 16 * warp;
      float sr[kChunk / 8][4];
#pragma unroll
      for (int nt = 0; nt < kChunk / 8; ++nt) sr[nt][0] = sr[nt][1] = sr[nt][2] = sr[nt][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        uint32_t a[4];
        ldsm_x4(a, Qs + (r0 + (lane & 15)) * LD + kk * 16 + (lane >> 4) * 8);
#pragma unroll
        for (int nt = 0; nt < kChunk / 8; ++nt) {
          uint32_t b0, b1;
          ldsm_x2(b0, b1, Ks + (nt * 8 + (lane & 7)) * LD + kk * 16 + ((lane >> 3) & 1) * 8);
          mma_bf16_16816(sr[nt], a, b0, b1, sr[nt]);
        }
      }
      const int ra = r0 + g, rbb = ra + 8;
      const int ia = ra / p.group, ib = rbb / p.group;
      const uint32_t ma = p.mask ? __ldg(p.mask + min(ia, p.M - 1)) : (ia >= 31 ? 0xFFFFFFFFu : ((2u << ia) - 1u));
      const uint32_t mb = p.mask ? __ldg(p.mask + min(ib, p.M - 1)) : (ib >= 31 ? 0xFFFFFFFFu : ((2u << ib) - 1u));
      float mxa = -INFINITY, mxb = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < kChunk / 8; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int col = nt * 8 + 2 * q4 + e, jw = col - wcol;
          const bool va = ra < p.R && col < npos && (jw < 0 || ((ma >> jw) & 1u));
          const bool vb = rbb < p.R && col < npos && (jw < 0 || ((mb >> jw) & 1u));
          sr[nt][e] = va ? sr[nt][e] * p.scale : -INFINITY;
          sr[nt][2 + e] = vb ? sr[nt][2 + e] * p.scale : -INFINITY;
          mxa = fmaxf(mxa, sr[nt][e]);
          mxb = fmaxf(mxb, sr[nt][2 + e]);
        }
#pragma unroll
      for (int o = 1; o <= 2; o <<= 1) {
        mxa = fmaxf(mxa, __shfl_xor_sync(0xFFFFFFFFu, mxa, o));
        mxb = fmaxf(mxb, __shfl_xor_sync(0xFFFFFFFFu, mxb, o));
      }
      const float ca = mxa == -INFINITY ? 0.f : mxa, cb = mxb == -INFINITY ? 0.f : mxb;
      float la = 0.f, lb = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) {  // position group w: tiles 2w, 2w + 1
        float pa = 0.f, pb = 0.f;
#pragma unroll
        for (int nt = 2 * w; nt < 2 * w + 2; ++nt) {
          sr[nt][0] = __expf(sr[nt][0] - ca);
          sr[nt][1] = __expf(sr[nt][1] - ca);
          sr[nt][2] = __expf(sr[nt][2] - cb);
          sr[nt][3] = __expf(sr[nt][3] - cb);
          pa += sr[nt][0];
          pa += sr[nt][1];
          pb += sr[nt][2];
          pb += sr[nt][3];
        }
#pragma unroll
        for (int o = 1; o <= 2; o <<= 1) {
          pa += __shfl_xor_sync(0xFFFFFFFFu, pa, o);
          pb += __shfl_xor_sync(0xFFFFFFFFu, pb, o);
        }
        if (w == 0) {
          la = pa;
          lb = pb;
        } else {
          la += pa;
          lb += pb;
        }
      }
      // o = P V over all dimensions, P = hi + lo in bf16 straight from the S fragments
      float acc[HD / 8][4];
#pragma unroll
      for (int dt = 0; dt < HD / 8; ++dt) acc[dt][0] = acc[dt][1] = acc[dt][2] = acc[dt][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < kChunk / 16; ++kk) {
        const float* p0 = sr[2 * kk];
        const float* p1 = sr[2 * kk + 1];
        const float h0 = bf16_rn_f(p0[0]), h1 = bf16_rn_f(p0[1]), h2 = bf16_rn_f(p0[2]), h3 = bf16_rn_f(p0[3]);
        const float h4 = bf16_rn_f(p1[0]), h5 = bf16_rn_f(p1[1]), h6 = bf16_rn_f(p1[2]), h7 = bf16_rn_f(p1[3]);
        const uint32_t ah[4] = {pack_bf16(h0, h1), pack_bf16(h2, h3), pack_bf16(h4, h5), pack_bf16(h6, h7)};
        const uint32_t al[4] = {pack_bf16(p0[0] - h0, p0[1] - h1), pack_bf16(p0[2] - h2, p0[3] - h3),
                                pack_bf16(p1[0] - h4, p1[1] - h5), pack_bf16(p1[2] - h6, p1[3] - h7)};
#pragma unroll
        for (int dt = 0; dt < HD / 8; ++dt) {
          uint32_t b0, b1;
          ldsm_x2_t(b0, b1, Vs + (kk * 16 + (lane & 15)) * LD + dt * 8);
          mma_bf16_16816(acc[dt], ah, b0, b1, acc[dt]);
          mma_bf16_16816(acc[dt], al, b0, b1, acc[dt]);
        }
      }
#pragma unroll
      for (int dt = 0; dt < HD / 8; ++dt) {
        const int d = dt * 8 + 2 * q4;
        if (ra < p.R) *reinterpret_cast<float2*>(base + (long long)ra * (HD + 2) + d) = make_float2(acc[dt][0], acc[dt][1]);
        if (rbb < p.R) *reinterpret_cast<float2*>(base + (long long)rbb * (HD + 2) + d) = make_float2(acc[dt][2], acc[dt][3]);
      }
      if (q4 == 0) {
        if (ra < p.R) *reinterpret_cast<float2*>(base + (long long)ra * (HD + 2) + HD) = make_float2(mxa, la);
        if (rbb < p.R) *reinterpret_cast<float2*>(base + (long long)rbb * (HD + 2) + HD) = make_float2(mxb, lb);
      }
    }
    return;
  }

  cp_async_wait<1>();  // this lane's K pieces
  __syncwarp();        // ... and the warp's

  for (int rb = 0; rb < nrb; ++rb) {
    // S = Q K^T for this row block and positions 16w.. (two 8-wide tiles)
    float s[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
      uint32_t a[4];
      ldsm_x4(a, Qs + (16 * rb + (lane & 15)) * LD + kk * 16 + (lane >> 4) * 8);
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        uint32_t b0, b1;
        ldsm_x2(b0, b1, Ks + (16 * warp + nt * 8 + (lane & 7)) * LD + kk * 16 + ((lane >> 3) & 1) * 8);
        mma_bf16_16816(s[nt], a, b0, b1, s[nt]);
      }
    }
    // scale, visibility, this warp's row maxima over its 16 positions
    const int ra = 16 * rb + g, rbb = ra + 8;
    const int ia = ra / p.group, ib = rbb / p.group;
    // window positions each row's token may see: bit j for window position j
    const uint32_t ma = p.mask ? __ldg(p.mask + min(ia, p.M - 1)) : (ia >= 31 ? 0xFFFFFFFFu : ((2u << ia) - 1u));
    const uint32_t mb = p.mask ? __ldg(p.mask + min(ib, p.M - 1)) : (ib >= 31 ? 0xFFFFFFFFu : ((2u << ib) - 1u));
    float mxa = -INFINITY, mxb = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int col = 16 * warp + nt * 8 + 2 * q4 + e, jw = col - wcol;  // jw: window position, if >= 0
        const bool va = ra < p.R && col < npos && (jw < 0 || ((ma >> jw) & 1u));
        const bool vb = rbb < p.R && col < npos && (jw < 0 || ((mb >> jw) & 1u));
        s[nt][e] = va ? s[nt][e] * p.scale : -INFINITY;
        s[nt][2 + e] = vb ? s[nt][2 + e] * p.scale : -INFINITY;
        mxa = fmaxf(mxa, s[nt][e]);
        mxb = fmaxf(mxb, s[nt][2 + e]);
      }
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      mxa = fmaxf(mxa, __shfl_xor_sync(0xFFFFFFFFu, mxa, o));
      mxb = fmaxf(mxb, __shfl_xor_sync(0xFFFFFFFFu, mxb, o));
    }
    if (q4 == 0) {
      red_m[warp * kAttnMaxRows + ra] = mxa;
      red_m[warp * kAttnMaxRows + rbb] = mxb;
    }
    __syncthreads();
    // p = exp(s - m), m the chunk's row maximum (a maximum: exact in any order)
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      mxa = fmaxf(mxa, red_m[w * kAttnMaxRows + ra]);
      mxb = fmaxf(mxb, red_m[w * kAttnMaxRows + rbb]);
    }
    const float ca = mxa == -INFINITY ? 0.f : mxa, cb = mxb == -INFINITY ? 0.f : mxb;
    float la = 0.f, lb = 0.f;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      // the fast exponential (relative error ~2^-21, far inside the contract's 1e-4; the same
      // instruction for every M); exp(-inf) = 0 for positions not seen
      const float p0 = __expf(s[nt][0] - ca), p1 = __expf(s[nt][1] - ca);
      const float p2 = __expf(s[nt][2] - cb), p3 = __expf(s[nt][3] - cb);
      la += p0;
      la += p1;
      lb += p2;
      lb += p3;
      const int col = 16 * warp + nt * 8 + 2 * q4;
      const float h0 = bf16_rn_f(p0), h1 = bf16_rn_f(p1), h2 = bf16_rn_f(p2), h3 = bf16_rn_f(p3);
      *reinterpret_cast<uint32_t*>(Ph + ra * PLD + col) = pack_bf16(h0, h1);
      *reinterpret_cast<uint32_t*>(Ph + rbb * PLD + col) = pack_bf16(h2, h3);
      *reinterpret_cast<uint32_t*>(Pl + ra * PLD + col) = pack_bf16(p0 - h0, p1 - h1);
      *reinterpret_cast<uint32_t*>(Pl + rbb * PLD + col) = pack_bf16(p2 - h2, p3 - h3);
    }
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      la += __shfl_xor_sync(0xFFFFFFFFu, la, o);
      lb += __shfl_xor_sync(0xFFFFFFFFu, lb, o);
    }
    if (q4 == 0) {
      red_l[warp * kAttnMaxRows + ra] = la;
      red_l[warp * kAttnMaxRows + rbb] = lb;
    }
  }
  cp_async_wait<0>();  // this lane's V pieces
  __syncthreads();     // every warp's V rows, P and row sums

  // o = P V: row blocks padded to nrbp (a power of two); warp w takes row block w % nrbp and
  // dimension groups w / nrbp + (NW / nrbp) j, j < nrbp
  const int nrbp = nrb <= 1 ? 1 : nrb <= 2 ? 2 : nrb <= 4 ? 4 : 8;
  const int prb = warp % nrbp, dg0 = warp / nrbp, dstride = NW / nrbp;
  if (nrbp == 1) pv_pieces<HD, 1>(Ph, Pl, Vs, prb, dg0, dstride, lane, base, p.R);
  else if (nrbp == 2) pv_pieces<HD, 2>(Ph, Pl, Vs, prb, dg0, dstride, lane, base, p.R);
  else if (nrbp == 4) pv_pieces<HD, 4>(Ph, Pl, Vs, prb, dg0, dstride, lane, base, p.R);
  else pv_pieces<HD, 8>(Ph, Pl, Vs, prb, dg0, dstride, lane, base, p.R);

  // ... the chunk's row maximum and sum (the warps' sums added in warp order)
  for (int r = threadIdx.x; r < p.R; r += kAttnThreads) {
    float m = red_m[r], l = red_l[r];
#pragma unroll
    for (int w = 1; w < NW; ++w) {
      m = fmaxf(m, red_m[w * kAttnMaxRows + r]);
      l += red_l[w * kAttnMaxRows + r];
    }
    *reinterpret_cast<float2*>(base + (long long)r * (HD + 2) + HD) = make_float2(m, l);
  }
}

// out[i][hq][d] = sum_c e_c o_c[d] / sum_c e_c l_c, e_c = exp(m_c - max_c m_c); zeros when
// the token sees no position. One CTA per (row, kv head) of kCombGroups x HD threads: group
// g adds the chunks c = g (mod kCombGroups) in index order (the first kPre chunks' loads leave
// with the loads of the chunks' maxima, later ones go eight at a time), then the groups' sums
// are added in group order. The chunks' (m, l) pass through
// shared memory. Chunks are added in index order, and their number, ceil((L + M) / 128),
// depends on L + M; a chunk holding no position the token may see has m = -inf, so its
// weight e_c is exactly 0 and its o_c and l_c are exact zeros: it adds nothing. That is
// what keeps a window token's bits equal to those of the same token decoded alone (whose
// sum has fewer chunks), given finite cached keys and values (a masked position still
// enters the P V product with P = 0, and 0 * Inf is NaN).
constexpr int kMaxChunks = 1024;
constexpr int kCombGroups = 4;
constexpr int kPre = 12;  // chunks per group whose partials load before the maxima are known
template <int HD>
__global__ void __launch_bounds__(HD * kCombGroups) attn_combine_kernel(const AttnParams p) {
  constexpr int PW = HD + 2, NT = HD * kCombGroups;
  __shared__ float sm_m[kMaxChunks], sm_l[kMaxChunks], sm_red[NT / 32];
  __shared__ float sm_num[kCombGroups][HD], sm_den[kCombGroups];
  const int r = blockIdx.x, kvh = blockIdx.y, t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int grp = t / HD, d = t - grp * HD;
  // launched while the chunk kernel runs (programmatic dependent launch): its partials are
  // complete and visible once this returns
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const float* base = p.part + (long long)kvh * p.nchunks * p.R * PW + (long long)r * PW;
  const long long cs = (long long)p.R * PW;
  // the partials of this thread's first kPre chunks: their loads do not depend on the
  // maxima, so they leave with the (m, l) loads instead of one round trip later (every chunk
  // of a context up to kPre * kCombGroups * 128 positions)
  float ov0[kPre];
#pragma unroll
  for (int j = 0; j < kPre; ++j) {
    const int cc = grp + j * kCombGroups;
    ov0[j] = cc < p.nchunks ? base[cc * cs + d] : 0.f;
  }
  float mloc = -INFINITY;
  for (int c = t; c < p.nchunks; c += NT) {
    const float2 ml = *reinterpret_cast<const float2*>(base + c * cs + HD);
    sm_m[c] = ml.x;
    sm_l[c] = ml.y;
    mloc = fmaxf(mloc, ml.x);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mloc = fmaxf(mloc, __shfl_xor_sync(0xFFFFFFFFu, mloc, o));
  if (lane == 0) sm_red[warp] = mloc;
  __syncthreads();
  float mt = sm_red[0];
#pragma unroll
  for (int w = 1; w < NT / 32; ++w) mt = fmaxf(mt, sm_red[w]);  // a maximum: exact in any order
  for (int c = t; c < p.nchunks; c += NT) sm_m[c] = (mt == -INFINITY || sm_m[c] == -INFINITY) ? 0.f : expf(sm_m[c] - mt);
  __syncthreads();
  // chunks grp, grp + 4, ... in index order, one FMA each (the first kPre from ov0)
  float num = 0.f, den = 0.f;
#pragma unroll
  for (int j = 0; j < kPre; ++j) {
    const int cc = grp + j * kCombGroups;
    if (cc < p.nchunks) {
      num = __fmaf_rn(sm_m[cc], ov0[j], num);
      den = __fmaf_rn(sm_m[cc], sm_l[cc], den);
    }
  }
  int c = grp + kPre * kCombGroups;
  for (; c + 7 * kCombGroups < p.nchunks; c += 8 * kCombGroups) {
    float ov[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) ov[j] = base[(c + j * kCombGroups) * cs + d];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      num = __fmaf_rn(sm_m[c + j * kCombGroups], ov[j], num);
      den = __fmaf_rn(sm_m[c + j * kCombGroups], sm_l[c + j * kCombGroups], den);
    }
  }
  for (; c < p.nchunks; c += kCombGroups) {
    num = __fmaf_rn(sm_m[c], base[c * cs + d], num);
    den = __fmaf_rn(sm_m[c], sm_l[c], den);
  }
  sm_num[grp][d] = num;
  if (d == 0) sm_den[grp] = den;
  __syncthreads();
  if (grp == 0) {
    float n = sm_num[0][d], dd = sm_den[0];
#pragma unroll
    for (int g = 1; g < kCombGroups; ++g) {
      n += sm_num[g][d];
      dd += sm_den[g];
    }
    const int i = r / p.group, hq = kvh * p.group + (r - i * p.group);
    const float res = dd > 0.f ? n / dd : 0.f;
    const long long oi = (long long)i * p.n_q * HD + hq * HD + d;
    if (p.o) p.o[oi] = res;
    if (p.o16) p.o16[oi] = __bfloat16_as_ushort(__float2bfloat16_rn(res));
  }
}

int attn_chunks(int L, int M) { return (L + M + kChunk - 1) / kChunk; }

template <int HD>
int launch_attn(const AttnParams& prm, cudaStream_t s, bool early, std::string* err) {
  constexpr int LD = HD + 8, PLD = kChunk + 8;
  const size_t smem = (size_t)(kAttnMaxRows + 2 * kChunk) * LD * 2 + (size_t)2 * kAttnMaxRows * PLD * 2 +
                      (size_t)2 * (kAttnThreads / 32) * kAttnMaxRows * 4;
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(attn_chunk_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) {
      *err = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e);
      return -1;
    }
    attr_done[dev] = true;
  }
  // early: the chunk kernel may start (shared-memory carve-up, its launch) while the previous
  // kernel in the stream finishes; it waits for it before touching memory
  cudaError_t e;
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(prm.nchunks, prm.n_kv, 1);
    cfg.blockDim = dim3(kAttnThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = early ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, attn_chunk_kernel<HD>, prm);
  }
  if (e == cudaSuccess) {  // the combine starts while the chunks run and waits for them
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(prm.R, prm.n_kv, 1);
    cfg.blockDim = dim3(HD * kCombGroups, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, attn_combine_kernel<HD>, prm);
  }
  if (e != cudaSuccess) {
    *err = std::string("attention launch: ") + cudaGetErrorString(e);
    return -1;
  }
  return 0;
}

}  // namespace

size_t attention_workspace(int M, int L, int n_q, int n_kv, int hd) {
  const int R = (n_q / n_kv) * M;
  return (size_t)n_kv * attn_chunks(L, M) * R * (hd + 2) * sizeof(float);
}

int launch_attention(const float* q, int q_stride, const uint16_t* k, const uint16_t* v, float* o, uint16_t* o16,
                     int M, int L, int n_q, int n_kv, int hd, const uint32_t* mask, float scale, void* ws,
                     cudaStream_t s, bool early, std::string* err) {
  AttnParams prm;
  prm.q = q;
  prm.q_stride = q_stride;
  prm.o16 = o16;
  prm.k = k;
  prm.v = v;
  prm.mask = mask;
  prm.part = static_cast<float*>(ws);
  prm.o = o;
  prm.M = M;
  prm.L = L;
  prm.n_q = n_q;
  prm.n_kv = n_kv;
  prm.group = n_q / n_kv;
  prm.R = prm.group * M;
  prm.nchunks = attn_chunks(L, M);
  prm.scale = scale;
  if (hd == 128) return launch_attn<128>(prm, s, early, err);
  if (hd == 64) return launch_attn<64>(prm, s, early, err);
  *err = "head_dim must be 64 or 128";
  return -1;
}

}  // namespace kq
