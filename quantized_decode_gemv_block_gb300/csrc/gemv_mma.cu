// Tensor-core GEMV / speculative-verify kernels for bf16 activations, M = 1..16.
//
// Computes Y[j][n] = sum_k deq(W)[n][k] * X[j][k] for block-quantized W (Kinetic
// README, "What makes it fast": a decode step reads every weight once per token, a
// speculative check runs all guesses through one pass over the weights).
//
// Two kernels, chosen by (format, N, K) only:
//  * gemv_tma_kernel (the streaming kernel, section below): one CTA per SM; each warp
//    streams its share of 16-row tiles through a private ring of shared-memory stages
//    filled by tensor copies; the activations of the CTA's K-slice are staged once (the
//    K-quant and Q8_0 formats as fp16 under an exact per-(token, super-block) power of two);
//    mma.sync m16n8k16 multiplies 16 weight rows by 8 token columns (tokens 8..15 take a
//    second column tile); K is split across a thread-block cluster when N alone gives too
//    few tiles, the ranks' partials meeting in distributed shared memory in rank order.
//  * gemv_chunked_kernel (K too long for the streaming kernel's staging): 128 rows per CTA,
//    register-streamed 8- and 16-byte loads two units ahead, activations staged in chunks,
//    K split over a cluster; per 32-group the fp32 MMA result is promoted by its scale and
//    the min/bias term added against the staged sums of x.
//
// Batch invariance (Kinetic README, "What makes it fast", last paragraph: every row
// of a batch is summed in the same order as that token alone): a token column's
// arithmetic is the same instruction sequence for every M. M only predicates the
// activation loads (absent tokens read as zero) and the stores, and the column
// tile count (1 or 2) leaves tile 0 unchanged.
#include <cooperative_groups.h>
#include <cuda.h>

#include <algorithm>
#include <cstring>

#include "kq_device.cuh"
#include "kq_internal.h"
#include "gemv_formats.cuh"

namespace cg = cooperative_groups;

namespace kq {
namespace {
using namespace gemv;

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRowsPerCta = 16 * kWarps;
constexpr int kUnit = 256;       // weights per K-unit (one Q4_K super-block, 8 Q8_0 / affine4 blocks)
constexpr int kChunkUnits = 8;   // K-units of activations staged in shared memory at a time
constexpr int kDepth = 2;        // K-units each warp keeps in flight

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

// Stage X[0:M][uc*256 : (uc+nun)*256] into shared memory (B-fragment order) and, when the
// format has a min or bias term, the fp32 sum of each 32-group of every token.
template <class F, int T>
__device__ void stage_x(const uint16_t* xg, int M, int K, int xstride, uint16_t* xs, float* ss,
                        int uc, int nun) {
  const int per_tok = nun * 32;  // 16-byte vectors per token
  for (int idx = threadIdx.x; idx < M * per_tok; idx += kThreads) {
    const int tok = idx / per_tok, v = idx - tok * per_tok;
    uint4 val = ldg128(xg + (long long)tok * K + (long long)uc * kUnit + v * 8);
    if (F::kPerm0213) {  // (e0 e1 e2 e3) -> (e0 e2 e1 e3) within each group of four
      const uint4 o = val;
      val.x = prmt(o.x, o.y, 0x5410u);
      val.y = prmt(o.x, o.y, 0x7632u);
      val.z = prmt(o.z, o.w, 0x5410u);
      val.w = prmt(o.z, o.w, 0x7632u);
    }
    *reinterpret_cast<uint4*>(xs + tok * xstride + v * 8) = val;
  }
  if (F::kNeedsSum) {
    for (int idx = threadIdx.x; idx < T * nun * 8; idx += kThreads) {
      const int grp = idx / T, tok = idx - grp * T;
      float s = 0.f;
      if (tok < M) {
        const uint16_t* src = xg + (long long)tok * K + (long long)uc * kUnit + grp * 32;
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
__global__ void __launch_bounds__(kThreads, 2) gemv_chunked_kernel(const Params p) {
  using F = typename FmtOf<FMT>::type;
  constexpr int T = 8 * NT;
  extern __shared__ __align__(128) uint8_t smem[];
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
      F::template load<LdGlobal>(raw[i], wa + (long long)(u0 + i) * F::kUnitBytes,
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
          stage_x<F, T>(p.x, p.M, p.K, p.xstride, xs, ss, uu, min(p.chunk_units, u1 - uu));
          __syncthreads();
        }
        const int ul = uu - chunk0;
        F::template compute<NT>(raw[i], acc, xs + ul * kUnit, p.xstride, ss + ul * 8 * T, lane,
                                p.M);
        if (uu + kDepth < u1)
          F::template load<LdGlobal>(raw[i], wa + (long long)(uu + kDepth) * F::kUnitBytes,
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
int launch_chunked(const Params& prm, size_t smem, cudaStream_t stream, std::string* err) {
  auto kern = gemv_chunked_kernel<FMT, NT>;
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


// ============================================================================
// Streaming kernel: one CTA per SM, weights brought in by 2-D tensor copies (TMA).
//
// The N rows are cut into 16-row tiles and K into 256-weight units. A cluster of C
// CTAs owns a contiguous range of tiles; CTA rank r owns K-slice r of those tiles.
// The CTA's (tile, unit) work list, tile-major, is cut into 8 contiguous pieces, one
// per warp, so every warp streams the same number of units. Each warp keeps a
// private ring of `depth` stages in shared memory; one stage holds up to `su`
// consecutive units of one tile for its 16 rows and is filled by ONE tensor copy (a
// 16-row box, rows past N arriving as zeros) completing on the stage's mbarrier. Q6_K rows
// are only 2-byte aligned, which no tensor map takes: there each row of a stage is its own
// 1-D bulk copy of the 16-byte-aligned span around its units (rows past N copy nothing and
// are never stored). The whole ring is requested before the activations are staged.
//
// A tile whose units one warp covers entirely is finished by that warp. A tile cut
// between warps leaves one partial per warp, added at the end in warp order (= K
// order). With C > 1 the CTAs' tile results meet in distributed shared memory and
// are added in rank order (= K order). Every cut depends on (N, K, SM count) only.
// ============================================================================
constexpr int kMaxSliceUnits = 10;     // K-units of activations a CTA stages
constexpr int kAuxScaleBytes = kMaxSliceUnits * 16 * 4;  // 2^-e per (staged unit, token)
constexpr int kMaxClusterTiles = 32;   // tiles per cluster when partials meet across CTAs
constexpr int kMaxClusterSize = 8;     // K-split ranks per cluster (the plan tries 1, 2, 4, 8)
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // bounded waits give up after 2 s

__device__ unsigned int g_device_errors = 0;  // bit 0: a bounded wait gave up

struct TmaParams {
  const uint16_t* x;
  float* y;
  int M, N, K;
  int units, tiles, C, G;
  int su, depth, row_stride, unit_bytes, xstride, max_tiles;
  int off_ss, off_ring, off_bar, off_pb, off_res, off_aux;
  int xts, s2ts;  // fp16 path: row strides (bytes) of the staged x and min-term operands
  // epilogue (GemvEpilogue): 0 y only; 1 y plus the bf16 GQA copies of rows [e_v0, e_v0 + e_vn);
  // 2 paired rows (tile t = gate rows 8t.. and up rows half + 8t..), out2 = bf16(silu(g) * u);
  // 3 y plus bf16 rows [e_v0, e_v0 + e_hd) into out2 and [e_v0 + e_hd, e_v0 + 2 e_hd) into
  // out3, row e_row0 + token of each (e_hd wide): a KV cache append
  int epi, e_v0, e_vn, e_hd, e_group, e_w, half, e_row0;
  uint16_t* out2;
  uint16_t* out3;
  // formats with per-row copies (F::kRowCopies): the weight rows, row_bytes apart
  const uint8_t* w;
  long long row_bytes;
};

template <class F, int NT>
__global__ void __launch_bounds__(kThreads, 1)
    gemv_tma_kernel(const __grid_constant__ CUtensorMap tmap, const TmaParams p) {
  constexpr int T = 8 * NT;
  extern __shared__ __align__(128) uint8_t smem[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);
  float* ss = reinterpret_cast<float*>(smem + p.off_ss);
  uint8_t* ring = smem + p.off_ring;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bar);
  float* pbuf = reinterpret_cast<float*>(smem + p.off_pb);  // [warp][2][16][T]
  float* res = reinterpret_cast<float*>(smem + p.off_res);  // [tile][16][T], C > 1
  float* ivs = reinterpret_cast<float*>(smem + p.off_aux);  // [super-block][16]: 2^-e (fp16 path)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  if constexpr (!F::kRowCopies) {
    if (threadIdx.x == 0) asm volatile("prefetch.tensormap [%0];" ::"l"(&tmap) : "memory");
  }
  int rank = 0;
  if (p.C > 1) rank = static_cast<int>(cg::this_cluster().block_rank());
  // all index math in 32-bit unsigned (every product below stays under 2^31)
  const unsigned cid = blockIdx.x / static_cast<unsigned>(p.C);
  const unsigned ug = static_cast<unsigned>(p.G), uc = static_cast<unsigned>(p.C);
  const int t0 = static_cast<int>(cid * static_cast<unsigned>(p.tiles) / ug);
  const int t1 = static_cast<int>((cid + 1u) * static_cast<unsigned>(p.tiles) / ug);
  const int k0 = static_cast<int>(static_cast<unsigned>(rank) * static_cast<unsigned>(p.units) / uc);
  const int k1 = static_cast<int>(static_cast<unsigned>(rank + 1) * static_cast<unsigned>(p.units) / uc);
  const int S = k1 - k0;
  const int nt = t1 - t0;
  const int ltot = nt * S;
  const int l0 = warp * ltot / kWarps, l1 = (warp + 1) * ltot / kWarps;

  // Barriers first: their release fence would otherwise wait for the activation loads.
  uint8_t* myring = ring + (size_t)warp * p.depth * 16 * p.row_stride;
  uint64_t* mybar = bars + warp * p.depth;
  if (lane == 0) {
    for (int s = 0; s < p.depth; ++s) mbar_init(&mybar[s], 1);
    fence_mbar_init();
  }
  __syncwarp();
  // Programmatic dependent launch: a following launch may begin now (it still waits for
  // this grid to finish before it reads anything this grid writes).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // Producer (lane 0): stage sequence over [l0, l1), never crossing a tile boundary.
  const int fdiv = S > 0 ? S : 1;
  int lp = l0, ptl = l0 / fdiv, pul = l0 - ptl * S;
  const uint32_t stage_bytes = 16u * static_cast<uint32_t>(p.row_stride);
  const int ucol = p.unit_bytes / 4;  // tensor map elements are 4-byte words
  auto issue = [&](int slot) {
    const int nu = min(p.su, min(l1 - lp, S - pul));
    if constexpr (F::kRowCopies) {
      // one bulk copy per row (lanes 0..15): the 16-byte-aligned span covering the row's nu
      // units; rows past N copy nothing (the buffer's end is 16-byte aligned: host check)
      const int row = (t0 + ptl) * 16 + lane;
      uint32_t bytes = 0;
      long long a0 = 0;
      if (lane < 16 && row < p.N) {
        const long long a = (long long)row * p.row_bytes + (long long)(k0 + pul) * F::kUnitBytes;
        a0 = a & ~15ll;
        bytes = static_cast<uint32_t>(((a + (long long)nu * F::kUnitBytes + 15) & ~15ll) - a0);
      }
      const uint32_t total = __reduce_add_sync(0xFFFFFFFFu, bytes);
      if (lane == 0) mbar_arrive_expect_tx(&mybar[slot], total);
      __syncwarp();
      if (bytes) bulk_g2s(myring + ((size_t)slot * 16 + lane) * p.row_stride, p.w + a0, bytes, &mybar[slot]);
    } else if (lane == 0) {
      mbar_arrive_expect_tx(&mybar[slot], stage_bytes);
      uint8_t* dst = myring + (size_t)slot * 16 * p.row_stride;
      if (p.epi == 2) {  // 8-row boxes: the tile's gate rows, then the matching up rows
        tma_load_2d(dst, &tmap, (k0 + pul) * ucol, (t0 + ptl) * 8, &mybar[slot]);
        tma_load_2d(dst + (size_t)8 * p.row_stride, &tmap, (k0 + pul) * ucol, p.half + (t0 + ptl) * 8, &mybar[slot]);
      } else {
        tma_load_2d(dst, &tmap, (k0 + pul) * ucol, (t0 + ptl) * 16, &mybar[slot]);
      }
    }
    lp += nu;
    pul += nu;
    if (pul == S) { pul = 0; ++ptl; }
  };
  for (int s = 0; s < p.depth && lp < l1; ++s) issue(s);

  // The weights may stream before the previous grid in the stream has finished (when this
  // launch was allowed to overlap it); the activations it produced may not: wait here.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  [[maybe_unused]] StageQ4KH<kThreads, F> stq;
  if constexpr (F::kHalfX) {
    if (S > 0) stq.load(p.x, p.M, p.K, k0, S, smem, p.xts, smem + p.off_ss, p.s2ts, ivs);
  }

  // This warp's first and last tile, and whether each is partial (kept for the combine).
  int* meta = reinterpret_cast<int*>(smem + p.off_aux + kAuxScaleBytes);  // [warp][4]
  const int w_first = l0 / fdiv, w_last = l1 > l0 ? (l1 - 1) / fdiv : -1;
  if (lane == 0) {
    meta[warp * 4 + 0] = l1 > l0 ? w_first : -1;
    meta[warp * 4 + 1] = w_last;
    meta[warp * 4 + 2] = (l1 > l0) && !(w_first * S >= l0 && (w_first + 1) * S <= l1);  // first partial
    meta[warp * 4 + 3] = (l1 > l0) && !(w_last * S >= l0 && (w_last + 1) * S <= l1);    // last partial
  }

  int xo[NT], so[NT], io[NT];  // this thread's token rows in the staged activations (fp16 path)
  if constexpr (F::kHalfX) {
    if (S > 0) stq.finish(p.M, S, smem, p.xts, smem + p.off_ss, p.s2ts, ivs);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int tok = 8 * t + g, row = tok < p.M ? tok : p.M;
      xo[t] = row * p.xts + F::kXq * q;
      so[t] = row * p.s2ts + 8 * q;
      io[t] = 8 * t + 2 * q;
    }
  } else {
    if (S > 0) stage_x<F, T>(p.x, p.M, p.K, p.xstride, xs, ss, k0, S);
  }
  __syncthreads();

  float acc[NT][4];
#pragma unroll
  for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;

  // Final value v of output row n (< N) for token tok: y, and in epilogue 1 the bf16 copies of
  // the GQA rows (row v0 + h*hd + d goes to columns (h*group + i)*hd + d, i < group).
  auto put = [&](int n, int tok, float v) {
    if (n >= p.N) return;
    p.y[(long long)tok * p.N + n] = v;
    if (p.epi == 1 && n >= p.e_v0 && n < p.e_v0 + p.e_vn) {
      const int h = (n - p.e_v0) / p.e_hd, d = (n - p.e_v0) - h * p.e_hd;
      const uint16_t b = f32_to_bf16_rn(v);
      uint16_t* o = p.out2 + (long long)tok * p.e_w + (long long)h * p.e_group * p.e_hd + d;
      for (int i = 0; i < p.e_group; ++i) o[i * p.e_hd] = b;
    } else if (p.epi == 3 && n >= p.e_v0 && n < p.e_v0 + 2 * p.e_hd) {
      const int c = n - p.e_v0;
      const long long r = (long long)(p.e_row0 + tok) * p.e_hd;
      if (c < p.e_hd) p.out2[r + c] = f32_to_bf16_rn(v);
      else p.out3[r + c - p.e_hd] = f32_to_bf16_rn(v);
    }
  };
  // Epilogue 2: gate row i and up row half + i (paired in one tile) for token tok.
  auto put2 = [&](int i, int tok, float vg, float vu) {
    if (p.y) {
      p.y[(long long)tok * p.N + i] = vg;
      p.y[(long long)tok * p.N + p.half + i] = vu;
    }
    p.out2[(long long)tok * p.half + i] = silu_mul_bf16(vg, vu);
  };

  // a finished CTA partial of local tile tl
  auto emit = [&](int tl, float (&a)[NT][4]) {
    if (p.C == 1) {
      const int na = (t0 + tl) * 16 + g, nb = na + 8;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const int j0 = 8 * t + 2 * q;
        if (p.epi == 2) {
          const int i = (t0 + tl) * 8 + g;
          if (j0 < p.M) put2(i, j0, a[t][0], a[t][2]);
          if (j0 + 1 < p.M) put2(i, j0 + 1, a[t][1], a[t][3]);
          continue;
        }
        if (j0 < p.M) {
          put(na, j0, a[t][0]);
          put(nb, j0, a[t][2]);
        }
        if (j0 + 1 < p.M) {
          put(na, j0 + 1, a[t][1]);
          put(nb, j0 + 1, a[t][3]);
        }
      }
    } else {
      float* r = res + (size_t)tl * 16 * T;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const int j0 = 8 * t + 2 * q;
        r[g * T + j0] = a[t][0];
        r[g * T + j0 + 1] = a[t][1];
        r[(g + 8) * T + j0] = a[t][2];
        r[(g + 8) * T + j0 + 1] = a[t][3];
      }
    }
  };

  bool ok = true;
  int lc = l0, stage = 0, ctl = w_first, cul = l0 - w_first * S;
  int slot = 0;            // stage % depth and the parity of stage / depth, kept as counters
  uint32_t parity = 0u;
  const size_t stage_stride = (size_t)16 * p.row_stride;
  const uint8_t* ring_g = myring + (size_t)g * p.row_stride;
  while (lc < l1) {
    const int tl = ctl, ul = cul;
    const int nu = min(p.su, min(l1 - lc, S - ul));
    if (ok && !mbar_wait_bounded(&mybar[slot], parity, kWaitLimitNs)) {
      ok = false;
      if (lane == 0) atomicOr(&g_device_errors, 1u);
    }
    ok = __all_sync(0xFFFFFFFFu, ok);  // the warp's MMAs and copies need every lane
    if (ok) {
      const uint8_t* sa = ring_g + (size_t)slot * stage_stride;
      const uint8_t* sb = sa + (size_t)8 * p.row_stride;
      if constexpr (F::kRowCopies) {  // where each row's copy put the stage's first unit
        const uint32_t u0 = static_cast<uint32_t>(k0 + ul) * F::kUnitBytes;
        const uint32_t na = static_cast<uint32_t>((t0 + tl) * 16 + g), rb = static_cast<uint32_t>(p.row_bytes);
        sa += (na * rb + u0) & 15u;  // modulo 2^32 keeps the residue modulo 16
        sb += ((na + 8u) * rb + u0) & 15u;
      }
      for (int i = 0; i < nu; ++i) {
        typename F::Raw raw;
        F::template load<LdShared>(raw, sa + i * p.unit_bytes, sb + i * p.unit_bytes, q);
        if constexpr (F::kHalfX)
          F::template compute<NT>(raw, acc, smem + (ul + i) * 512, xo, smem + p.off_ss + (ul + i) * 32,
                                  so, ivs + (ul + i) * 16, io, lane);
        else
          F::template compute<NT>(raw, acc, xs + (ul + i) * kUnit, p.xstride, ss + (ul + i) * 8 * T,
                                  lane, p.M);
      }
    }
    __syncwarp();
    lc += nu;
    cul += nu;
    ++stage;
    if (lc == l1 || cul == S) {  // leaving tile tl
      const bool whole = tl * S >= l0 && (tl + 1) * S <= l1;
      if (whole) {
        emit(tl, acc);
      } else {
        float* pb = pbuf + ((size_t)(warp * 2 + (tl == w_first ? 0 : 1)) * 16) * T;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const int j0 = 8 * t + 2 * q;
          pb[g * T + j0] = acc[t][0];
          pb[g * T + j0 + 1] = acc[t][1];
          pb[(g + 8) * T + j0] = acc[t][2];
          pb[(g + 8) * T + j0 + 1] = acc[t][3];
        }
      }
#pragma unroll
      for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
    }
    if (cul == S) { cul = 0; ++ctl; }
    if (ok && lp < l1) {
      fence_proxy_async_smem();
      issue(slot);
    }
    if (++slot == p.depth) {
      slot = 0;
      parity ^= 1u;
    }
  }
  if (!ok) {  // let this warp's copies in flight land before the CTA can exit
    for (int s2 = stage; s2 < stage + p.depth; ++s2)
      mbar_wait_bounded(&mybar[s2 % p.depth], static_cast<uint32_t>(s2 / p.depth) & 1u, kWaitLimitNs);
  }
  __syncthreads();

  // Tiles cut between warps. A cut tile's last unit lies in exactly one warp's range, and
  // for that warp the tile is its first tile and a partial one: that warp adds the
  // partials of every warp touching the tile, in warp order (empty warps skipped).
  if (l1 > l0 && meta[warp * 4 + 2] && (w_first + 1) * S <= l1) {
    const int t = w_first;
    int wa = warp;
    for (int ww = warp - 1; ww >= 0; --ww) {
      if (meta[ww * 4 + 0] < 0) continue;  // empty range
      if (meta[ww * 4 + 1] != t) break;
      wa = ww;
    }
    auto cut_sum = [&](int row, int tok) {
      float v = 0.f;
      for (int ww = wa; ww <= warp; ++ww) {
        if (meta[ww * 4 + 0] < 0) continue;
        const int slot = meta[ww * 4 + 0] == t ? 0 : 1;
        v += pbuf[((size_t)(ww * 2 + slot) * 16 + row) * T + tok];
      }
      return v;
    };
    if (p.epi == 2) {  // C == 1 here: rows r and r + 8 are a gate / up pair
      for (int e = lane; e < 8 * p.M; e += 32) {
        const int row = e / p.M, tok = e - row * p.M;
        put2((t0 + t) * 8 + row, tok, cut_sum(row, tok), cut_sum(row + 8, tok));
      }
    } else {
      for (int e = lane; e < 16 * p.M; e += 32) {
        const int row = e / p.M, tok = e - row * p.M;
        const float v = cut_sum(row, tok);
        if (p.C == 1)
          put((t0 + t) * 16 + row, tok, v);
        else
          res[((size_t)t * 16 + row) * T + tok] = v;
      }
    }
  }
  if (p.C == 1) return;

  // K-split across the cluster: add the ranks' tile results in rank order. Every rank's
  // value is loaded before the first addition, so the C remote reads are in flight together.
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();  // a cluster barrier: it also orders this CTA's own threads
  const float* rsrc[kMaxClusterSize];
#pragma unroll
  for (int r = 0; r < kMaxClusterSize; ++r) rsrc[r] = r < p.C ? cluster.map_shared_rank(res, r) : res;
  const int total = nt * 16 * p.M;
  const int e0 = (int)((long long)rank * total / p.C), e1 = (int)((long long)(rank + 1) * total / p.C);
  for (int e = e0 + threadIdx.x; e < e1; e += kThreads) {
    const int tok = e % p.M, rt = e / p.M;  // rt = tile * 16 + row
    const size_t off = (size_t)rt * T + tok;
    float part[kMaxClusterSize];
#pragma unroll
    for (int r = 0; r < kMaxClusterSize; ++r) part[r] = r < p.C ? rsrc[r][off] : 0.f;
    float v = 0.f;
#pragma unroll
    for (int r = 0; r < kMaxClusterSize; ++r)
      if (r < p.C) v += part[r];
    put(t0 * 16 + rt, tok, v);
  }
  cluster.sync();
}

template <class F, int NT>
int launch_tma(const CUtensorMap& tm, const TmaParams& prm, size_t smem, int grid, cudaStream_t stream,
               bool overlap, std::string* err) {
  auto kern = gemv_tma_kernel<F, NT>;
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemCap);
    if (e != cudaSuccess) {
      *err = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e);
      return -1;
    }
    attr_done[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (prm.C > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = prm.C;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (overlap) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tm, prm);
  if (e != cudaSuccess) {
    *err = std::string("gemv (stream) launch: ") + cudaGetErrorString(e);
    return -1;
  }
  return 0;
}

int unit_bytes_of(int fmt) {
  return fmt == FMT_Q4_K ? 144 : (fmt == FMT_Q5_K ? 176 : (fmt == FMT_Q6_K ? 210 : (fmt == FMT_Q8_0 ? 272 : 160)));
}
// Units per stage: one tensor copy brings 16 rows of >= 544 bytes each (row-strided copies
// below ~576 bytes per row measured well under the HBM rate).
int stage_units_of(int fmt) { return fmt == FMT_Q8_0 ? 2 : 4; }

// Shared-memory layout of the streaming kernel for a plan and M tokens. The stage is the
// largest (units per row) that leaves a ring of >= 2 stages per warp. A row of a stage is
// `row_stride` bytes: the units plus a pad that puts consecutive rows in distinct banks
// for the fragment loads (the box reads the pad bytes from the next unit, or zeros past
// the end of the row). Returns false if nothing fits.
bool tma_layout(int fmt, const TmaPlan& pl, int M, TmaParams* prm, size_t* smem) {
  auto al = [](size_t v) { return (v + 127) & ~size_t(127); };
  const int T = M > 8 ? 16 : 8;
  const int ub = unit_bytes_of(fmt);
  const bool half_x = fmt == FMT_Q4_K || fmt == FMT_Q5_K || fmt == FMT_Q6_K || fmt == FMT_Q8_0;
  const bool row_copies = fmt == FMT_Q6_K;
  const int smax = (pl.units + pl.C - 1) / pl.C;
  int xstride = 0, xts = 0, s2ts = 0;
  size_t xbytes = 0, sbytes = 0;
  if (half_x) {  // M token rows + one zero row
    xts = smax * 512 + 64;
    s2ts = 32 * ((smax & 1) ? smax : smax + 1);
    xbytes = (size_t)(M + 1) * xts;
    sbytes = (size_t)(M + 1) * s2ts;
  } else {
    xstride = smax * kUnit + 32;
    xbytes = (size_t)T * xstride * 2;
    sbytes = (size_t)smax * 8 * T * 4;
  }
  size_t off = al(xbytes);
  const size_t off_ss = off;
  off = al(off + sbytes);
  const size_t off_aux = off;
  off = al(off + kAuxScaleBytes + 128);
  const size_t off_pb = off;
  off = al(off + (size_t)kWarps * 2 * 16 * T * 4);
  const size_t off_res = off;
  if (pl.C > 1) off = al(off + (size_t)pl.max_tiles * 16 * T * 4);
  const size_t off_bar = off;
  off = al(off + (size_t)kWarps * 8 * 8);
  const size_t off_ring = off;
  for (int su = stage_units_of(fmt); su >= 1; --su) {
    int stride = row_copies ? (su * ub + 30 + 15) / 16 * 16 : su * ub;  // + the span's alignment slack
    if (half_x && fmt != FMT_Q8_0) {  // quad loads of 16 bytes at 16 + 32q: rows must differ by 16 mod 32 bytes
      while (stride % 32 != 16) stride += 16;
    } else {       // 8-byte loads of 4 rows per phase: rows must differ by 32 or 96 mod 128
      while (stride % 128 != 32 && stride % 128 != 96) stride += 16;
    }
    if (!row_copies && stride / 4 > 256) continue;  // tensor-map box limit (256 elements)
    const size_t per_stage = (size_t)kWarps * 16 * stride;
    if (off + 2 * per_stage > (size_t)kSmemCap) continue;
    const int depth = (int)std::min<size_t>(8, ((size_t)kSmemCap - off) / per_stage);
    prm->su = su;
    prm->depth = depth;
    prm->row_stride = stride;
    prm->unit_bytes = ub;
    prm->xstride = xstride;
    prm->xts = xts;
    prm->s2ts = s2ts;
    prm->off_ss = (int)off_ss;
    prm->off_aux = (int)off_aux;
    prm->off_pb = (int)off_pb;
    prm->off_res = (int)off_res;
    prm->off_bar = (int)off_bar;
    prm->off_ring = (int)off_ring;
    *smem = off + (size_t)depth * per_stage;
    return true;
  }
  return false;
}

// Max co-resident clusters of C CTAs for the streaming kernel of `fmt` at `smem` bytes of
// shared memory per CTA. Cached per device, format and C. Returns 0 if the query fails.
int max_clusters(int fmt, int C, size_t smem) {
  static int cache[64][8][5];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return 0;
  int ci = 0;
  while ((1 << ci) < C) ++ci;
  int& slot = cache[dev][fmt & 7][ci];
  if (slot > 0) return slot;
  const void* fn = nullptr;
  if (fmt == FMT_Q4_K) fn = (const void*)gemv_tma_kernel<FmtQ4KH, 2>;
  else if (fmt == FMT_Q5_K) fn = (const void*)gemv_tma_kernel<FmtQ5KH, 2>;
  else if (fmt == FMT_Q6_K) fn = (const void*)gemv_tma_kernel<FmtQ6KH, 2>;
  else if (fmt == FMT_Q8_0) fn = (const void*)gemv_tma_kernel<FmtQ8_0H, 2>;
  else fn = (const void*)gemv_tma_kernel<FmtAffine4, 2>;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemCap) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  slot = n;
  return n;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr) ==
            cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

}  // namespace

TmaPlan plan_gemv_tma(int fmt, int N, int K, int num_sms) {
  TmaPlan best;
  best.ok = false;
  const int U = K / kUnit, tiles = (N + 15) / 16;
  long long best_work = -1;
  for (int C = 1; C <= kMaxClusterSize; C *= 2) {
    if (C > U) break;
    const int smax = (U + C - 1) / C;
    if (smax > kMaxSliceUnits) continue;
    // every launch of this kernel holds more than half an SM's shared memory, so the
    // co-resident cluster count depends on C only; query it at the full allowance
    int G = max_clusters(fmt, C, (size_t)kSmemCap);
    if (G <= 0) G = num_sms / C;
    if (G <= 0) break;
    if (G > tiles) G = tiles;
    const int ntmax = (tiles + G - 1) / G;
    if (C > 1 && ntmax > kMaxClusterTiles) continue;
    TmaPlan pl;
    pl.ok = true;
    pl.units = U;
    pl.tiles = tiles;
    pl.C = C;
    pl.G = G;
    pl.max_tiles = ntmax;
    TmaParams tmp;
    size_t sm16 = 0;
    if (!tma_layout(fmt, pl, 16, &tmp, &sm16)) continue;  // must fit for every M
    const long long work = ((long long)ntmax * smax + kWarps - 1) / kWarps;
    if (best_work < 0 || work < best_work) {
      best = pl;
      best_work = work;
    }
  }
  return best;
}

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

bool gemv_epilogue_ok(int fmt, int N, int K, int kind, int num_sms) {
  if (kind == 0) return true;
  if (fmt != FMT_Q4_K && fmt != FMT_Q5_K && fmt != FMT_Q8_0 && fmt != FMT_AFFINE4) return false;
  const TmaPlan tp = plan_gemv_tma(fmt, N, K, num_sms);
  if (!tp.ok || !encode_tiled_fn()) return false;
  return kind == 1 || kind == 3 || (kind == 2 && tp.C == 1 && N % 16 == 0);
}

int launch_gemv_mma(int fmt, const void* w, const void* x, float* y, int M, int N, int K,
                    long long row_bytes, int num_sms, cudaStream_t stream, bool overlap, std::string* err,
                    const GemvEpilogue* epi) {
  const bool two = M > 8;
  const TmaPlan tp = plan_gemv_tma(fmt, N, K, num_sms);
  EncodeTiledFn enc = encode_tiled_fn();
  const int kind = epi ? epi->kind : 0;
  if (kind != 0 && !gemv_epilogue_ok(fmt, N, K, kind, num_sms)) {
    *err = "internal: this GEMV shape cannot run the fused epilogue";
    return -1;
  }
  if (fmt == FMT_Q6_K) {
    // per-row copies round each row's span out to 16 bytes, which stays inside the weights
    // only if their total size is a multiple of 16; other shapes take the CUDA-core kernel
    if (!tp.ok || ((long long)N * row_bytes) % 16 != 0)
      return launch_gemv_q6k_bf16(w, static_cast<const uint16_t*>(x), y, M, N, K, row_bytes, stream, overlap, err);
  }
  if (tp.ok && (enc || fmt == FMT_Q6_K)) {
    TmaParams prm;
    prm.x = static_cast<const uint16_t*>(x);
    prm.y = y;
    prm.M = M;
    prm.N = N;
    prm.K = K;
    prm.units = tp.units;
    prm.tiles = tp.tiles;
    prm.C = tp.C;
    prm.G = tp.G;
    prm.max_tiles = tp.max_tiles;
    prm.epi = kind;
    prm.out2 = epi ? epi->out : nullptr;
    prm.e_v0 = epi ? epi->v0 : 0;
    prm.e_vn = epi ? epi->vn : 0;
    prm.e_hd = epi ? epi->hd : 1;
    prm.e_group = epi ? epi->group : 1;
    prm.e_w = epi ? epi->out_w : 0;
    prm.out3 = epi ? epi->out_b : nullptr;
    prm.e_row0 = epi ? epi->row0 : 0;
    prm.half = N / 2;
    prm.w = static_cast<const uint8_t*>(w);
    prm.row_bytes = row_bytes;
    size_t smem = 0;
    if (!tma_layout(fmt, tp, M, &prm, &smem)) {
      *err = "internal: streaming plan does not fit shared memory";
      return -1;
    }
    // W as a 2-D tensor of 4-byte words: rows of row_bytes, box = 16 rows x row_stride bytes
    CUtensorMap tm;
    std::memset(&tm, 0, sizeof(tm));
    if (fmt == FMT_Q6_K)  // rows copied one by one: no tensor map
      return two ? launch_tma<FmtQ6KH, 2>(tm, prm, smem, tp.G * tp.C, stream, overlap, err)
                 : launch_tma<FmtQ6KH, 1>(tm, prm, smem, tp.G * tp.C, stream, overlap, err);
    const cuuint64_t gdim[2] = {(cuuint64_t)(row_bytes / 4), (cuuint64_t)N};
    const cuuint64_t gstride[1] = {(cuuint64_t)row_bytes};
    const cuuint32_t box[2] = {(cuuint32_t)(prm.row_stride / 4), kind == 2 ? 8u : 16u};
    const cuuint32_t estride[2] = {1u, 1u};
    const CUresult cr = enc(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(w), gdim, gstride, box,
                            estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS) {
      *err = "cuTensorMapEncodeTiled failed (" + std::to_string((int)cr) + ")";
      return -1;
    }
    const int grid = tp.G * tp.C;
    switch (fmt) {
      case FMT_Q4_K:
        return two ? launch_tma<FmtQ4KH, 2>(tm, prm, smem, grid, stream, overlap, err)
                   : launch_tma<FmtQ4KH, 1>(tm, prm, smem, grid, stream, overlap, err);
      case FMT_Q8_0:
        return two ? launch_tma<FmtQ8_0H, 2>(tm, prm, smem, grid, stream, overlap, err)
                   : launch_tma<FmtQ8_0H, 1>(tm, prm, smem, grid, stream, overlap, err);
      case FMT_AFFINE4:
        return two ? launch_tma<FmtAffine4, 2>(tm, prm, smem, grid, stream, overlap, err)
                   : launch_tma<FmtAffine4, 1>(tm, prm, smem, grid, stream, overlap, err);
      case FMT_Q5_K:
        return two ? launch_tma<FmtQ5KH, 2>(tm, prm, smem, grid, stream, overlap, err)
                   : launch_tma<FmtQ5KH, 1>(tm, prm, smem, grid, stream, overlap, err);
    }
    *err = "unsupported format";
    return -1;
  }
  // K too long for one CTA's activation slice: register-streaming kernel with chunked staging.
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
  switch (fmt) {
    case FMT_Q4_K:
      return two ? launch_chunked<FMT_Q4_K, 2>(prm, smem, stream, err)
                 : launch_chunked<FMT_Q4_K, 1>(prm, smem, stream, err);
    case FMT_Q8_0:
      return two ? launch_chunked<FMT_Q8_0, 2>(prm, smem, stream, err)
                 : launch_chunked<FMT_Q8_0, 1>(prm, smem, stream, err);
    case FMT_AFFINE4:
      return two ? launch_chunked<FMT_AFFINE4, 2>(prm, smem, stream, err)
                 : launch_chunked<FMT_AFFINE4, 1>(prm, smem, stream, err);
    case FMT_Q5_K:
      return two ? launch_chunked<FMT_Q5_K, 2>(prm, smem, stream, err)
                 : launch_chunked<FMT_Q5_K, 1>(prm, smem, stream, err);
  }
  *err = "unsupported format";
  return -1;
}

unsigned int take_device_errors(std::string* err) {
  unsigned int v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_errors, sizeof(v));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_device_errors, &zero, sizeof(zero));
  if (e != cudaSuccess) {
    *err = std::string("reading the device error word: ") + cudaGetErrorString(e);
    return 0xFFFFFFFFu;
  }
  return v;
}

}  // namespace kq
