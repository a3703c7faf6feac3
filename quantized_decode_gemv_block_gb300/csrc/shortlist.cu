// Shortlist output head: the greedy next token of each of M <= 16 hidden states over a Q8_0
// output layer (Kinetic README, "What makes it fast": choosing the next token reads an
// output layer of up to a quarter of a million rows; every row's score is bounded from a
// small copy and exact scores are computed only for the rows that can still win).
//
// One call, three launches on the caller's stream:
//  1. the approximate scores a[j][n] = x_j . w'_n over the small copy (the Q4_K copy of the
//     head), by the streaming GEMV kernel (the caller's entry point runs it);
//  2. shortlist_lower_kernel: per chunk of 1024 rows and token, the largest lower bound
//     a[j][n] - B_n ||x_j|| and the largest upper bound a[j][n] + B_n ||x_j|| (B_n from the
//     small copy's build);
//  3. shortlist_exact_kernel: one CTA per chunk. A chunk whose largest upper bound reaches
//     no token's largest lower bound is skipped whole; in the others every row whose upper
//     bound reaches the largest lower bound of some token is scored exactly against the
//     Q8_0 weights, and the largest exact score wins (ties: the lowest row); the last CTA to
//     finish writes the tokens and scores.
// Every bound is evaluated with directed rounding (||x|| rounded up, B_n ||x|| rounded up,
// lower bounds rounded down, upper bounds rounded up), so the rounding of the bound
// arithmetic never prunes a row. B_n itself covers the copy's error and the fp32 rounding of
// both products, so the row with the largest exact score is never pruned: the result is the
// argmax of the exact scores of every row (the same as with the shortlist turned off).
//
// An exact score is one warp's fixed-order sum: lane l takes blocks l, l + 32, ... of the
// row, each block a sequential fp32 FMA chain over its 32 codes promoted by d with one FMA,
// and the lanes meet in a fixed butterfly. It does not depend on which warp, CTA or call
// computes it, nor on M (every token's chain is the same instructions).
//
// Launch chain: 2 and 3 use programmatic dependent launch. The bounds pass computes ||x||
// (x is complete before the GEMV starts) and the exact pass stages x in shared memory
// before they wait for their predecessor's results. While they wait, each runs its own code
// once on inputs that are not ready yet, storing nothing: run cold after the wait, the
// unrolled code was measured stalling on instruction fetch for several microseconds (the
// dry run of the exact pass saves 2.4 us per call at M = 1). Everything a kernel of the
// call produced (the scores, the chunk maxima, the norms) is read with L2-only loads
// (ld.global.cg): a dry pass reads those addresses before they are written, and a line it
// left in L1 must not answer the real pass.
#include "kq_device.cuh"
#include "kq_internal.h"

namespace kq {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kLowerRows = 1024;            // rows per CTA of the lower-bound pass
constexpr int kMaxTok = 16;
constexpr int kXSmemMax = 160 * 1024;       // x staged in shared memory up to this size

struct ShortlistState {
  float nx[kMaxTok];                  // ||x_j||, rounded up
  unsigned long long key[kMaxTok];    // (ordered score << 32) | (0xFFFFFFFF - row), max wins
  unsigned int scored;                // rows scored exactly
  unsigned int done;                  // CTAs of the exact pass finished
};

__device__ __forceinline__ uint32_t ordered_bits(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float from_ordered_bits(uint32_t o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}


// ||x_j||_2 rounded up for every token (every product, sum and the square root rounded
// toward +inf), in the same fixed order in every CTA: thread t sums its 16-byte chunks
// t, t + 256, ... element by element; then a warp butterfly; then the warps in order.
template <class XT>
__device__ void xnorms_up(const XT* __restrict__ x, int M, int K, float (*red)[kWarps], float* nx) {
  constexpr int kVec = 16 / sizeof(XT);
  float acc[kMaxTok];
#pragma unroll
  for (int j = 0; j < kMaxTok; ++j) acc[j] = 0.f;
  for (int c = threadIdx.x; c * kVec < K; c += kThreads) {
#pragma unroll
    for (int j = 0; j < kMaxTok; ++j) {
      if (j < M) {
        const uint4 u = ldg128(x + (size_t)j * K + (size_t)c * kVec);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if constexpr (sizeof(XT) == 2) {
            const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xFFFF0000u);
            acc[j] = __fmaf_ru(lo, lo, acc[j]);
            acc[j] = __fmaf_ru(hi, hi, acc[j]);
          } else {
            const float v = __uint_as_float(w[e]);
            acc[j] = __fmaf_ru(v, v, acc[j]);
          }
        }
      }
    }
  }
  const int warp = threadIdx.x >> 5;
#pragma unroll
  for (int j = 0; j < kMaxTok; ++j) {
    if (j < M) {
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) acc[j] = __fadd_ru(acc[j], __shfl_xor_sync(0xffffffffu, acc[j], off));
      if ((threadIdx.x & 31) == 0) red[j][warp] = acc[j];
    }
  }
  __syncthreads();
  if (threadIdx.x < M) {
    float s = 0.f;
    for (int w = 0; w < kWarps; ++w) s = __fadd_ru(s, red[threadIdx.x][w]);
    nx[threadIdx.x] = __fsqrt_ru(s);
  }
  __syncthreads();
}

// cta_max[c][0][j]: the largest lower bound of chunk c for token j; cta_max[c][1][j]: the
// largest upper bound (ordered bit patterns, 0 below everything). At most 80 registers a
// thread, so that a CTA fits beside a GEMV CTA (167 registers x 256 threads) and can start,
// and run its dry pass, while the GEMV streams.
template <class XT>
__global__ void __launch_bounds__(kThreads, 3) shortlist_lower_kernel(const float* __restrict__ ya,
                                                                   const float* __restrict__ bound,
                                                                   const XT* __restrict__ x, int M, int N, int K,
                                                                   uint32_t* __restrict__ cta_max,
                                                                   ShortlistState* __restrict__ st, int scan) {
  __shared__ float red[kMaxTok][kWarps];
  __shared__ float nx[kMaxTok];
  __shared__ uint32_t smax[2][kMaxTok];
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x < 2 * kMaxTok) smax[threadIdx.x / kMaxTok][threadIdx.x % kMaxTok] = 0u;
  xnorms_up(x, M, K, red, nx);
  if (blockIdx.x == 0) {  // fresh state for the exact pass, which reads it after this grid ends
    if (threadIdx.x < kMaxTok) {
      st->key[threadIdx.x] = 0ull;
      st->nx[threadIdx.x] = threadIdx.x < M ? nx[threadIdx.x] : 0.f;
    }
    if (threadIdx.x == 0) {
      st->scored = 0u;
      st->done = 0u;
    }
  }
  if (!scan) return;
  // Two passes over the same code: a dry one while the small copy's GEMV still runs (its
  // values are not ready and are discarded; it brings this code into the instruction
  // caches, which a single cold pass would wait on line by line), then the real one.
  const int n0 = blockIdx.x * kLowerRows;
#pragma unroll 1
  for (int pass = 0; pass < 2; ++pass) {
    if (pass == 1) asm volatile("griddepcontrol.wait;" ::: "memory");
    // rows n0 + t + 256 i, i < 4: every load issued first, then the bounds
    float bnd[4], yv[kMaxTok][4];
    int nn[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      nn[i] = n0 + threadIdx.x + kThreads * i;
      bnd[i] = nn[i] < N ? bound[nn[i]] : 0.f;
    }
#pragma unroll
    for (int j = 0; j < kMaxTok; ++j)
#pragma unroll
      for (int i = 0; i < 4; ++i) yv[j][i] = (j < M && nn[i] < N) ? __ldcg(ya + (size_t)j * N + nn[i]) : 0.f;
    uint32_t m[kMaxTok], u[kMaxTok];
#pragma unroll
    for (int j = 0; j < kMaxTok; ++j) {
      m[j] = 0u;
      u[j] = 0u;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (j < M && nn[i] < N) {
          // a NaN bound or score is not comparable: that row can never win, and it takes no
          // part in the maxima
          const float U = __fmul_ru(bnd[i], nx[j]), lo = __fsub_rd(yv[j][i], U), up = __fadd_ru(yv[j][i], U);
          if (lo == lo) m[j] = max(m[j], ordered_bits(lo));
          if (up == up) u[j] = max(u[j], ordered_bits(up));
        }
    }
#pragma unroll
    for (int j = 0; j < kMaxTok; ++j) {
      if (j < M) {
        const uint32_t r = __reduce_max_sync(0xffffffffu, m[j]), ru = __reduce_max_sync(0xffffffffu, u[j]);
        if ((threadIdx.x & 31) == 0 && pass == 1) {
          atomicMax(&smax[0][j], r);
          atomicMax(&smax[1][j], ru);
        }
      }
    }
  }
  __syncthreads();
  if (threadIdx.x < M) {
    cta_max[(blockIdx.x * 2) * kMaxTok + threadIdx.x] = smax[0][threadIdx.x];
    cta_max[(blockIdx.x * 2 + 1) * kMaxTok + threadIdx.x] = smax[1][threadIdx.x];
  }
}

// 8 consecutive activations (a 16- or 32-byte aligned group, in global or shared memory).
__device__ __forceinline__ void load_x8(const float* x, float (&v)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(x), b = *reinterpret_cast<const float4*>(x + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void load_x8(const uint16_t* x, float (&v)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(x);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    v[2 * e] = __uint_as_float(w[e] << 16);
    v[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
  }
}

// Exact scores of row `row` for tokens 0..MT-1 (tokens >= M repeat token M-1 and are
// ignored by the caller); x holds the M token rows K apart, in global or shared memory.
// Per block and token one sequential FMA chain over the 32 codes (taken 8 at a time by a
// compact loop: this code runs for a handful of rows per call, so its size, not its issue
// rate, sets its time), then acc += d * chain. Every lane returns the full sums.
template <class XT, int MT>
__device__ void exact_scores(const uint8_t* __restrict__ wq, const XT* x, int M, int K, int row, int lane,
                             float (&acc)[MT]) {
  const int nb = K / 32;
#pragma unroll
  for (int j = 0; j < MT; ++j) acc[j] = 0.f;
  const uint8_t* qrow = wq + (size_t)row * nb * 34;
  for (int g = lane; g < nb; g += 32) {
    const uint16_t* blk = reinterpret_cast<const uint16_t*>(qrow + (size_t)g * 34);  // 2-byte aligned
    const float d = __half2float(__ushort_as_half(blk[0]));
    float p[MT];
#pragma unroll
    for (int j = 0; j < MT; ++j) p[j] = 0.f;
#pragma unroll 1
    for (int i0 = 0; i0 < 32; i0 += 8) {
      float q[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t two = blk[1 + i0 / 2 + i];
        q[2 * i] = static_cast<float>(static_cast<int8_t>(two & 0xFFu));
        q[2 * i + 1] = static_cast<float>(static_cast<int8_t>(two >> 8));
      }
#pragma unroll
      for (int j = 0; j < MT; ++j) {
        float xv[8];
        load_x8(x + (size_t)min(j, M - 1) * K + (size_t)g * 32 + i0, xv);
#pragma unroll
        for (int i = 0; i < 8; ++i) p[j] = __fmaf_rn(q[i], xv[i], p[j]);
      }
    }
#pragma unroll
    for (int j = 0; j < MT; ++j) acc[j] = __fmaf_rn(d, p[j], acc[j]);
  }
#pragma unroll
  for (int j = 0; j < MT; ++j)
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) acc[j] = __fadd_rn(acc[j], __shfl_xor_sync(0xffffffffu, acc[j], off));
}

template <class XT, int MT>
__global__ void __launch_bounds__(kThreads, 2) shortlist_exact_kernel(
    const uint8_t* __restrict__ wq, const float* __restrict__ ya, const float* __restrict__ bound,
    const XT* __restrict__ x, int M, int N, int K, const uint32_t* __restrict__ cta_max, int nchunks,
    ShortlistState* __restrict__ st, int* __restrict__ token, float* __restrict__ score,
    unsigned int* __restrict__ scored, int all_rows, int staged) {
  extern __shared__ __align__(16) uint8_t xsm[];
  __shared__ float L[kMaxTok], nx[kMaxTok];
  __shared__ uint32_t lb[kMaxTok];
  __shared__ bool last, open;
  // x into shared memory (it is complete before this call's first kernel started)
  if (staged) {
    const int nvec = M * K * (int)sizeof(XT) / 16;
    const uint4* src = reinterpret_cast<const uint4*>(x);
    uint4* dst = reinterpret_cast<uint4*>(xsm);
#pragma unroll 4
    for (int v = threadIdx.x; v < nvec; v += kThreads) dst[v] = ldg128(src + v);
  }
  __syncthreads();
  const XT* xs = staged ? reinterpret_cast<const XT*>(xsm) : x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kLowerRows;
  unsigned int mine = 0u;
  // Two passes over the same code: a dry one while the bounds pass still runs (its inputs
  // are not ready; nothing is stored, and four warps score one row each, so the scoring code
  // too is in the instruction caches), then the real one behind griddepcontrol.wait.
#pragma unroll 1
  for (int pass = 0; pass < 2; ++pass) {
    const bool dry = pass == 0;
    if (!dry) asm volatile("griddepcontrol.wait;" ::: "memory");
    if (threadIdx.x < kMaxTok) lb[threadIdx.x] = 0u;
    if (threadIdx.x == 0) open = all_rows != 0;
    __syncthreads();
    // thread t reads the lower maxima of chunks t/16, t/16 + 16, ... for token t % 16: loads
    // eight at a time, then one shared max per thread
    if (!all_rows && (threadIdx.x & (kMaxTok - 1)) < M) {
      uint32_t m = 0u;
      const int j = threadIdx.x & (kMaxTok - 1);
      for (int c0 = threadIdx.x / kMaxTok; c0 < nchunks; c0 += 8 * (kThreads / kMaxTok)) {
        uint32_t v[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const int c = c0 + r * (kThreads / kMaxTok);
          v[r] = c < nchunks ? __ldcg(cta_max + (2 * c) * kMaxTok + j) : 0u;
        }
#pragma unroll
        for (int r = 0; r < 8; ++r) m = max(m, v[r]);
      }
      atomicMax(&lb[j], m);
    }
    __syncthreads();
    if (threadIdx.x < M) {
      L[threadIdx.x] = dry ? __uint_as_float(0x7F800000u) : from_ordered_bits(lb[threadIdx.x]);
      nx[threadIdx.x] = __ldcg(&st->nx[threadIdx.x]);
      // this chunk can hold a winner only if its largest upper bound reaches some token's L
      if (!all_rows && __ldcg(cta_max + (2 * blockIdx.x + 1) * kMaxTok + threadIdx.x) >= lb[threadIdx.x]) open = true;
    }
    __syncthreads();
    if (open || dry) {
      // rows n0 + 4t + i, i < 4 (16-byte loads when N % 4 == 0): every load first, then one
      // ballot per i
      unsigned int masks[4];
      const int nt = n0 + 4 * threadIdx.x;
      if (all_rows) {
#pragma unroll
        for (int i = 0; i < 4; ++i) masks[i] = __ballot_sync(0xffffffffu, nt + i < N);
      } else {
        float bnd[4], yv[kMaxTok][4];
        const bool vec = (N & 3) == 0 && nt < N;
        if (vec) {
          const float4 b4 = *reinterpret_cast<const float4*>(bound + nt);
          bnd[0] = b4.x; bnd[1] = b4.y; bnd[2] = b4.z; bnd[3] = b4.w;
#pragma unroll
          for (int j = 0; j < kMaxTok; ++j) {
            float4 y4 = make_float4(0.f, 0.f, 0.f, 0.f);
            if (j < M) y4 = __ldcg(reinterpret_cast<const float4*>(ya + (size_t)j * N + nt));
            yv[j][0] = y4.x; yv[j][1] = y4.y; yv[j][2] = y4.z; yv[j][3] = y4.w;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            bnd[i] = nt + i < N ? bound[nt + i] : 0.f;
#pragma unroll
            for (int j = 0; j < kMaxTok; ++j) yv[j][i] = (j < M && nt + i < N) ? __ldcg(ya + (size_t)j * N + nt + i) : 0.f;
          }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          bool cand = false;
#pragma unroll
          for (int j = 0; j < kMaxTok; ++j)
            if (j < M && nt + i < N) cand |= __fadd_ru(yv[j][i], __fmul_ru(bnd[i], nx[j])) >= L[j];
          masks[i] = __ballot_sync(0xffffffffu, cand);
        }
      }
      if (dry) {
        masks[0] = (warp < 4 && n0 + 128 * warp < N) ? 1u : 0u;
        masks[1] = masks[2] = masks[3] = 0u;
      }
#pragma unroll 1
      for (int i = 0; i < 4; ++i) {
        unsigned int mask = i == 0 ? masks[0] : i == 1 ? masks[1] : i == 2 ? masks[2] : masks[3];
        if (!dry) mine += __popc(mask);
        while (mask) {
          const int row = n0 + 4 * (warp * 32 + __ffs(mask) - 1) + i;
          mask &= mask - 1u;
          float acc[MT];
          exact_scores<XT, MT>(wq, xs, M, K, row, lane, acc);
          float v = acc[0];
#pragma unroll
          for (int j = 1; j < MT; ++j)
            if (lane == j) v = acc[j];
          if (!dry && lane < M && v == v) {  // a NaN score never wins
            const unsigned long long key = (static_cast<unsigned long long>(ordered_bits(v)) << 32) |
                                           static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<uint32_t>(row));
            atomicMax(&st->key[lane], key);
          }
        }
      }
    }
    __syncthreads();
  }
  if (lane == 0 && mine) atomicAdd(&st->scored, mine);
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    last = atomicAdd(&st->done, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  if (threadIdx.x < M) {
    const unsigned long long key = atomicAdd(&st->key[threadIdx.x], 0ull);
    if (key == 0ull) {  // no row had a comparable (non-NaN) score
      token[threadIdx.x] = -1;
      score[threadIdx.x] = __uint_as_float(0x7FC00000u);
    } else {
      token[threadIdx.x] = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(key & 0xFFFFFFFFull));
      score[threadIdx.x] = from_ordered_bits(static_cast<uint32_t>(key >> 32));
    }
  }
  if (threadIdx.x == 0 && scored) *scored = atomicAdd(&st->scored, 0u);
}

// One launch of kThreads-thread CTAs, optionally allowed to begin before the previous kernel
// on the stream finishes (it then waits with griddepcontrol.wait before reading its output).
template <class... KArgs, class... Args>
cudaError_t launch_chained(void (*kern)(KArgs...), int grid, size_t smem, bool pdl, cudaStream_t s,
                           Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

size_t al256(size_t v) { return (v + 255) & ~size_t(255); }
int lower_ctas_of(int N) { return (N + kLowerRows - 1) / kLowerRows; }

struct SelectArgs {
  const uint8_t* w;
  const float* ya;
  const float* bound;
  const void* x;
  int M, N, K;
  uint32_t* cta_max;
  int lc;
  ShortlistState* st;
  int* token;
  float* score;
  unsigned int* scored;
  bool all_rows;
  int num_sms;
};

template <class XT, int MT>
cudaError_t launch_select(const SelectArgs& a, cudaStream_t s) {
  const XT* x = static_cast<const XT*>(a.x);
  const size_t xbytes = (size_t)a.M * a.K * sizeof(XT);
  const bool staged = xbytes <= (size_t)kXSmemMax;
  auto exact = shortlist_exact_kernel<XT, MT>;
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(exact, cudaFuncAttributeMaxDynamicSharedMemorySize, kXSmemMax);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  // the bounds pass follows the small copy's GEMV with programmatic dependent launch; with
  // every row scored it follows whatever the caller ran last, so it waits for it in full
  cudaError_t e = launch_chained(shortlist_lower_kernel<XT>, a.all_rows ? 1 : a.lc, 0, !a.all_rows, s, a.ya,
                                 a.bound, x, a.M, a.N, a.K, a.cta_max, a.st, a.all_rows ? 0 : 1);
  if (e != cudaSuccess) return e;
  // one CTA per chunk of rows
  return launch_chained(exact, a.lc, staged ? xbytes : 0, true, s, a.w, a.ya, a.bound, x, a.M, a.N, a.K,
                        static_cast<const uint32_t*>(a.cta_max), a.lc, a.st, a.token, a.score, a.scored,
                        a.all_rows ? 1 : 0, staged ? 1 : 0);
}

template <class XT>
cudaError_t launch_select_m(const SelectArgs& a, cudaStream_t s) {
  if (a.M <= 1) return launch_select<XT, 1>(a, s);
  if (a.M <= 2) return launch_select<XT, 2>(a, s);
  if (a.M <= 4) return launch_select<XT, 4>(a, s);
  if (a.M <= 8) return launch_select<XT, 8>(a, s);
  return launch_select<XT, 16>(a, s);
}

}  // namespace

size_t shortlist_small_bytes(int N, int K) { return al256((size_t)N * (K / 256) * 144); }
size_t shortlist_bytes(int N, int K) { return shortlist_small_bytes(N, K) + al256((size_t)N * 4); }

size_t head_argmax_workspace(int M, int N) {
  return al256((size_t)M * N * 4) + al256((size_t)lower_ctas_of(N) * 2 * kMaxTok * 4) + al256(sizeof(ShortlistState));
}

int launch_head_select(const void* wq, const void* shortlist, bool x_bf16, const void* x, int M, int N, int K,
                       int* token, float* score, unsigned int* scored, void* ws, bool all_rows, int num_sms,
                       cudaStream_t s, std::string* err) {
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  SelectArgs a;
  a.w = static_cast<const uint8_t*>(wq);
  a.ya = reinterpret_cast<const float*>(w8);
  a.bound = all_rows ? nullptr
                     : reinterpret_cast<const float*>(static_cast<const uint8_t*>(shortlist) +
                                                      shortlist_small_bytes(N, K));
  a.x = x;
  a.M = M;
  a.N = N;
  a.K = K;
  a.lc = lower_ctas_of(N);
  a.cta_max = reinterpret_cast<uint32_t*>(w8 + al256((size_t)M * N * 4));
  a.st = reinterpret_cast<ShortlistState*>(w8 + al256((size_t)M * N * 4) + al256((size_t)a.lc * 2 * kMaxTok * 4));
  a.token = token;
  a.score = score;
  a.scored = scored;
  a.all_rows = all_rows;
  a.num_sms = num_sms;
  const cudaError_t e = x_bf16 ? launch_select_m<uint16_t>(a, s) : launch_select_m<float>(a, s);
  if (e != cudaSuccess) {
    *err = std::string("shortlist launch: ") + cudaGetErrorString(e);
    return -1;
  }
  return 0;
}

}  // namespace kq
