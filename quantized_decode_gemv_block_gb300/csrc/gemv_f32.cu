// CUDA-core GEMV for fp32 activations (every format) and for bf16 activations of Q6_K
// blocks whose shape the tensor-core streaming kernel does not take (a K-slice too long for
// its shared memory, or a weight buffer whose size is not a multiple of 16 bytes), M = 1..16.
// Q6_K's 210-byte blocks leave rows only 2-byte aligned, so Q6_K is read with 16-bit loads here.
//
// Same product as the tensor-core path, Y[j][n] = sum_k deq(W)[n][k] * X[j][k]
// (Kinetic README, "What makes it fast"), for callers whose activations are fp32
// (an fp32 value does not fit a bf16 MMA operand exactly). Each warp owns two rows;
// lane (gi, q) takes weights 8q..8q+7 of 32-group gi of every 256-weight unit. Per
// 8-weight slice it forms P = sum code*x and S = sum x in fp32 and promotes with
// acc = fma(scale, P, acc) and acc = fma(offset, S, acc); the 32 lane partials are
// added by a fixed butterfly. Each token's chain of operations is the same for every
// M (the kernel is instantiated for 1, 2, 4, 8 or 16 token slots and M only masks),
// so a row's bits do not depend on the batch.
#include "kq_device.cuh"
#include "kq_internal.h"

namespace kq {
namespace {

constexpr int kThreadsF = 256;
constexpr int kRowsPerWarp = 2;

__device__ __forceinline__ uint32_t ldg16(const void* p) {
  unsigned short v;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

template <int FMT>
__device__ __forceinline__ void decode_slice(const uint8_t* unit, int gi, int q, float (&c)[8],
                                             float& scale, float& offset) {
  if (FMT == FMT_Q6_K) {
    // weights 32gi + 8q + k: half n = gi/4, quarter kq = gi%4, l = 8q + k; sub-block 2gi + q/2
    const int n = gi >> 2, kq = gi & 3;
    const uint8_t* qlp = unit + 64 * n + 32 * (kq & 1) + 8 * q;
    const uint8_t* qhp = unit + 128 + 32 * n + 8 * q;
    const int b = 2 * gi + (q >> 1);
    const uint32_t sp = ldg16(unit + 192 + (b & ~1));
    const int sc = static_cast<int>(static_cast<int8_t>((b & 1) ? (sp >> 8) : (sp & 0xFFu)));
    scale = half_bits_to_float(ldg16(unit + 208)) * static_cast<float>(sc);  // exact: 11-bit x 8-bit
    offset = 0.f;
    const int nsh = (kq >= 2) ? 4 : 0, hsh = 2 * kq;
#pragma unroll
    for (int k = 0; k < 8; k += 2) {
      const uint32_t l2 = ldg16(qlp + k), h2 = ldg16(qhp + k);
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const uint32_t lo4 = ((l2 >> (8 * e)) >> nsh) & 15u, hi2 = ((h2 >> (8 * e)) >> hsh) & 3u;
        c[k + e] = static_cast<float>(static_cast<int>(lo4 | (hi2 << 4)) - 32);
      }
    }
  } else if (FMT == FMT_Q4_K) {
    const uint4 h = ldg128(unit);
    const int ch = gi >> 1;
    const uint2 b = ldg64(unit + 16 + 32 * ch + 8 * q);
    const uint32_t s0 = h.y, s1 = h.z, s2 = h.w;
    uint32_t scw, mw;
    if (gi < 4) {
      scw = s0 & 0x3F3F3F3Fu;
      mw = s1 & 0x3F3F3F3Fu;
    } else {
      scw = (s2 & 0x0F0F0F0Fu) | ((s0 >> 2) & 0x30303030u);
      mw = ((s2 >> 4) & 0x0F0F0F0Fu) | ((s1 >> 2) & 0x30303030u);
    }
    const int sh = 8 * (gi & 3);
    const float sc = static_cast<float>((scw >> sh) & 0xFFu);
    const float m = static_cast<float>((mw >> sh) & 0xFFu);
    const float d = half_bits_to_float(h.x), dmin = half_bits_to_float(h.x >> 16);
    scale = d * sc;      // exact: 11-bit x 6-bit
    offset = -dmin * m;  // exact
    const int nsh = (gi & 1) ? 4 : 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      c[k] = static_cast<float>((b.x >> (8 * k + nsh)) & 15u);
      c[4 + k] = static_cast<float>((b.y >> (8 * k + nsh)) & 15u);
    }
  } else if (FMT == FMT_Q5_K) {  // Q4_K's scales; low nibbles at 48, fifth bits (bit gi of qh[l]) at 16
    const uint4 h = ldg128(unit);
    const int ch = gi >> 1;
    const uint2 b = ldg64(unit + 48 + 32 * ch + 8 * q);
    const uint2 hb = ldg64(unit + 16 + 8 * q);
    const uint32_t s0 = h.y, s1 = h.z, s2 = h.w;
    uint32_t scw, mw;
    if (gi < 4) {
      scw = s0 & 0x3F3F3F3Fu;
      mw = s1 & 0x3F3F3F3Fu;
    } else {
      scw = (s2 & 0x0F0F0F0Fu) | ((s0 >> 2) & 0x30303030u);
      mw = ((s2 >> 4) & 0x0F0F0F0Fu) | ((s1 >> 2) & 0x30303030u);
    }
    const int sh = 8 * (gi & 3);
    const float sc = static_cast<float>((scw >> sh) & 0xFFu);
    const float m = static_cast<float>((mw >> sh) & 0xFFu);
    const float d = half_bits_to_float(h.x), dmin = half_bits_to_float(h.x >> 16);
    scale = d * sc;      // exact: 11-bit x 6-bit
    offset = -dmin * m;  // exact
    const int nsh = (gi & 1) ? 4 : 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      c[k] = static_cast<float>(((b.x >> (8 * k + nsh)) & 15u) | (((hb.x >> (8 * k + gi)) & 1u) << 4));
      c[4 + k] = static_cast<float>(((b.y >> (8 * k + nsh)) & 15u) | (((hb.y >> (8 * k + gi)) & 1u) << 4));
    }
  } else if (FMT == FMT_Q8_0) {
    const uint8_t* blk = unit + 34 * gi;
    scale = half_bits_to_float(ldg16(blk));
    offset = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t v = ldg16(blk + 2 + 8 * q + 2 * k);
      c[2 * k] = static_cast<float>(static_cast<int8_t>(v & 0xFFu));
      c[2 * k + 1] = static_cast<float>(static_cast<int8_t>(v >> 8));
    }
  } else {
    const uint8_t* grp = unit + 20 * gi;
    const uint32_t sb = ldg32(grp);
    const uint32_t cw = ldg32(grp + 4 + 4 * q);
    scale = half_bits_to_float(sb);
    offset = half_bits_to_float(sb >> 16);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      c[2 * k] = static_cast<float>((cw >> (8 * k)) & 15u);
      c[2 * k + 1] = static_cast<float>((cw >> (8 * k + 4)) & 15u);
    }
  }
}

// Raw bytes one lane needs from a Q6_K unit for its 8-weight slice (16-bit loads: Q6_K rows
// are only 2-byte aligned): 8 bytes of ql, 8 of qh, the scale pair, d.
struct Q6Raw {
  unsigned short l[4], h[4], s, d;
};
__device__ __forceinline__ void q6_load_raw(Q6Raw& r, const uint8_t* unit, int ql_off, int qh_off, int s_off) {
  const unsigned short* u16 = reinterpret_cast<const unsigned short*>(unit);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    r.l[k] = __ldg(u16 + (ql_off >> 1) + k);
    r.h[k] = __ldg(u16 + (qh_off >> 1) + k);
  }
  r.s = __ldg(u16 + (s_off >> 1));
  r.d = __ldg(u16 + 104);
}

template <int FMT>
constexpr int unit_bytes() {
  return FMT == FMT_Q4_K ? 144 : (FMT == FMT_Q5_K ? 176 : (FMT == FMT_Q6_K ? 210 : (FMT == FMT_Q8_0 ? 272 : 160)));
}

// 8 activations of token j at k (a multiple of 8) as fp32: XT = float, or uint16_t (bf16 bits).
template <class XT>
__device__ __forceinline__ void load_x8f(const XT* x, long long off, float (&xv)[8]) {
  if constexpr (sizeof(XT) == 4) {
    const uint4 v0 = ldg128(x + off), v1 = ldg128(x + off + 4);
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) xv[k] = __uint_as_float(w[k]);
  } else {
    const uint4 v = ldg128(x + off);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      xv[2 * k] = __uint_as_float(w[k] << 16);
      xv[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
  }
}

// KS warps share each row pair, each taking a contiguous 1/KS of the K units; their sums
// meet in shared memory and are added in slice order (KS depends on N, K and the SM count).
template <int FMT, int MT, class XT, int KS>
__global__ void __launch_bounds__(kThreadsF) gemv_f32_kernel(const uint8_t* __restrict__ w,
                                                             const XT* __restrict__ x,
                                                             float* __restrict__ y, int M, int N,
                                                             int K, long long row_bytes) {
  constexpr int kGroups = 8 / KS;  // row pairs per CTA
  __shared__ float red[KS > 1 ? 8 * kRowsPerWarp * MT : 1];
  // Programmatic dependent launch (when the launch allows it): a following launch may begin
  // now; this one loads its first unit's weights before it waits for the previous grid, and
  // reads x and writes y only after that wait (a no-op for a plain launch).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gi = lane >> 2, q = lane & 3;
  const int rg = warp / KS, ks = warp - rg * KS;
  const int nbase = (blockIdx.x * kGroups + rg) * kRowsPerWarp;
  float acc[kRowsPerWarp][MT];
#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i)
#pragma unroll
    for (int j = 0; j < MT; ++j) acc[i][j] = 0.f;

  const int units_all = K / 256;
  const int u0 = ks * units_all / KS, u1 = (ks + 1) * units_all / KS;
  if (FMT == FMT_Q6_K) {
    // Q6_K: the next unit's raw bytes are loaded (plain, schedulable loads) before the
    // current unit is decoded, so each warp keeps two units of loads in flight.
    const int n = gi >> 2, kq = gi & 3;
    const int ql_off = 64 * n + 32 * (kq & 1) + 8 * q, qh_off = 128 + 32 * n + 8 * q;
    const int b = 2 * gi + (q >> 1), s_off = 192 + (b & ~1);
    const int nsh = (kq >= 2) ? 4 : 0, hsh = 2 * kq;
    Q6Raw nxt[kRowsPerWarp];
    if (u0 < u1) {
#pragma unroll
      for (int i = 0; i < kRowsPerWarp; ++i)
        q6_load_raw(nxt[i], w + min(nbase + i, N - 1) * row_bytes + (long long)u0 * 210, ql_off, qh_off, s_off);
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int u = u0; u < u1; ++u) {
      Q6Raw cur[kRowsPerWarp];
#pragma unroll
      for (int i = 0; i < kRowsPerWarp; ++i) cur[i] = nxt[i];
      if (u + 1 < u1) {
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i)
          q6_load_raw(nxt[i], w + min(nbase + i, N - 1) * row_bytes + (long long)(u + 1) * 210, ql_off, qh_off, s_off);
      }
      float c[kRowsPerWarp][8], sc[kRowsPerWarp];
#pragma unroll
      for (int i = 0; i < kRowsPerWarp; ++i) {
        const int scv = static_cast<int>(static_cast<int8_t>((b & 1) ? (cur[i].s >> 8) : (cur[i].s & 0xFFu)));
        sc[i] = half_bits_to_float(cur[i].d) * static_cast<float>(scv);  // exact: 11-bit x 8-bit
#pragma unroll
        for (int k = 0; k < 4; ++k) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const uint32_t lo4 = ((static_cast<uint32_t>(cur[i].l[k]) >> (8 * e)) >> nsh) & 15u;
            const uint32_t hi2 = ((static_cast<uint32_t>(cur[i].h[k]) >> (8 * e)) >> hsh) & 3u;
            c[i][2 * k + e] = static_cast<float>(static_cast<int>(lo4 | (hi2 << 4)) - 32);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < MT; ++j) {
        if (j < M) {
          float xv[8];
          load_x8f<XT>(x, (long long)j * K + u * 256 + 32 * gi + 8 * q, xv);
#pragma unroll
          for (int i = 0; i < kRowsPerWarp; ++i) {
            float p = 0.f;
#pragma unroll
            for (int k = 0; k < 8; ++k) p = __fmaf_rn(c[i][k], xv[k], p);
            acc[i][j] = __fmaf_rn(sc[i], p, acc[i][j]);
          }
        }
      }
    }
  } else {
  for (int u = u0; u < u1; ++u) {
    float c[kRowsPerWarp][8], sc[kRowsPerWarp], off[kRowsPerWarp];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
      const int row = min(nbase + i, N - 1);
      decode_slice<FMT>(w + row * row_bytes + (long long)u * unit_bytes<FMT>(), gi, q, c[i], sc[i],
                        off[i]);
    }
    if (u == u0) asm volatile("griddepcontrol.wait;" ::: "memory");
#pragma unroll
    for (int j = 0; j < MT; ++j) {
      if (j < M) {
        float xv[8];
        load_x8f<XT>(x, (long long)j * K + u * 256 + 32 * gi + 8 * q, xv);
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) s = __fadd_rn(s, xv[k]);
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) {
          float p = 0.f;
#pragma unroll
          for (int k = 0; k < 8; ++k) p = __fmaf_rn(c[i][k], xv[k], p);
          acc[i][j] = __fmaf_rn(sc[i], p, acc[i][j]);
          if (FMT != FMT_Q8_0 && FMT != FMT_Q6_K) acc[i][j] = __fmaf_rn(off[i], s, acc[i][j]);  // min / bias
        }
      }
    }
  }
  }
  if (u0 >= u1) asm volatile("griddepcontrol.wait;" ::: "memory");  // a warp with no units still stores
#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) {
#pragma unroll
    for (int j = 0; j < MT; ++j) {
      float v = acc[i][j];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
      if (KS == 1) {
        if (lane == 0 && j < M && nbase + i < N) y[(long long)j * N + nbase + i] = v;
      } else if (lane == 0) {
        red[(warp * kRowsPerWarp + i) * MT + j] = v;
      }
    }
  }
  if (KS > 1) {
    __syncthreads();
    if (ks == 0 && lane < kRowsPerWarp * MT) {
      const int i = lane / MT, j = lane - i * MT;
      float v = red[(warp * kRowsPerWarp + i) * MT + j];
#pragma unroll
      for (int k2 = 1; k2 < KS; ++k2) v = __fadd_rn(v, red[((warp + k2) * kRowsPerWarp + i) * MT + j]);
      if (j < M && nbase + i < N) y[(long long)j * N + nbase + i] = v;
    }
  }
}

template <int FMT, int MT, class XT, int KS>
void launch_one(const uint8_t* w, const XT* x, float* y, int M, int N, int K, long long row_bytes,
                cudaStream_t s, bool overlap) {
  const int rows = (8 / KS) * kRowsPerWarp;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((N + rows - 1) / rows, 1, 1);
  cfg.blockDim = dim3(kThreadsF, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap ? 1 : 0;
  cudaLaunchKernelEx(&cfg, gemv_f32_kernel<FMT, MT, XT, KS>, w, x, y, M, N, K, row_bytes);
}

template <int FMT, class XT, int KS>
void launch_ks(const uint8_t* w, const XT* x, float* y, int M, int N, int K, long long row_bytes,
               cudaStream_t s, bool overlap) {
  if (M <= 1) launch_one<FMT, 1, XT, KS>(w, x, y, M, N, K, row_bytes, s, overlap);
  else if (M <= 2) launch_one<FMT, 2, XT, KS>(w, x, y, M, N, K, row_bytes, s, overlap);
  else if (M <= 4) launch_one<FMT, 4, XT, KS>(w, x, y, M, N, K, row_bytes, s, overlap);
  else if (M <= 8) launch_one<FMT, 8, XT, KS>(w, x, y, M, N, K, row_bytes, s, overlap);
  else launch_one<FMT, 16, XT, KS>(w, x, y, M, N, K, row_bytes, s, overlap);
}

// The K split: the smallest KS (1, 2, 4, 8) that gives at least eight CTAs per SM while every
// slice keeps at least two units. A function of (N, K, SM count) only.
int pick_ks(int N, int K) {
  static int sms[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  int n_sm = dev < 64 ? sms[dev] : 0;
  if (n_sm == 0) {
    cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
    if (n_sm <= 0) n_sm = 1;
    if (dev < 64) sms[dev] = n_sm;
  }
  const int units = K / 256;
  int ks = 1;
  while (ks < 8 && (long long)((N + (8 / ks) * kRowsPerWarp - 1) / ((8 / ks) * kRowsPerWarp)) < 8LL * n_sm &&
         units / (2 * ks) >= 2)
    ks *= 2;
  return ks;
}

template <int FMT, class XT>
int launch_fmt(const uint8_t* w, const XT* x, float* y, int M, int N, int K,
               long long row_bytes, cudaStream_t s, bool overlap) {
  switch (pick_ks(N, K)) {
    case 1: launch_ks<FMT, XT, 1>(w, x, y, M, N, K, row_bytes, s, overlap); break;
    case 2: launch_ks<FMT, XT, 2>(w, x, y, M, N, K, row_bytes, s, overlap); break;
    case 4: launch_ks<FMT, XT, 4>(w, x, y, M, N, K, row_bytes, s, overlap); break;
    default: launch_ks<FMT, XT, 8>(w, x, y, M, N, K, row_bytes, s, overlap); break;
  }
  return 0;
}

}  // namespace

int launch_gemv_f32(int fmt, const void* w, const float* x, float* y, int M, int N, int K,
                    long long row_bytes, cudaStream_t stream, bool overlap, std::string* err) {
  const uint8_t* wb = static_cast<const uint8_t*>(w);
  switch (fmt) {
    case FMT_Q4_K: launch_fmt<FMT_Q4_K>(wb, x, y, M, N, K, row_bytes, stream, overlap); break;
    case FMT_Q8_0: launch_fmt<FMT_Q8_0>(wb, x, y, M, N, K, row_bytes, stream, overlap); break;
    case FMT_AFFINE4: launch_fmt<FMT_AFFINE4>(wb, x, y, M, N, K, row_bytes, stream, overlap); break;
    case FMT_Q5_K: launch_fmt<FMT_Q5_K>(wb, x, y, M, N, K, row_bytes, stream, overlap); break;
    case FMT_Q6_K: launch_fmt<FMT_Q6_K>(wb, x, y, M, N, K, row_bytes, stream, overlap); break;
    default: *err = "unsupported format"; return -1;
  }
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    *err = std::string("gemv (fp32 x) launch: ") + cudaGetErrorString(e);
    return -1;
  }
  return 0;
}

int launch_gemv_q6k_bf16(const void* w, const uint16_t* x, float* y, int M, int N, int K, long long row_bytes,
                         cudaStream_t stream, bool overlap, std::string* err) {
  launch_fmt<FMT_Q6_K>(static_cast<const uint8_t*>(w), x, y, M, N, K, row_bytes, stream, overlap);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    *err = std::string("gemv (Q6_K, bf16 x) launch: ") + cudaGetErrorString(e);
    return -1;
  }
  return 0;
}

}  // namespace kq
