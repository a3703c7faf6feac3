// Prefill product on the 5th-generation tensor cores (tcgen05): Y = X * deq(W)^T for many
// tokens (Kinetic README, "What makes it fast": long prompts run as tiled matrix products,
// so each weight block is unpacked once and used for many tokens).
//
// Q4_K weights, bf16 activations, fp32 output. The Q4_K weight of sub-block b of super-block
// s is w = d_s * (sc_b * q) - dmin_s * m_b, so
//   Y[j][n] = sum_s d_s * (sum_{k in s} x[j][k] * t[n][k])  -  sum_b (dmin*m)_b * S_b(x[j]),
// with t = sc*q a small integer (<= 945, exact in fp16) and S_b(x) the sum of x over the 32
// k of sub-block b. Every product the tensor cores form is exact:
//  * a pre-pass writes X as fp16 under an exact per-token power of two (the token's largest
//    |x| lands in [2^14, 2^15)), followed by the per-sub-block sums S/64 split into fp16
//    hi + lo, and writes -64*dmin*m (exact in fp32) split into fp16 hi + lo for W;
//  * the main k-tiles multiply X by t, one super-block (4 k-tiles of 64) per accumulator
//    group in tensor memory; an extra group multiplies [S_hi S_lo S_hi] by [M_hi M_hi M_lo]
//    (the min term to 2^-22);
//  * epilogue warps read each finished group from tensor memory and add d_s times it (fp32)
//    into registers, so the only roundings are fp32 ones.
//
// Orientation: the tensor-core A operand is the weight tile (128 rows of W), B is the token
// tile (256 tokens), so tensor-memory lane = weight row and column = token: d_s is one scalar
// per thread, and Y stores are 128-byte rows. Roles in a CTA (persistent over output tiles):
//   warps 0..7   epilogue (warp w: lanes 32*(w%4).., tokens 128*(w/4)..), 128 fp32 sums each
//   warps 8..9   unpack t = sc*q for the 128 weight rows of the tile (2 rows per thread) into
//                the K-major 128-byte-swizzled A tile of the stage ring
//   warp 10      TMA: token tiles (256 x 64 fp16) and the W min-term tiles (128 x 64 fp16)
//   warp 11      one thread issues tcgen05.mma (M=128, N=256, K=16) and owns tensor memory
// Every mbarrier wait is bounded: a timeout records the device error word, raises an abort
// flag that every role checks, and the CTA drains its own copies and MMAs and returns.
#include <cuda.h>
#include <cuda_fp16.h>

#include "kq_device.cuh"
#include "kq_internal.h"

namespace kq {

__device__ unsigned int g_tc_errors = 0;  // bit 0: a bounded wait in the prefill kernel gave up

namespace {

constexpr int TM = 128;  // weight rows per tile (MMA M)
constexpr int TN = 256;  // tokens per tile (MMA N)
constexpr int BK = 64;   // k per stage (one 128-byte swizzle row of fp16)
constexpr int STAGES = 4;
constexpr int kWTileBytes = TM * BK * 2;  // 16 KB
constexpr int kXTileBytes = TN * BK * 2;  // 32 KB
constexpr int kStageBytes = kWTileBytes + kXTileBytes;
constexpr int kEpiWarps = 8, kDqWarps = 2;
constexpr int kDqBase = kEpiWarps * 32;
constexpr int kDqThreads = kDqWarps * 32;  // each unpacks rows u and u + 64
constexpr int kTmaWarp = kEpiWarps + kDqWarps, kMmaWarp = kTmaWarp + 1;
constexpr int kTcThreads = (kMmaWarp + 1) * 32;
constexpr int kTmemCols = 2 * TN;  // two accumulator groups in flight
constexpr int kInvBytes = kEpiWarps * (TN / 2) * 4;  // per epilogue warp: its tokens' 2^-e_j
constexpr int kTcSmem = STAGES * kStageBytes + 1024 /*barriers*/ + kInvBytes + 1024 /*alignment slack*/;
constexpr uint64_t kTcWaitNs = 2000000000ull;
static_assert(kDqThreads * 2 == TM, "two weight rows per unpacking thread");

struct TcParams {
  const uint8_t* w;
  float* y;
  const float* inv_scale;  // per token (padded to a multiple of TN entries)
  int M, N, K;
  long long row_bytes;
  int n_ext;    // min-term k-tiles per tile
  int m_tiles;  // token tiles
  int tiles;    // m_tiles * weight-row tiles
};

// UMMA shared-memory descriptor: K-major operand, 128-byte swizzle, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) /* LBO (unused for SW128 K-major) */
         | ((uint64_t)(1024 >> 4) << 32) /* SBO */ | ((uint64_t)1 << 46) /* version */
         | ((uint64_t)2 << 61) /* SWIZZLE_128B */;
}

// Instruction descriptor, kind::f16: D fp32, A and B fp16, both K-major, M = 128, N = 256.
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(TN >> 3) << 17) | ((uint32_t)(TM >> 4) << 24);

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(kIdesc), "r"(accumulate)
      : "memory");
}
// Arrive on `bar` once every tcgen05.mma issued so far by this thread has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// 16 consecutive fp32 columns of this warp's 32 tensor-memory lanes.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tma_load_2d_sw(void* dst, const void* tmap, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_addr(dst)), "l"(tmap), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

// Byte offset of 16-byte chunk `kchunk` of row r in a K-major 64-wide fp16 tile with the
// 128-byte swizzle: 8-row groups of 1024 B; within a 128-B row, chunk c sits at c ^ (r % 8).
__device__ __forceinline__ int sw128_off(int r, int kchunk) {
  return (r >> 3) * 1024 + (r & 7) * 128 + ((kchunk ^ (r & 7)) << 4);
}

// fp16 pair (v, v) of a float.
__device__ __forceinline__ uint32_t h2_splat(float v) {
  const uint32_t b = __half_as_ushort(__float2half_rn(v));
  return b | (b << 16);
}

// The 64 values t = sc*q of k-chunk kc (0..3) of one Q4_K super-block, as fp16 (exact), into
// row r of the swizzled tile. s0..s2 = the block's 12 scale bytes (words 1..3 of its header);
// qa, qb = quant bytes 32kc..32kc+31 (low nibbles: sub-block 2kc, k = 0..31 of the chunk;
// high nibbles: sub-block 2kc+1, k = 32..63). A nibble pair is placed in fp16 words as
// 1024 + q (low) or 1024 + 16q (high); one fma removes the offset and multiplies by sc.
__device__ __forceinline__ void unpack_t(uint32_t s0, uint32_t s2, const uint4& qa, const uint4& qb, int kc,
                                         uint8_t* tile, int r) {
  int scl, sch;
  if (kc < 2) {  // sub-blocks 0..3: low 6 bits of scale bytes 0..3
    scl = (s0 >> (16 * kc)) & 63;
    sch = (s0 >> (16 * kc + 8)) & 63;
  } else {  // sub-blocks 4..7: low 4 bits from bytes 8..11, top 2 bits from bytes 0..3
    const int bl = 16 * (kc - 2), bh = bl + 8;
    scl = ((s2 >> bl) & 15) | (((s0 >> (bl + 6)) & 3) << 4);
    sch = ((s2 >> bh) & 15) | (((s0 >> (bh + 6)) & 3) << 4);
  }
  const uint32_t a_l = h2_splat((float)scl), c_l = h2_splat(-1024.f * (float)scl);
  const uint32_t a_h = h2_splat((float)sch * 0.0625f), c_h = h2_splat(-64.f * (float)sch);
  const uint32_t qw[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
  uint32_t lo[16], hi[16];  // fp16 pairs: lo[2i], lo[2i+1] = k (4i, 4i+1), (4i+2, 4i+3)
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t p01 = prmt(qw[i], 0u, 0x3120u), p23 = prmt(qw[i], 0u, 0x1302u);
    lo[2 * i] = h2_fma(and_or(p01, 0x000F000Fu, 0x64006400u), a_l, c_l);
    lo[2 * i + 1] = h2_fma(and_or(p23, 0x000F000Fu, 0x64006400u), a_l, c_l);
    hi[2 * i] = h2_fma(and_or(p01, 0x00F000F0u, 0x64006400u), a_h, c_h);
    hi[2 * i + 1] = h2_fma(and_or(p23, 0x00F000F0u, 0x64006400u), a_h, c_h);
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) {  // chunk c: k = 8c..8c+7 (low), chunk c + 4: k = 32 + 8c.. (high)
    *reinterpret_cast<uint4*>(tile + sw128_off(r, c)) = make_uint4(lo[4 * c], lo[4 * c + 1], lo[4 * c + 2], lo[4 * c + 3]);
    *reinterpret_cast<uint4*>(tile + sw128_off(r, c + 4)) =
        make_uint4(hi[4 * c], hi[4 * c + 1], hi[4 * c + 2], hi[4 * c + 3]);
  }
}

// Bring super-block `sb` of a weight row into L2 (no registers, no completion to wait for).
__device__ __forceinline__ void prefetch_block_l2(const uint8_t* rowp, int sb) {
  const uint8_t* b = rowp + (long long)sb * 144;  // 144 bytes: at most two 128-byte lines
  asm volatile("prefetch.global.L2 [%0];" ::"l"(b) : "memory");
  asm volatile("prefetch.global.L2 [%0];" ::"l"(b + 143) : "memory");
}
constexpr int kPrefetchBlocks = 3;  // super-blocks (12 k-tiles) ahead of the unpacking

struct RowChunk {  // what one row needs for one k-tile: header words, 32 quant bytes
  uint4 h, a, b;
};

__device__ __forceinline__ void load_chunk(RowChunk& c, const uint8_t* rowp, int kt, bool new_block) {
  const uint8_t* blk = rowp + (long long)(kt >> 2) * 144;
  if (new_block) c.h = ldg128(blk);
  c.a = ldg128(blk + 16 + 32 * (kt & 3));
  c.b = ldg128(blk + 32 + 32 * (kt & 3));
}

__global__ void __launch_bounds__(kTcThreads, 1)
    gemm_q4k_tc_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap emap,
                       const TcParams p) {
  extern __shared__ uint8_t tc_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_x = reinterpret_cast<uint64_t*>(smem + STAGES * kStageBytes);  // TMA bytes landed
  uint64_t* full_w = full_x + STAGES;                                             // t tile written
  uint64_t* empty = full_w + STAGES;                                              // MMAs read the stage
  uint64_t* acc_full = empty + STAGES;                                            // [2] group finished
  uint64_t* acc_empty = acc_full + 2;                                             // [2] group read out
  uint64_t* mma_done = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  unsigned int* abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nsb = p.K / 256, kt_main = p.K / BK, kt_tile = p.n_ext + kt_main;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_x[s], 1);
      mbar_init(&full_w[s], kDqThreads);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], kEpiWarps);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0u;
    fence_mbar_init();
    asm volatile("prefetch.tensormap [%0];" ::"l"(&xmap) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&emap) : "memory");
  }
  if (warp == kMmaWarp) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto aborted = [&]() { return *(volatile unsigned int*)abort_flag != 0u; };
  auto fail = [&]() {
    atomicOr(&g_tc_errors, 1u);
    atomicOr(abort_flag, 1u);
  };
  auto stage_free = [&](int it) {  // wait until the MMAs of the stage's previous use are done
    return it < STAGES ||
           mbar_wait_bounded(&empty[it % STAGES], static_cast<uint32_t>(it / STAGES - 1) & 1u, kTcWaitNs);
  };

  if (warp == kTmaWarp) {
    if (lane == 0) {
      int it = 0;
      bool stop = false;
      for (int tile = blockIdx.x; tile < p.tiles && !stop; tile += gridDim.x) {
        const int m0 = (tile % p.m_tiles) * TN, n0 = (tile / p.m_tiles) * TM;
        for (int kt = 0; kt < kt_tile; ++kt) {
          const int s = it % STAGES;
          if (!stage_free(it)) { fail(); stop = true; break; }
          if (aborted()) { stop = true; break; }
          uint8_t* st = smem + s * kStageBytes;
          if (kt < p.n_ext) {  // min-term tile: the tokens' sums and W's -64*dmin*m, both by TMA
            mbar_arrive_expect_tx(&full_x[s], kXTileBytes + kWTileBytes);
            tma_load_2d_sw(st + kWTileBytes, &xmap, p.K + kt * BK, m0, &full_x[s]);
            tma_load_2d_sw(st, &emap, kt * BK, n0, &full_x[s]);
          } else {
            mbar_arrive_expect_tx(&full_x[s], kXTileBytes);
            tma_load_2d_sw(st + kWTileBytes, &xmap, (kt - p.n_ext) * BK, m0, &full_x[s]);
          }
          ++it;
        }
      }
      // On an abort, let the copies still in flight land before the CTA can exit.
      if (aborted())
        for (int j = max(0, it - STAGES); j < it; ++j)
          mbar_wait_bounded(&full_x[j % STAGES], static_cast<uint32_t>(j / STAGES) & 1u, kTcWaitNs);
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      int it = 0, grp = 0;
      bool stop = false;
      for (int tile = blockIdx.x; tile < p.tiles && !stop; tile += gridDim.x) {
        for (int g = 0; g <= nsb && !stop; ++g, ++grp) {  // group 0: min term; 1..nsb: super-blocks
          const int buf = grp & 1;
          if (grp >= 2 && !mbar_wait_bounded(&acc_empty[buf], static_cast<uint32_t>(grp / 2 - 1) & 1u, kTcWaitNs)) {
            fail();
            stop = true;
            break;
          }
          tc_fence_after();
          const int kt0 = g == 0 ? 0 : p.n_ext + 4 * (g - 1), kt1 = g == 0 ? p.n_ext : kt0 + 4;
          for (int kt = kt0; kt < kt1; ++kt) {
            const int s = it % STAGES;
            const uint32_t par = static_cast<uint32_t>(it / STAGES) & 1u;
            if (!mbar_wait_bounded(&full_x[s], par, kTcWaitNs) || !mbar_wait_bounded(&full_w[s], par, kTcWaitNs)) {
              fail();
              stop = true;
              break;
            }
            if (aborted()) { stop = true; break; }
            tc_fence_after();
            const uint32_t wa = smem_addr(smem + s * kStageBytes), xa = wa + kWTileBytes;
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              umma_f16(tmem + (uint32_t)(buf * TN), smem_desc_sw128(wa + 32 * kk), smem_desc_sw128(xa + 32 * kk),
                       (kt != kt0 || kk != 0) ? 1u : 0u);
            umma_commit(&empty[s]);
            ++it;
          }
          if (!stop) umma_commit(&acc_full[buf]);
        }
      }
      umma_commit(mma_done);  // the wait point for every MMA this thread issued
      if (!mbar_wait_bounded(mma_done, 0u, kTcWaitNs)) fail();
    }
  } else if (warp >= kEpiWarps) {  // warps 8..9: unpack t = sc*q for rows u and u + 64
    const int u = threadIdx.x - kDqBase;
    int it = 0;
    bool stop = false;
    for (int tile = blockIdx.x; tile < p.tiles && !stop; tile += gridDim.x) {
      const int n0 = (tile / p.m_tiles) * TM;
      // rows past N repeat row N-1; their outputs are never stored
      const uint8_t* rowa = p.w + (long long)min(n0 + u, p.N - 1) * p.row_bytes;
      const uint8_t* rowb = p.w + (long long)min(n0 + u + 64, p.N - 1) * p.row_bytes;
      RowChunk na, nb;
      load_chunk(na, rowa, 0, true);
      load_chunk(nb, rowb, 0, true);
      // the unpacking reads each row from HBM one k-tile ahead, too late to hide its latency:
      // keep the next few super-blocks of both rows on their way into L2
      for (int j = 1; j <= kPrefetchBlocks && j < nsb; ++j) {
        prefetch_block_l2(rowa, j);
        prefetch_block_l2(rowb, j);
      }
      for (int kt = 0; kt < kt_tile; ++kt) {
        const int s = it % STAGES;
        const RowChunk ca = na, cb = nb;
        const int km = kt - p.n_ext;  // main k-tile index, < 0 for min-term tiles
        if (km >= 0 && km + 1 < kt_main) {  // next chunk's bytes in flight while this one unpacks
          load_chunk(na, rowa, km + 1, ((km + 1) & 3) == 0);
          load_chunk(nb, rowb, km + 1, ((km + 1) & 3) == 0);
        }
        if (km >= 0 && (km & 3) == 0 && (km >> 2) + kPrefetchBlocks + 1 < nsb) {
          prefetch_block_l2(rowa, (km >> 2) + kPrefetchBlocks + 1);
          prefetch_block_l2(rowb, (km >> 2) + kPrefetchBlocks + 1);
        }
        if (!stage_free(it)) { fail(); stop = true; break; }
        if (aborted()) { stop = true; break; }
        if (km >= 0) {
          uint8_t* wt = smem + s * kStageBytes;
          unpack_t(ca.h.y, ca.h.w, ca.a, ca.b, km & 3, wt, u);
          unpack_t(cb.h.y, cb.h.w, cb.a, cb.b, km & 3, wt, u + 64);
          fence_proxy_async_smem();  // generic-proxy smem writes -> visible to the tensor core
        }
        mbar_arrive(&full_w[s]);
        ++it;
      }
    }
  } else {  // warps 0..7: epilogue
    const int quarter = warp & 3, half = warp >> 2;
    int grp = 0;
    bool stop = false;
    for (int tile = blockIdx.x; tile < p.tiles && !stop; tile += gridDim.x) {
      const int m0 = (tile % p.m_tiles) * TN, n0 = (tile / p.m_tiles) * TM;
      const int n = n0 + quarter * 32 + lane;
      const uint8_t* rowp = p.w + (long long)min(n, p.N - 1) * p.row_bytes;
      float acc[TN / 2];
#pragma unroll
      for (int c = 0; c < TN / 2; ++c) acc[c] = 0.f;
      // this warp's tokens' 2^-e_j, fetched now (their latency hides behind the first group)
      // and read back from shared memory by the stores at the end of the tile
      float* winv = reinterpret_cast<float*>(smem + STAGES * kStageBytes + 1024) + warp * (TN / 2);
      for (int c = lane; c < TN / 2; c += 32) winv[c] = p.inv_scale[m0 + half * (TN / 2) + c];
      for (int g = 0; g <= nsb; ++g, ++grp) {
        const int buf = grp & 1;
        const float scale = g == 0 ? 1.0f : half_bits_to_float(ldg32(rowp + (long long)(g - 1) * 144));
        const bool ok = mbar_wait_bounded(&acc_full[buf], static_cast<uint32_t>(grp / 2) & 1u, kTcWaitNs);
        if (!__all_sync(0xFFFFFFFFu, ok)) { fail(); stop = true; break; }
        if (__any_sync(0xFFFFFFFFu, aborted())) { stop = true; break; }
        tc_fence_after();
        const uint32_t base = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(buf * TN + half * (TN / 2));
#pragma unroll
        for (int c0 = 0; c0 < TN / 2; c0 += 16) {
          float v[16];
          tmem_ld16(base + (uint32_t)c0, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) acc[c0 + i] = __fmaf_rn(scale, v[i], acc[c0 + i]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);
      }
      if (stop) break;
      // Y[j][n] = acc * 2^-e_j: for each token, the warp's 32 lanes write 32 consecutive floats
      const int j0 = m0 + half * (TN / 2);
      const bool nok = n < p.N;
      __syncwarp();
#pragma unroll
      for (int c0 = 0; c0 < TN / 2; c0 += 4) {
        const float4 inv = *reinterpret_cast<const float4*>(winv + c0);
        const float iv[4] = {inv.x, inv.y, inv.z, inv.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int j = j0 + c0 + i;
          // Y is written once and not read here: stream it (evict-first in L2)
          if (nok && j < p.M) __stcs(p.y + (long long)j * p.N + n, acc[c0 + i] * iv[i]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// The pre-pass, one launch:
//  blocks [0, M): token j. x'[k] = fp16(x[k] * 2^e) (exact; the token's max |x| lands in
//    [2^14, 2^15)), then for each sub-block b the fp32 sum S of its 32 x' (four sums of 8,
//    k ascending, added as (s0 + s1) + (s2 + s3)), S/64 = hi + lo in fp16, written as
//    [x' (K) | hi (K/32) | lo (K/32) | hi (K/32) | 0 ...].
//    inv_scale[j] = 2^-e.
//  blocks [M, ...): one thread per (weight row, super-block): -64*dmin*m_b (exact in fp32)
//    = hi + lo in fp16, written as [hi (K/32) | hi (K/32) | lo (K/32) | 0 ...].
__global__ void __launch_bounds__(256) prefill_prep_kernel(const uint16_t* __restrict__ x, __half* __restrict__ xc,
                                                           float* __restrict__ inv_scale, const uint8_t* __restrict__ w,
                                                           __half* __restrict__ wext, int M, int N, int K, int kc_x,
                                                           int k_ext, long long row_bytes) {
  const int G = K / 32;
  if ((int)blockIdx.x < M) {
    __shared__ unsigned int smax;
    const int tok = blockIdx.x, nch = K / 8;  // 16-byte chunks of the row; 4 per sub-block
    if (threadIdx.x == 0) smax = 0u;
    __syncthreads();
    const uint16_t* xr = x + (long long)tok * K;
    unsigned int best = 0u;
    for (int c = threadIdx.x; c < nch; c += 256) {
      const uint4 v = ldg128(xr + 8 * c);
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) best = max(best, max((wv[i] & 0x7FFFu) << 16, wv[i] & 0x7FFF0000u));
    }
    atomicMax(&smax, best);
    __syncthreads();
    const unsigned int mb = smax;
    const int E = static_cast<int>(mb >> 23);
    int e = 0;
    if (mb != 0u && E < 255) e = max(-126, min(127, 14 - (E == 0 ? -126 : E - 127)));
    const float sc = __int_as_float((e + 127) << 23);
    if (threadIdx.x == 0) inv_scale[tok] = 1.0f / sc;
    __half* xo = xc + (long long)tok * kc_x;
    // every thread converts whole chunks; a sub-block's four chunks sit in four adjacent
    // lanes, whose sums (each k ascending) meet as (c0 + c1) + (c2 + c3)
    for (int base = 0; base < nch; base += 256) {
      const int c = base + threadIdx.x;
      float s = 0.f;
      if (c < nch) {
        const uint4 v = ldg128(xr + 8 * c);
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const __half a = __float2half_rn(__uint_as_float(wv[i] << 16) * sc);
          const __half b = __float2half_rn(__uint_as_float(wv[i] & 0xFFFF0000u) * sc);
          s += __half2float(a);
          s += __half2float(b);
          o[i] = (uint32_t)__half_as_ushort(a) | ((uint32_t)__half_as_ushort(b) << 16);
        }
        *reinterpret_cast<uint4*>(xo + 8 * c) = make_uint4(o[0], o[1], o[2], o[3]);
      }
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      s += __shfl_xor_sync(0xffffffffu, s, 2);
      if (c < nch && (c & 3) == 0) {
        const int g = c >> 2;
        const float s64 = s * 0.015625f;
        const __half hi = __float2half_rn(s64);
        const __half lo = __float2half_rn(s64 - __half2float(hi));
        xo[K + g] = hi;
        xo[K + G + g] = lo;
        xo[K + 2 * G + g] = hi;
      }
    }
    for (int i = K + 3 * G + threadIdx.x; i < kc_x; i += 256) xo[i] = __ushort_as_half(0);
  } else {
    const int nsb = K / 256;
    const long long idx = (long long)(blockIdx.x - M) * 256 + threadIdx.x;
    if (idx >= (long long)N * nsb) return;
    const int n = (int)(idx / nsb), sb = (int)(idx - (long long)n * nsb);
    const uint8_t* blk = w + (long long)n * row_bytes + (long long)sb * 144;
    const uint4 h = ldg128(blk);
    const float dmin = half_bits_to_float(h.x >> 16);
    const uint32_t s1 = h.z, s2 = h.w;
    uint32_t ohi[4], olo[4];
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
      uint32_t hv[2], lv[2];
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int b = j + t;  // min of sub-block b: bytes 4..7 (b < 4), else bytes 8..11 and 4..7
        int m;
        if (b < 4) m = (s1 >> (8 * b)) & 63;
        else m = ((s2 >> (8 * (b - 4) + 4)) & 15) | (((s1 >> (8 * (b - 4) + 6)) & 3) << 4);
        const float v = -64.f * dmin * (float)m;  // exact: 11-bit dmin times 6-bit m
        const __half hi = __float2half_rn(v);
        const __half lo = __float2half_rn(v - __half2float(hi));
        hv[t] = __half_as_ushort(hi);
        lv[t] = __half_as_ushort(lo);
      }
      ohi[j / 2] = hv[0] | (hv[1] << 16);
      olo[j / 2] = lv[0] | (lv[1] << 16);
    }
    __half* er = wext + (long long)n * k_ext;
    *reinterpret_cast<uint4*>(er + 8 * sb) = make_uint4(ohi[0], ohi[1], ohi[2], ohi[3]);
    *reinterpret_cast<uint4*>(er + G + 8 * sb) = make_uint4(ohi[0], ohi[1], ohi[2], ohi[3]);
    *reinterpret_cast<uint4*>(er + 2 * G + 8 * sb) = make_uint4(olo[0], olo[1], olo[2], olo[3]);
    if (sb == 0)
      for (int i = 3 * G; i < k_ext; i += 8) *reinterpret_cast<uint4*>(er + i) = make_uint4(0u, 0u, 0u, 0u);
  }
}

struct TcLayout {
  int k_ext;  // min-term columns, a multiple of BK (>= 3K/32)
  int kc_x;   // converted token row length: K + k_ext
  int m_pad;  // tokens rounded up to TN (inv_scale entries)
  size_t off_inv, off_wext, bytes;
};

TcLayout tc_layout(int M, int N, int K) {
  auto al = [](size_t v) { return (v + 255) & ~size_t(255); };
  TcLayout L;
  L.k_ext = ((3 * (K / 32) + BK - 1) / BK) * BK;
  L.kc_x = K + L.k_ext;
  L.m_pad = ((M + TN - 1) / TN) * TN;
  L.off_inv = al((size_t)M * L.kc_x * 2);
  L.off_wext = L.off_inv + al((size_t)L.m_pad * 4);
  L.bytes = L.off_wext + al((size_t)N * L.k_ext * 2);
  return L;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// fp16 rows x cols row-major matrix as a 2-D tensor map with 128-byte swizzled 64 x box_rows boxes.
int encode_f16_2d(CUtensorMap* map, void* base, int cols, int rows, int box_rows, std::string* err) {
  static EncodeTiledFn enc = nullptr;
  if (!enc) {
    void* fp = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fp, 12000, cudaEnableDefault, &qr) != cudaSuccess ||
        qr != cudaDriverEntryPointSuccess) {
      *err = "cuTensorMapEncodeTiled is unavailable";
      return -1;
    }
    enc = reinterpret_cast<EncodeTiledFn>(fp);
  }
  const cuuint64_t gdim[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t gstride[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  const cuuint32_t es[2] = {1u, 1u};
  const CUresult cr = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, gdim, gstride, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) {
    *err = "cuTensorMapEncodeTiled failed (" + std::to_string((int)cr) + ")";
    return -1;
  }
  return 0;
}

}  // namespace

size_t gemm_tc_workspace(int M, int N, int K) { return tc_layout(M, N, K).bytes; }

int launch_gemm_tc(const void* w, const void* x, float* y, int M, int N, int K, long long row_bytes, void* ws,
                   int num_sms, cudaStream_t stream, std::string* err) {
  const TcLayout L = tc_layout(M, N, K);
  const long long m_tiles = (M + TN - 1) / TN, n_tiles = (N + TM - 1) / TM;
  if (m_tiles * n_tiles > 0x7FFFFFFFLL) { *err = "M x N has too many output tiles"; return -1; }
  const long long prep_w_blocks = ((long long)N * (K / 256) + 255) / 256;
  if ((long long)M + prep_w_blocks > 0x7FFFFFFFLL) { *err = "M and N too large for the pre-pass grid"; return -1; }
  uint8_t* base = static_cast<uint8_t*>(ws);
  __half* xc = reinterpret_cast<__half*>(base);
  float* inv = reinterpret_cast<float*>(base + L.off_inv);
  __half* wext = reinterpret_cast<__half*>(base + L.off_wext);
  prefill_prep_kernel<<<(unsigned)(M + prep_w_blocks), 256, 0, stream>>>(
      static_cast<const uint16_t*>(x), xc, inv, static_cast<const uint8_t*>(w), wext, M, N, K, L.kc_x, L.k_ext,
      row_bytes);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) { *err = std::string("prefill pre-pass launch: ") + cudaGetErrorString(e); return -1; }
  CUtensorMap xmap, emap;
  if (encode_f16_2d(&xmap, xc, L.kc_x, M, TN, err) || encode_f16_2d(&emap, wext, L.k_ext, N, TM, err)) return -1;
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    e = cudaFuncSetAttribute(gemm_q4k_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
    if (e != cudaSuccess) { *err = std::string("cudaFuncSetAttribute (gemm): ") + cudaGetErrorString(e); return -1; }
    attr_done[dev] = true;
  }
  TcParams prm;
  prm.w = static_cast<const uint8_t*>(w);
  prm.y = y;
  prm.inv_scale = inv;
  prm.M = M;
  prm.N = N;
  prm.K = K;
  prm.row_bytes = row_bytes;
  prm.n_ext = L.k_ext / BK;
  prm.m_tiles = (int)m_tiles;
  prm.tiles = (int)(m_tiles * n_tiles);
  const int grid = (int)std::min<long long>(prm.tiles, num_sms);
  gemm_q4k_tc_kernel<<<grid, kTcThreads, kTcSmem, stream>>>(xmap, emap, prm);
  e = cudaGetLastError();
  if (e != cudaSuccess) { *err = std::string("gemm launch: ") + cudaGetErrorString(e); return -1; }
  return 0;
}

unsigned int take_tc_errors() {
  unsigned int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_tc_errors, sizeof(v)) != cudaSuccess) return 0xFFFFFFFFu;
  cudaMemcpyToSymbol(g_tc_errors, &z, sizeof(z));
  return v;
}

}  // namespace kq
