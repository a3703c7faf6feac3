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
// Two SMs per MMA (tcgen05 cta_group::2): a cluster of two CTAs owns an output tile of 256
// weight rows x 256 tokens. CTA rank r holds the A operand for weight rows 128r.. of the tile
// and the B operand for tokens 128r..; one thread of rank 0 issues M = 256, N = 256, K = 16
// MMAs that read both CTAs' shared memory, and each CTA's tensor memory receives its own 128
// rows x 256 tokens. Per SM and k-tile that is 16 KB of t and 16 KB of tokens written and read
// once, against 16 + 32 KB for a one-SM MMA of the same shape: the copies, the unpacking
// stores and the tensor core's operand reads share each SM's shared-memory bandwidth.
//
// Orientation: A = weight tile, B = token tile, so tensor-memory lane = weight row and column =
// token: d_s is one scalar per thread, and Y stores are 128-byte rows. Roles in each CTA
// (persistent over output tiles, both CTAs of a pair walk the same tile sequence):
//   warps 0..7   epilogue (warp w: lanes 32*(w%4).., tokens 128*(w/4)..), 128 fp32 sums each
//   warps 8..9   unpack t = sc*q for the CTA's 128 weight rows (2 rows per thread) from raw
//                Q4_K super-blocks that a tensor copy brought into shared memory, into the
//                K-major 128-byte-swizzled A tile of the stage ring
//   warp 10      tensor copies: the CTA's half of each token tile (128 x 64 fp16) and of the
//                W min-term tiles (128 x 64 fp16), completing on rank 0's barrier
//   warp 11      tensor memory (both ranks); rank 0: one thread issues the MMAs
// Stage handshakes meet on rank 0's barriers: the copies by byte count, the unpacking and
// epilogue warps of rank 1 through one forwarding thread of rank 1 (a cluster-scope release
// stalls the warp that makes it); MMA completions are multicast to both CTAs. Every mbarrier wait is bounded: a
// timeout records the device error word, raises the abort flag of both CTAs (every role checks
// it), and the CTAs drain their copies and MMAs and return.
#include <cooperative_groups.h>
#include <cuda.h>
#include <cuda_fp16.h>

#include "kq_device.cuh"
#include "kq_internal.h"

namespace cg = cooperative_groups;

namespace kq {

__device__ unsigned int g_tc_errors = 0;  // bit 0: a bounded wait in the prefill kernel gave up

namespace {

constexpr int TM = 128;  // weight rows per CTA (half of the pair's MMA M = 256)
constexpr int TN = 256;  // tokens per tile (MMA N); each CTA stages TN / 2 of them
constexpr int BK = 64;   // k per stage (one 128-byte swizzle row of fp16)
constexpr int STAGES = 5;
constexpr int RAW_STAGES = 3;
// A parity wait is only sound while its barrier cannot be two phases behind the one awaited.
// Stages free in k-tile order (MMA completion); a waiter for k-tile e waits for the MMAs of
// e - STAGES and already knows those of some e - d to be done; it needs d <= 2 * STAGES.
constexpr int kWTileBytes = TM * BK * 2;        // 16 KB
constexpr int kXTileBytes = (TN / 2) * BK * 2;  // 16 KB: this CTA's half of the token tile
constexpr int kStageBytes = kWTileBytes + kXTileBytes;
constexpr int kRawBytes = TM * 144;  // one Q4_K super-block of the CTA's 128 rows
// Four warpgroups: 0-1 epilogue, 2 unpacking, 3 copies / MMA (warps 14-15 idle). The
// epilogue's 128 fp32 sums per thread need more registers than the 128 a 512-thread CTA starts
// with: warpgroups 2 and 3 hand theirs over (setmaxnreg), 2*128*176 + 128*104 + 128*56 = 512*128.
constexpr int kEpiWarps = 8, kDqWarps = 4;
constexpr int kDqBase = kEpiWarps;  // first unpacking warp
constexpr int kTmaWarp = kEpiWarps + kDqWarps, kMmaWarp = kTmaWarp + 1;
constexpr int kTcThreads = 16 * 32;
constexpr int kLaunchRegs = 128, kEpiRegs = 176, kDqRegs = 104, kCtlRegs = 56;
static_assert(kTcThreads * kLaunchRegs == 65536, "the CTA holds the whole register file");
static_assert(kDqWarps <= STAGES, "an unpacking warp's previous wait was kDqWarps + STAGES k-tiles back");
static_assert(2 * 128 * kEpiRegs + 128 * kDqRegs + 128 * kCtlRegs == kTcThreads * kLaunchRegs, "register split");
constexpr int kTmemCols = 2 * TN;  // two accumulator groups in flight
constexpr int kBarBytes = 1024;
constexpr int kInvBytes = kEpiWarps * (TN / 2) * 4;  // per epilogue warp: its tokens' 2^-e_j
constexpr int kTcSmem = STAGES * kStageBytes + RAW_STAGES * kRawBytes + kBarBytes + kInvBytes + 1024 /*alignment*/;
constexpr uint64_t kTcWaitNs = 2000000000ull;
static_assert(kTcSmem <= 232448, "shared memory per CTA");

struct TcParams {
  const uint8_t* w;
  float* y;
  const float* inv_scale;  // per token (padded to a multiple of TN entries)
  int M, N, K;
  long long row_bytes;
  int n_ext;    // min-term k-tiles per tile
  int m_tiles;  // token tiles
  int tiles;    // m_tiles * weight-row tiles (of 2 * TM rows)
};

// UMMA shared-memory descriptor: K-major operand, 128-byte swizzle, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) /* LBO (unused for SW128 K-major) */
         | ((uint64_t)(1024 >> 4) << 32) /* SBO */ | ((uint64_t)1 << 46) /* version */
         | ((uint64_t)2 << 61) /* SWIZZLE_128B */;
}

// Instruction descriptor, kind::f16: D fp32, A and B fp16, both K-major, M = 256 (the pair),
// N = 256.
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(TN >> 3) << 17) | ((uint32_t)((2 * TM) >> 4) << 24);

// Tensor memory of the pair: one warp of each CTA takes part in both calls.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void umma_pair_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(kIdesc), "r"(accumulate)
      : "memory");
}
// Arrive once on `bar` (the same offset in both CTAs of the pair) when every tcgen05.mma issued
// so far by this thread has completed.
__device__ __forceinline__ void umma_commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_addr(bar)),
      "h"((uint16_t)3)
      : "memory");
}
// The shared::cluster address of `p`'s counterpart in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
  return r;
}
// Arrive on a barrier of either CTA (default semantics: a cluster-scope release here stalled
// the arriving thread for ~0.4 us per call).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}
__device__ __forceinline__ void mbar_arrive_local(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
// Non-blocking test of a phase (this CTA's barrier).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
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

// 2-D tensor copy into this CTA's shared memory whose completion (bytes) is counted on a
// barrier of either CTA of the pair (bar: shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const void* tmap, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3}], [%4];" ::"r"(smem_addr(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(bar)
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

// k-chunk kc of the super-block of row r (144 bytes at row * 144 of a raw stage) into row r of
// the swizzled tile.
__device__ __forceinline__ void unpack_row(const uint8_t* raw_stage, int r, int kc, uint8_t* tile) {
  const uint8_t* b = raw_stage + r * 144;
  const uint4 h = lds128(b), qa = lds128(b + 16 + 32 * kc), qb = lds128(b + 32 + 32 * kc);
  unpack_t(h.y, h.w, qa, qb, kc, tile, r);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kTcThreads, 1)
    gemm_q4k_tc_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap emap,
                       const __grid_constant__ CUtensorMap wmap, const TcParams p) {
  extern __shared__ uint8_t tc_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* raw = smem + STAGES * kStageBytes;     // stage s: t tile, then this CTA's token tile
  uint64_t* full_x = reinterpret_cast<uint64_t*>(raw + RAW_STAGES * kRawBytes);  // rank 0: copies landed
  uint64_t* full_w = full_x + STAGES;             // each: the CTA's t tile written (rank 0: and rank 1's)
  uint64_t* empty = full_w + STAGES;              // each: the pair's MMAs read the stage
  uint64_t* acc_full = empty + STAGES;            // each [2]: group finished
  uint64_t* acc_empty = acc_full + 2;             // each [2]: the CTA's epilogue read the group (rank 0: and rank 1's)
  uint64_t* raw_full = acc_empty + 2;             // each [RAW_STAGES]: raw super-block landed
  uint64_t* raw_empty = raw_full + RAW_STAGES;    // each [RAW_STAGES]: the super-block's 4 k-tiles unpacked
  uint64_t* mma_done = raw_empty + RAW_STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  unsigned int* abort_flag = tmem_slot + 1;
  float* inv_base = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(full_x) + kBarBytes);

  cg::cluster_group cluster = cg::this_cluster();
  const uint32_t rank = cluster.block_rank();
  const bool leader = rank == 0;
  const int pair = static_cast<int>(blockIdx.x >> 1), npairs = static_cast<int>(gridDim.x >> 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nsb = p.K / 256, kt_main = p.K / BK, kt_tile = p.n_ext + kt_main;

  if (threadIdx.x == 0) {
    // rank 1's unpacking and epilogue warps arrive on their own barriers; one thread of rank 1
    // forwards each completed phase to rank 0 (a cluster-scope release per stage, not per warp)
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_x[s], 1);
      mbar_init(&full_w[s], 1 + (leader ? 1 : 0));  // the warp that unpacked the stage (+ rank 1's)
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], kEpiWarps + (leader ? 1 : 0));
    }
    for (int r = 0; r < RAW_STAGES; ++r) {
      mbar_init(&raw_full[r], 1);
      mbar_init(&raw_empty[r], 4);  // one arrival per k-tile of the super-block
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0u;
    fence_mbar_init();
    asm volatile("prefetch.tensormap [%0];" ::"l"(&xmap) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&emap) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&wmap) : "memory");
  }
  if (warp == kMmaWarp) tmem_alloc_pair(tmem_slot, kTmemCols);
  tc_fence_before();
  cluster.sync();  // both CTAs' barriers initialised and tensor memory allocated
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto aborted = [&]() { return *(volatile unsigned int*)abort_flag != 0u; };
  auto fail = [&]() {
    atomicOr(&g_tc_errors, 1u);
    atomicOr(abort_flag, 1u);
    atomicOr(cluster.map_shared_rank(abort_flag, rank ^ 1u), 1u);
  };
  auto stage_free = [&](int it) {  // wait until the MMAs of the stage's previous use are done
    return it < STAGES ||
           mbar_wait_bounded(&empty[it % STAGES], static_cast<uint32_t>(it / STAGES - 1) & 1u, kTcWaitNs);
  };

  const int wg = warp >> 2;  // each role's register budget is set at the top of its branch
  if (wg == 3) {
   asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtlRegs));
   if (warp == kTmaWarp) {
    if (lane == 0) {
      // the token tiles and the min-term tiles are the pre-pass's output (the weights' raw
      // super-blocks and their unpacking are not, so those roles start at once)
      asm volatile("griddepcontrol.wait;" ::: "memory");
      int it = 0;
      bool stop = false;
      for (int tile = pair; tile < p.tiles && !stop; tile += npairs) {
        const int m0 = (tile % p.m_tiles) * TN + static_cast<int>(rank) * (TN / 2);
        const int n0 = (tile / p.m_tiles) * (2 * TM) + static_cast<int>(rank) * TM;
        for (int kt = 0; kt < kt_tile; ++kt) {
          const int s = it % STAGES;
          if (!stage_free(it)) { fail(); stop = true; break; }
          if (aborted()) { stop = true; break; }
          uint8_t* st = smem + s * kStageBytes;
          const uint32_t fb = cluster_addr(&full_x[s], 0);
          if (kt < p.n_ext) {  // min-term tile: the tokens' sums and W's -64*dmin*m, both by TMA
            if (leader) mbar_arrive_expect_tx(&full_x[s], 2 * (kXTileBytes + kWTileBytes));
            tma_load_2d_pair(st + kWTileBytes, &xmap, p.K + kt * BK, m0, fb);
            tma_load_2d_pair(st, &emap, kt * BK, n0, fb);
          } else {
            if (leader) mbar_arrive_expect_tx(&full_x[s], 2 * kXTileBytes);
            tma_load_2d_pair(st + kWTileBytes, &xmap, (kt - p.n_ext) * BK, m0, fb);
          }
          ++it;
        }
      }
    }
  } else if (warp == kMmaWarp) {
    if (leader && lane == 0) {
      int it = 0, grp = 0;
      bool stop = false;
      for (int tile = pair; tile < p.tiles && !stop; tile += npairs) {
        for (int g = 0; g <= nsb && !stop; ++g, ++grp) {  // group 0: min term; 1..nsb: super-blocks
          const int buf = grp & 1;
          if (grp >= 2 &&
              !mbar_wait_bounded(&acc_empty[buf], static_cast<uint32_t>(grp / 2 - 1) & 1u, kTcWaitNs)) {
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
              umma_pair_f16(tmem + (uint32_t)(buf * TN), smem_desc_sw128(wa + 32 * kk),
                            smem_desc_sw128(xa + 32 * kk), (kt != kt0 || kk != 0) ? 1u : 0u);
            umma_commit_pair(&empty[s]);
            ++it;
          }
          if (!stop) umma_commit_pair(&acc_full[buf]);
        }
      }
      umma_commit_pair(mma_done);  // the wait point for every MMA this thread issued
      if (!mbar_wait_bounded(mma_done, 0u, kTcWaitNs)) fail();
    } else if (!leader && lane == 0) {
      // forwarder: passes on, in order, each stage's "t written" and each group's "read out"
      // (polling both sequences, so neither waits behind the other)
      const int my_tiles = pair < p.tiles ? (p.tiles - 1 - pair) / npairs + 1 : 0;
      const int ns = my_tiles * kt_tile, ng = my_tiles * (nsb + 1);
      int i = 0, j = 0;
      uint64_t t_last = globaltimer_ns();
      while (i < ns || j < ng) {
        bool moved = false;
        if (i < ns && mbar_test_wait(&full_w[i % STAGES], static_cast<uint32_t>(i / STAGES) & 1u)) {
          mbar_arrive_remote(cluster_addr(&full_w[i % STAGES], 0));
          ++i;
          moved = true;
        }
        if (j < ng && mbar_test_wait(&acc_empty[j & 1], static_cast<uint32_t>(j >> 1) & 1u)) {
          mbar_arrive_remote(cluster_addr(&acc_empty[j & 1], 0));
          ++j;
          moved = true;
        }
        if (moved) {
          t_last = globaltimer_ns();
        } else if (aborted()) {
          break;
        } else if (globaltimer_ns() - t_last > kTcWaitNs) {
          fail();
          break;
        }
      }
    }
   }
  } else if (wg == 2) {  // warps 8..11: unpack t = sc*q, whole k-tiles (all 128 rows) in turn
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kDqRegs));
    const int dw = warp - kDqBase;
    // raw super-blocks in the order they are unpacked: item i = super-block i % nsb of the
    // (i / nsb)-th tile of this pair
    auto raw_issue = [&](int item) {
      const int k = item / nsb, g = item - k * nsb;
      const int tile = pair + k * npairs;
      if (tile >= p.tiles) return;
      const int n0 = (tile / p.m_tiles) * (2 * TM) + static_cast<int>(rank) * TM;
      uint64_t* b = &raw_full[item % RAW_STAGES];
      mbar_arrive_expect_tx(b, kRawBytes);
      tma_load_2d(raw + (item % RAW_STAGES) * kRawBytes, &wmap, g * 36, n0, b);  // 36 words = 144 bytes
    };
    if (dw == 0 && lane == 0)
      for (int i = 0; i < RAW_STAGES; ++i) raw_issue(i);
    const int my_tiles = pair < p.tiles ? (p.tiles - 1 - pair) / npairs + 1 : 0;
    const int total = my_tiles * kt_tile;
    for (int it = dw; it < total; it += kDqWarps) {
      const int tk = it / kt_tile, kt = it - tk * kt_tile;
      const int s = it % STAGES;
      const int km = kt - p.n_ext;  // main k-tile index, < 0 for min-term tiles
      const int q = km >= 0 ? tk * nsb + (km >> 2) : 0;  // its raw super-block
      const int slot = q % RAW_STAGES;
      const uint32_t rpar = static_cast<uint32_t>(q / RAW_STAGES) & 1u;
      // every lane waits; the outcome is made warp-uniform so that no lane leaves the loop alone
      // (a lane that left would strand the others at the __syncwarp below)
      bool ok = km < 0 || mbar_wait_bounded(&raw_full[slot], rpar, kTcWaitNs);
      ok = ok && stage_free(it);
      if (!__all_sync(0xFFFFFFFFu, ok)) {
        if (lane == 0) fail();
        break;
      }
      if (__any_sync(0xFFFFFFFFu, aborted())) break;
      if (km >= 0) {
        uint8_t* wt = smem + s * kStageBytes;
        const uint8_t* rs = raw + slot * kRawBytes;
#pragma unroll 1
        for (int r = lane; r < TM; r += 32) unpack_row(rs, r, km & 3, wt);
        fence_proxy_async_smem();  // generic-proxy smem writes -> visible to the tensor core
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_local(&full_w[s]);
        if (km >= 0) {
          mbar_arrive_local(&raw_empty[slot]);
          if ((km & 3) == 3) {  // the super-block's last k-tile: refill the slot once all four are done
            if (!mbar_wait_bounded(&raw_empty[slot], rpar, kTcWaitNs)) {
              fail();
            } else {
              fence_proxy_async_smem();
              raw_issue(q + RAW_STAGES);
            }
          }
        }
      }
    }
  } else {  // warps 0..7: epilogue
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kEpiRegs));
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the tokens' 2^-e_j are the pre-pass's
    const int quarter = warp & 3, half = warp >> 2;
    int grp = 0;
    bool stop = false;
    for (int tile = pair; tile < p.tiles && !stop; tile += npairs) {
      // tensor-memory column c holds token m0 + c (rank 0's tokens, then rank 1's)
      const int m0 = (tile % p.m_tiles) * TN;
      const int n = (tile / p.m_tiles) * (2 * TM) + static_cast<int>(rank) * TM + quarter * 32 + lane;
      const uint8_t* rowp = p.w + (long long)min(n, p.N - 1) * p.row_bytes;
      float acc[TN / 2];
#pragma unroll
      for (int c = 0; c < TN / 2; ++c) acc[c] = 0.f;
      // this warp's tokens' 2^-e_j, fetched now (their latency hides behind the first group)
      // and read back from shared memory by the stores at the end of the tile
      float* winv = inv_base + warp * (TN / 2);
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
        if (lane == 0) mbar_arrive_local(&acc_empty[buf]);
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
  // After an abort, copies issued before it may still be landing (their byte counts go to
  // rank 0's barriers): give them time before either CTA can exit.
  if (threadIdx.x == 0 && aborted()) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 200000ull) {
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster.sync();  // no remote arrival or MMA operand read is still aimed at either CTA
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
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
// 128 threads per CTA (registers bound the CTAs per SM): about twice as many rows convert at
// once as with 256, the grid in ~1.5 waves instead of ~2.7 at the prefill shape
constexpr int kPrepThreads = 128;
__global__ void __launch_bounds__(kPrepThreads) prefill_prep_kernel(const uint16_t* __restrict__ x, __half* __restrict__ xc,
                                                           float* __restrict__ inv_scale, const uint8_t* __restrict__ w,
                                                           __half* __restrict__ wext, int M, int N, int K, int kc_x,
                                                           int k_ext, long long row_bytes) {
  // the GEMM that follows may launch now: it waits for this grid before it reads what it wrote
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int G = K / 32;
  if ((int)blockIdx.x < M) {
    __shared__ unsigned int smax;
    const int tok = blockIdx.x, nch = K / 8;  // 16-byte chunks of the row; 4 per sub-block
    if (threadIdx.x == 0) smax = 0u;
    __syncthreads();
    const uint16_t* xr = x + (long long)tok * K;
    // the first kKeep chunks of each thread stay in registers for the conversion pass (every
    // row up to K = 4096 is read once); the rest, if any, are read again there
    constexpr int kKeep = 4;
    uint4 keep[kKeep];
#pragma unroll
    for (int r = 0; r < kKeep; ++r) {
      const int c = threadIdx.x + kPrepThreads * r;
      keep[r] = c < nch ? ldg128(xr + 8 * c) : make_uint4(0u, 0u, 0u, 0u);
    }
    unsigned int best = 0u;
#pragma unroll
    for (int r = 0; r < kKeep; ++r) {
      const uint32_t wv[4] = {keep[r].x, keep[r].y, keep[r].z, keep[r].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) best = max(best, max((wv[i] & 0x7FFFu) << 16, wv[i] & 0x7FFF0000u));
    }
    for (int c = threadIdx.x + kPrepThreads * kKeep; c < nch; c += kPrepThreads) {
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
    for (int base = 0; base < nch; base += kPrepThreads) {
      const int c = base + threadIdx.x;
      float s = 0.f;
      if (c < nch) {
        uint4 v;
        if (base < kPrepThreads * kKeep) {
#pragma unroll
          for (int r = 0; r < kKeep; ++r)
            if (base == kPrepThreads * r) v = keep[r];
        } else {
          v = ldg128(xr + 8 * c);
        }
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
    for (int i = K + 3 * G + threadIdx.x; i < kc_x; i += kPrepThreads) xo[i] = __ushort_as_half(0);
  } else {
    const int nsb = K / 256;
    const long long idx = (long long)(blockIdx.x - M) * kPrepThreads + threadIdx.x;
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

// Q4_K weight rows as a 2-D tensor of 4-byte words (rows of row_bytes), 36-word (one
// super-block) x TM-row boxes, no swizzle: the raw stages the unpacking warps read.
int encode_raw_w(CUtensorMap* map, const void* w, int N, long long row_bytes, std::string* err) {
  void* fp = nullptr;
  cudaDriverEntryPointQueryResult qr;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fp, 12000, cudaEnableDefault, &qr) != cudaSuccess ||
      qr != cudaDriverEntryPointSuccess) {
    *err = "cuTensorMapEncodeTiled is unavailable";
    return -1;
  }
  EncodeTiledFn enc = reinterpret_cast<EncodeTiledFn>(fp);
  const cuuint64_t gdim[2] = {(cuuint64_t)(row_bytes / 4), (cuuint64_t)N};
  const cuuint64_t gstride[1] = {(cuuint64_t)row_bytes};
  const cuuint32_t box[2] = {36u, (cuuint32_t)TM};
  const cuuint32_t es[2] = {1u, 1u};
  const CUresult cr = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(w), gdim, gstride, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) {
    *err = "cuTensorMapEncodeTiled failed for the weights (" + std::to_string((int)cr) + ")";
    return -1;
  }
  return 0;
}

// Co-resident pairs of the prefill kernel (clusters of two CTAs at kTcSmem each), per device.
int max_pairs(int num_sms) {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return num_sms / 2;
  if (cache[dev] > 0) return cache[dev];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kTcThreads, 1, 1);
  cfg.dynamicSmemBytes = kTcSmem;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemm_q4k_tc_kernel, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return num_sms / 2;
  }
  cache[dev] = n;
  return n;
}

}  // namespace

size_t gemm_tc_workspace(int M, int N, int K) { return tc_layout(M, N, K).bytes; }

int launch_gemm_tc(const void* w, const void* x, float* y, int M, int N, int K, long long row_bytes, void* ws,
                   int num_sms, cudaStream_t stream, std::string* err) {
  const TcLayout L = tc_layout(M, N, K);
  const long long m_tiles = (M + TN - 1) / TN, n_tiles = (N + 2 * TM - 1) / (2 * TM);
  if (m_tiles * n_tiles > 0x7FFFFFFFLL) { *err = "M x N has too many output tiles"; return -1; }
  const long long prep_w_blocks = ((long long)N * (K / 256) + kPrepThreads - 1) / kPrepThreads;
  if ((long long)M + prep_w_blocks > 0x7FFFFFFFLL) { *err = "M and N too large for the pre-pass grid"; return -1; }
  uint8_t* base = static_cast<uint8_t*>(ws);
  __half* xc = reinterpret_cast<__half*>(base);
  float* inv = reinterpret_cast<float*>(base + L.off_inv);
  __half* wext = reinterpret_cast<__half*>(base + L.off_wext);
  prefill_prep_kernel<<<(unsigned)(M + prep_w_blocks), kPrepThreads, 0, stream>>>(
      static_cast<const uint16_t*>(x), xc, inv, static_cast<const uint8_t*>(w), wext, M, N, K, L.kc_x, L.k_ext,
      row_bytes);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) { *err = std::string("prefill pre-pass launch: ") + cudaGetErrorString(e); return -1; }
  CUtensorMap xmap, emap, wmap;
  if (encode_f16_2d(&xmap, xc, L.kc_x, M, TN / 2, err) || encode_f16_2d(&emap, wext, L.k_ext, N, TM, err) ||
      encode_raw_w(&wmap, w, N, row_bytes, err))
    return -1;
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64 || !attr_done[dev]) {
    e = cudaFuncSetAttribute(gemm_q4k_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
    if (e != cudaSuccess) { *err = std::string("cudaFuncSetAttribute (gemm): ") + cudaGetErrorString(e); return -1; }
    // the warpgroups' register budgets add up to exactly 512 threads x kLaunchRegs: a build
    // that starts the CTA with fewer registers would leave the epilogue's increase waiting forever
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, gemm_q4k_tc_kernel);
    if (e != cudaSuccess) { *err = std::string("cudaFuncGetAttributes (gemm): ") + cudaGetErrorString(e); return -1; }
    if (fa.numRegs != kLaunchRegs) {
      *err = "internal: the prefill kernel was built with " + std::to_string(fa.numRegs) + " registers per thread, not " +
             std::to_string(kLaunchRegs);
      return -1;
    }
    if (dev < 64) attr_done[dev] = true;
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
  const int pairs = (int)std::min<long long>(prm.tiles, max_pairs(num_sms));
  // programmatic dependent launch: the CTAs start (tensor memory, barriers, the weights' raw
  // copies and their unpacking) while the pre-pass drains; the copies of its output wait for it
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(kTcThreads, 1, 1);
  cfg.dynamicSmemBytes = kTcSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, gemm_q4k_tc_kernel, xmap, emap, wmap, prm);
  if (e == cudaSuccess) e = cudaGetLastError();
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
