// Fused block-diagonal transform + token reduction (tcgen05), for 128-wide
// super-blocks (b <= 128).
//
// For a row-major activation A (T x d), the super-block matrices S_s
// (rows = output features, K-major) and a second activation C (T x d):
//   out[:, s]  = A[:, s] S_s^T                       (block transform)
//   G[slot][s] = sum over this CTA's tokens of A[:, s]^T C[:, s]   (reduction)
// The backward pass uses it twice: (A, C) = (dz, h) gives dh and the R-side
// generator reduction, (A, C) = (dv, u) gives du and the P-side one.  Each
// token tile of A is staged in shared memory once and feeds both MMA chains
// (K-major view for the transform, MN-major view for the reduction), so the
// separate reduction pass and its second read of A disappear.
//
// CTA b works on super-block s = b % nsb and token tiles slot, slot + nslots,
// ... with slot = b / nsb, nslots = gridDim.x / nsb; the reduction
// accumulates in TMEM over all its tiles and is written once as partial
// `slot` of super-block s (layout [slot][s][128][128] fp32).
// Warps: 0 TMA producer, 1 TMEM allocator + MMA issuer, 2..9 epilogue.
// Stage: A tile (128 tokens x 128 features) and C tile, each as two 64-column
// boxes with 128-byte swizzle: 64 KB, two stages.  The CTA's super-block
// matrix S_s (128 x 128, 32 KB) is loaded once; the output is staged in two
// alternating 32 KB tiles, so a tile's store need not finish reading before
// the next tile is staged.
#pragma once

#include "ptx.cuh"

namespace poetx {

struct BdgrArgs {
  int M;          // tokens
  int N;          // features d
  int nsb;        // super-blocks
  int nslots;     // CTAs per super-block
  int b;          // block size (32, 64 or 128): only the b x b diagonal blocks of a partial are written
  float* partial; // [nslots][nsb][128][128]
  uint64_t timeout_ns;
};

struct BdgrCfg {
  static constexpr int BOX = 128 * 64 * 2;  // 16 KB
  static constexpr int TILE = 2 * BOX;      // 32 KB (128 x 128 bf16)
  static constexpr int STAGE = 2 * TILE;    // A, C
  static constexpr int STAGES = 2;
  static constexpr int OUT = 2 * TILE;      // two bf16 output staging tiles
  static constexpr int SMEM = 1024 + STAGES * STAGE + TILE /* S */ + OUT + 256;
  static_assert(SMEM <= 232448, "shared memory");
};

__global__ void __launch_bounds__(320, 1)
    tc_bdgr_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmS,
                   const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmOut,
                   const BdgrArgs args) {
  using Cfg = BdgrCfg;
  constexpr int STAGES = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned by pointer arithmetic on the shared array, so that the
  // compiler keeps shared-memory instructions for the accesses through it
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* s_tile = smem + STAGES * Cfg::STAGE;
  uint8_t* out_stage = s_tile + Cfg::TILE;
  uint64_t* full = reinterpret_cast<uint64_t*>(out_stage + Cfg::OUT);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* gdone = tempty + 2;
  uint64_t* sfull = gdone + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sfull + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint64_t tmo = args.timeout_ns;
  const int s = blockIdx.x % args.nsb;
  const int slot = blockIdx.x / args.nsb;
  const int mtiles = (args.M + 127) / 128;
  const int ntiles = (mtiles > slot) ? (mtiles - slot + args.nslots - 1) / args.nslots : 0;
  const int f0 = s * 128;  // first feature of the super-block

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 256);
    }
    mbar_init(gdone, 1);
    mbar_init(sfull, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmS);
    tma_prefetch_desc(&tmC);
    tma_prefetch_desc(&tmOut);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);  // [0,256): transform accumulators x2, [256,384): reduction
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  griddep_enter();

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      mbar_arrive_expect_tx(sfull, Cfg::TILE);
      tma_load_2d(s_tile, &tmS, sfull, 0, f0);
      tma_load_2d(s_tile + Cfg::BOX, &tmS, sfull, 64, f0);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_phase[STAGES] = {0, 0};
      bool issued[STAGES] = {false, false};
      for (int i = 0; i < ntiles; ++i) {
        const int m0 = (slot + i * args.nslots) * 128;
        if (!mbar_wait(&empty[stage], phase ^ 1u, tmo, abort_flag)) break;
        uint8_t* sa = smem + stage * Cfg::STAGE;
        uint8_t* sc = sa + Cfg::TILE;
        mbar_arrive_expect_tx(&full[stage], Cfg::STAGE);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          tma_load_2d(sa + h * Cfg::BOX, &tmA, &full[stage], f0 + 64 * h, m0);
          tma_load_2d(sc + h * Cfg::BOX, &tmC, &full[stage], f0 + 64 * h, m0);
        }
        issued[stage] = true;
        issued_phase[stage] = phase;
        if (++stage == STAGES) stage = 0, phase ^= 1u;
      }
      volatile int never = 0;
      for (int i = 0; i < STAGES; ++i)
        if (issued[i]) mbar_wait(&full[i], issued_phase[i], tmo, &never);
      mbar_wait(sfull, 0, tmo, &never);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t idesc_t = idesc_bf16_f32(128, 128, false, false);  // A S^T
      constexpr uint32_t idesc_g = idesc_bf16_f32(128, 128, true, true);    // A^T C
      const uint32_t d_g = tmem_base + 256;
      const uint32_t ss = smem_u32(s_tile);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = ntiles == 0 || mbar_wait(sfull, 0, tmo, abort_flag);
      for (int i = 0; i < ntiles && ok; ++i) {
        const int acc = i & 1;
        const uint32_t acc_phase = (i >> 1) & 1;
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, tmo, abort_flag)) break;
        if (!mbar_wait(&full[stage], phase, tmo, abort_flag)) break;
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + stage * Cfg::STAGE);
        const uint32_t sc = sa + Cfg::TILE;
        const uint32_t d_t = tmem_base + acc * 128;
        // transform: K = 128 input features, 8 steps of 16 (two 64-wide boxes)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * Cfg::BOX + (kk & 3) * 32;
          mma_bf16_f32(d_t, smem_desc_sw128(sa + off, 16, 1024), smem_desc_sw128(ss + off, 16, 1024),
                       idesc_t, kk != 0 ? 1u : 0u);
        }
        // reduction: K = 128 tokens, 8 steps of 16 rows; M = N = 128 features as
        // two 64-wide chunks one box apart
#pragma unroll
        for (int kt = 0; kt < 8; ++kt) {
          const uint32_t off = kt * 16 * 128;
          mma_bf16_f32(d_g, smem_desc_sw128(sa + off, Cfg::BOX, 1024),
                       smem_desc_sw128(sc + off, Cfg::BOX, 1024), idesc_g,
                       (i | kt) != 0 ? 1u : 0u);
        }
        mma_commit(&empty[stage]);
        mma_commit(&tfull[acc]);
        if (++stage == STAGES) stage = 0, phase ^= 1u;
      }
      mma_commit(gdone);  // the reduction accumulator is complete
      volatile int never = 0;
      mbar_wait(gdone, 0, tmo, &never);
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int g = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row = g * 32 + lane;
    const bool leader = (warp == 2 && lane == 0);
    for (int i = 0; i < ntiles; ++i) {
      const int m0 = (slot + i * args.nslots) * 128;
      const int acc = i & 1;
      const uint32_t acc_phase = (i >> 1) & 1;
      const bool waited = mbar_wait(&tfull[acc], acc_phase, tmo, abort_flag);
      // leave together: the named barriers below have no deadline
      if (named_barrier_any(1, 256, !waited)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + acc * 128 + half * 64 + (static_cast<uint32_t>(g * 32) << 16);
      uint32_t r[2][32];
      tmem_ld_32x32b_x32(taddr, r[0]);
      tmem_ld_32x32b_x32(taddr + 32, r[1]);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      // the store from this staging tile, two tiles back, must have read it
      if (leader) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
      named_barrier(1, 256);
      uint8_t* ostage = out_stage + (i & 1) * Cfg::TILE;
      uint8_t* box = ostage + half * Cfg::BOX;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const uint32_t* src = r[q >> 2] + (q & 3) * 8;
        uint4 v;
        v.x = pack_bf16x2(__uint_as_float(src[0]), __uint_as_float(src[1]));
        v.y = pack_bf16x2(__uint_as_float(src[2]), __uint_as_float(src[3]));
        v.z = pack_bf16x2(__uint_as_float(src[4]), __uint_as_float(src[5]));
        v.w = pack_bf16x2(__uint_as_float(src[6]), __uint_as_float(src[7]));
        *reinterpret_cast<uint4*>(box + row * 128 + ((q ^ (row & 7)) << 4)) = v;
      }
      fence_proxy_async_smem();
      named_barrier(1, 256);
      if (leader) {
        tma_store_2d(&tmOut, ostage, f0, m0);
        if (f0 + 64 < args.N) tma_store_2d(&tmOut, ostage + Cfg::BOX, f0 + 64, m0);
        bulk_commit();
      }
    }
    if (leader) bulk_wait_all();
    // reduction partial of this CTA: rows = features of A, columns = of C
    const bool have = (ntiles > 0) && mbar_wait(gdone, 0, tmo, abort_flag);
    if (have) tc_fence_after();
    float* out = args.partial +
                 (static_cast<int64_t>(slot) * args.nsb + s) * 128 * 128 + static_cast<int64_t>(row) * 128;
#pragma unroll 1
    for (int c = 0; c < 2; ++c) {
      const int col = half * 64 + c * 32;
      // the reduction is read only on the diagonal b x b blocks (one block
      // per warp's 32 rows, b >= 32): other column chunks are skipped
      if (col / args.b != row / args.b) continue;
      uint32_t r[32];
      if (ntiles > 0) {
        tmem_ld_32x32b_x32(tmem_base + 256 + col + (static_cast<uint32_t>(g * 32) << 16), r);
        tmem_ld_wait();
      }
      if (!have) {
#pragma unroll
        for (int q = 0; q < 32; ++q) r[q] = 0u;
      }
#pragma unroll
      for (int q = 0; q < 8; ++q)
        reinterpret_cast<uint4*>(out + col)[q] = make_uint4(r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

}  // namespace poetx
