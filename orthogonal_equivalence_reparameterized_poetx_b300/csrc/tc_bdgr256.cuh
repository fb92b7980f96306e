// Fused block-diagonal transform + token reduction (tcgen05) for 256-wide
// super-blocks (b = 256), the counterpart of tc_bdgr.cuh.
//
// For a row-major activation A (T x d), the super-block matrices S_s (256 x
// 256, rows = output features, K-major) and a second activation C (T x d):
//   out[:, s] = A[:, s] S_s^T                        (block transform)
//   G[slot][s] = sum over this CTA's tokens of A[:, s]^T C[:, s]  (reduction)
// CTA b works on super-block s, half r of its 256 features and token tiles
// slot, slot + nslots, ... of 64 tokens: (s, r, slot) = (b / 2 % nsb, b % 2,
// b / (2 nsb)).  It computes
//   out[:, s][:, 128r .. 128r+127] = A[:, s] (rows 128r.. of S_s)^T
//     as a transposed MMA: D (128 output features x 64 tokens) = S_half A_tile^T
//   G rows 128r .. 128r+127 (all 256 columns) += A[:, s half r]^T C[:, s]
// keeping its half of S_s resident in TMEM (loaded once, the A operand of the
// transform MMAs, so no shared-memory operand traffic for it) and its
// 128 x 256 reduction rows in TMEM for all its tiles; the rows are written
// once as partial `slot` (layout [slot][s][256][256] fp32).
// Warps: 0 TMA producer, 1 TMEM allocator + MMA issuer, 2..9 S loader, then
// epilogue.
// Stage: A tile and C tile, 64 tokens x 256 features each as four 64-feature
// boxes with 128-byte swizzle (2 x 32 KB); three stages, plus a 16 KB output
// tile.  TMEM: [0, 256) reduction, [256, 384) two transform accumulators,
// [384, 512) the S half (row f in lane f, features 2c, 2c + 1 in column c).
#pragma once

#include "ptx.cuh"

namespace poetx {

struct Bdgr256Args {
  int M;          // tokens
  int N;          // features d
  int nsb;        // 256-wide super-blocks
  int nslots;     // CTAs per (super-block, half)
  float* partial; // [nslots][nsb][256][256]
  const __nv_bfloat16* S;  // super-block matrices: nsb * 256 rows of 256
  uint64_t timeout_ns;
};

struct Bdgr256Cfg {
  static constexpr int TBOX = 64 * 64 * 2;     // 64 tokens x 64 features: 8 KB
  static constexpr int TILE = 4 * TBOX;        // 64 tokens x 256 features: 32 KB
  static constexpr int STAGE = 2 * TILE;       // A and C
  static constexpr int STAGES = 3;
  static constexpr int OUT = 2 * TBOX;         // 64 tokens x 128 features: 16 KB
  static constexpr int SMEM = 1024 + STAGES * STAGE + OUT + 256;
  static_assert(SMEM <= 232448, "shared memory");
};

__global__ void __launch_bounds__(320, 1)
    tc_bdgr256_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmC,
                      const __grid_constant__ CUtensorMap tmOut, const Bdgr256Args args) {
  using Cfg = Bdgr256Cfg;
  constexpr int STAGES = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned by pointer arithmetic on the shared array, so that the
  // compiler keeps shared-memory instructions for the accesses through it
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* stages = smem;
  uint8_t* out_stage = stages + STAGES * Cfg::STAGE;
  uint64_t* full = reinterpret_cast<uint64_t*>(out_stage + Cfg::OUT);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* sfull = tempty + 2;
  uint64_t* gdone = sfull + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gdone + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint64_t tmo = args.timeout_ns;
  const int r = blockIdx.x % 2;
  const int s = (blockIdx.x / 2) % args.nsb;
  const int slot = blockIdx.x / (2 * args.nsb);
  const int mtiles = (args.M + 63) / 64;
  const int ntiles = (mtiles > slot) ? (mtiles - slot + args.nslots - 1) / args.nslots : 0;
  const int f0 = s * 256;  // first feature of the super-block

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 256);
    }
    mbar_init(sfull, 256);  // the S loader threads
    mbar_init(gdone, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmC);
    tma_prefetch_desc(&tmOut);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);  // [0,256): reduction rows, [256,384): transform x2
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
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_phase[STAGES];
      bool issued[STAGES];
      for (int i = 0; i < STAGES; ++i) issued[i] = false, issued_phase[i] = 0;
      for (int i = 0; i < ntiles; ++i) {
        const int m0 = (slot + i * args.nslots) * 64;
        if (!mbar_wait(&empty[stage], phase ^ 1u, tmo, abort_flag)) break;
        uint8_t* sa = stages + stage * Cfg::STAGE;
        uint8_t* sc = sa + Cfg::TILE;
        mbar_arrive_expect_tx(&full[stage], Cfg::STAGE);
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          tma_load_2d(sa + h * Cfg::TBOX, &tmA, &full[stage], f0 + 64 * h, m0);
          tma_load_2d(sc + h * Cfg::TBOX, &tmC, &full[stage], f0 + 64 * h, m0);
        }
        issued[stage] = true;
        issued_phase[stage] = phase;
        if (++stage == STAGES) stage = 0, phase ^= 1u;
      }
      volatile int never = 0;
      for (int i = 0; i < STAGES; ++i)
        if (issued[i]) mbar_wait(&full[i], issued_phase[i], tmo, &never);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      // transform: D (128 features x 64 tokens) = S_half (TMEM) x A_tile^T (K-major)
      constexpr uint32_t idesc_t = idesc_bf16_f32(128, 64, false, false);
      // reduction: G (128 features x 256 features) += A_half^T (MN-major) x C (MN-major)
      constexpr uint32_t idesc_g = idesc_bf16_f32(128, 256, true, true);
      const uint32_t d_g = tmem_base;
      const uint32_t s_tmem = tmem_base + 384;
      bool ok = ntiles == 0 || mbar_wait(sfull, 0, tmo, abort_flag);
      if (ok) tc_fence_after();
      int stage = 0;
      uint32_t phase = 0;
      for (int i = 0; i < ntiles && ok; ++i) {
        const int acc = i & 1;
        const uint32_t acc_phase = (i >> 1) & 1;
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, tmo, abort_flag)) break;
        if (!mbar_wait(&full[stage], phase, tmo, abort_flag)) break;
        tc_fence_after();
        const uint32_t sa = smem_u32(stages + stage * Cfg::STAGE);
        const uint32_t sc = sa + Cfg::TILE;
        const uint32_t d_t = tmem_base + 256 + acc * 64;
        // K = 256 features in 16 steps of 16 (four 64-wide boxes)
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
          const uint32_t kb = (kk >> 2) * Cfg::TBOX + (kk & 3) * 32;
          mma_bf16_f32_ta(d_t, s_tmem + 8 * kk, smem_desc_sw128(sa + kb, 16, 1024), idesc_t,
                          kk != 0 ? 1u : 0u);
        }
        // K = 64 tokens in 4 steps of 16 rows; A's 128 features are boxes
        // 2r, 2r + 1 (one box apart), C's 256 features are all four boxes
#pragma unroll
        for (int kt = 0; kt < 4; ++kt) {
          const uint32_t off = kt * 16 * 128;
          mma_bf16_f32(d_g, smem_desc_sw128(sa + 2 * r * Cfg::TBOX + off, Cfg::TBOX, 1024),
                       smem_desc_sw128(sc + off, Cfg::TBOX, 1024), idesc_g, (i | kt) != 0 ? 1u : 0u);
        }
        mma_commit(&empty[stage]);
        mma_commit(&tfull[acc]);
        if (++stage == STAGES) stage = 0, phase ^= 1u;
      }
      mma_commit(gdone);
      volatile int never = 0;
      mbar_wait(gdone, 0, tmo, &never);
    }
  } else {
    // -------------------------------------------------------------- epilogue
    // warp w reads TMEM lanes (features) 32 (w % 4) .. and token columns
    // 32 * half .. of the transform accumulator
    const int g = warp & 3;
    const int half = (warp - 2) >> 2;
    const int f = g * 32 + lane;  // output feature within the half
    const bool leader = (warp == 2 && lane == 0);
    if (ntiles > 0) {
      // S half into TMEM: this thread's row f (feature f0 + 128 r + f),
      // features [128 half, 128 half + 128) as 64 columns of two bf16
      const uint4* src = reinterpret_cast<const uint4*>(
          args.S + static_cast<int64_t>(f0 + 128 * r + f) * 256 + 128 * half);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t w[32];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 x = __ldg(src + 8 * c + u);
          w[4 * u] = x.x;
          w[4 * u + 1] = x.y;
          w[4 * u + 2] = x.z;
          w[4 * u + 3] = x.w;
        }
        tmem_st_32x32b_x32(tmem_base + 384 + 64 * half + 32 * c + (static_cast<uint32_t>(g * 32) << 16), w);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(sfull);
    }
    for (int i = 0; i < ntiles; ++i) {
      const int m0 = (slot + i * args.nslots) * 64;
      const int acc = i & 1;
      const uint32_t acc_phase = (i >> 1) & 1;
      const bool waited = mbar_wait(&tfull[acc], acc_phase, tmo, abort_flag);
      // leave together: the named barriers below have no deadline
      if (named_barrier_any(1, 256, !waited)) break;
      tc_fence_after();
      uint32_t v[32];
      tmem_ld_32x32b_x32(tmem_base + 256 + acc * 64 + half * 32 + (static_cast<uint32_t>(g * 32) << 16), v);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      if (leader) bulk_wait_read_all();
      named_barrier(1, 256);
      // output tile [64 tokens][128 features] as two 64-feature boxes with
      // 128-byte swizzle: feature f of token t at box f / 64, row t,
      // 16-byte chunk ((f % 64) / 8) ^ (t % 8), element f % 8
      uint8_t* box = out_stage + (f / 64) * Cfg::TBOX;
      const int fc = (f % 64) / 8, fe = f % 8;
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const int t = half * 32 + c;
        const __nv_bfloat16 bv = __float2bfloat16_rn(__uint_as_float(v[c]));
        *reinterpret_cast<__nv_bfloat16*>(box + t * 128 + ((fc ^ (t & 7)) << 4) + 2 * fe) = bv;
      }
      fence_proxy_async_smem();
      named_barrier(1, 256);
      if (leader) {  // boxes that start past the last feature (ragged d) are not stored
        const int x = f0 + 128 * r;
        if (x < args.N) tma_store_2d(&tmOut, out_stage, x, m0);
        if (x + 64 < args.N) tma_store_2d(&tmOut, out_stage + Cfg::TBOX, x + 64, m0);
        bulk_commit();
      }
    }
    if (leader) bulk_wait_all();
    // reduction rows 128 r + (g * 32 + lane), columns [0, 256): warp half
    // `half` writes columns 128 half .. 128 half + 127
    const bool have = (ntiles > 0) && mbar_wait(gdone, 0, tmo, abort_flag);
    if (have) tc_fence_after();
    float* out = args.partial + (static_cast<int64_t>(slot) * args.nsb + s) * 256 * 256 +
                 static_cast<int64_t>(128 * r + f) * 256;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      const int col = half * 128 + c * 32;
      uint32_t q[32];
      if (ntiles > 0) {
        tmem_ld_32x32b_x32(tmem_base + col + (static_cast<uint32_t>(g * 32) << 16), q);
        tmem_ld_wait();
      }
      if (!have) {
#pragma unroll
        for (int e = 0; e < 32; ++e) q[e] = 0u;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e)
        reinterpret_cast<uint4*>(out + col)[e] = make_uint4(q[4 * e], q[4 * e + 1], q[4 * e + 2], q[4 * e + 3]);
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
