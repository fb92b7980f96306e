// Backward dgrad GEMM with the P-side block work in its epilogue (blocks of
// at most 128, i.e. 128-wide super-blocks):
//   dv = dh W0'                  main loop, 128 x 128 tiles (B operand MN-major)
//   du[:, s] = dv[:, s] S_s^T    epilogue MMA 1 (S_s: super-block of B_P^T)
//   G[slot][s] += dv[:, s]^T u[:, s]   epilogue MMA 2, accumulated in TMEM
// over this CTA's token tiles ("POET-X: Memory-efficient LLM Training by
// Scaling Orthogonal Transformation", Methodologie §1 and §3).  dv never
// reaches HBM: each bf16 dv tile is staged in 128-byte-swizzled shared
// memory, where it is the K-major A operand of the transform and the MN-major
// A operand of the token reduction.
//
// CTA b owns output-feature tile (super-block) s = b % nsb and token tiles
// slot, slot + nslots, ... with slot = b / nsb (as the fused transform +
// reduction kernel does), so the reduction accumulates in TMEM and is
// written once as partial `slot` of super-block s ([slot][s][128][128] fp32;
// for blocks b < 128 only the b x b diagonal blocks are written).
// Warps: 0 TMA producer, 1 TMEM allocator and main-loop MMA issuer, 2..9
// epilogue; warp 2 lane 0 also issues the epilogue MMAs and the S_s and u
// loads.  TMEM: two 128-column accumulators, 128 columns for du, 128 for G.
// Every wait is bounded; after a timeout the CTA drains what it issued.
#pragma once

#include "ptx.cuh"

namespace poetx {

struct TcGemmPArgs {
  int M;          // tokens
  int N;          // output features (n)
  int K;          // contraction (m)
  int nsb;        // super-blocks of the P side
  int nslots;     // CTAs per super-block
  int b;          // block size (32, 64 or 128)
  float* partial; // [nslots][nsb][128][128]
  uint64_t timeout_ns;
};

struct TcGemmPCfg {
  static constexpr int BOX = 128 * 64 * 2;  // 128 rows x 64 bf16 (16 KB)
  static constexpr int STAGE = 2 * BOX;     // A box + two 64 x 64 B boxes
  static constexpr int STAGES = 4;
  static constexpr int TILE = 2 * BOX;      // 128 x 128 bf16
  static constexpr int SMEM = 1024 + STAGES * STAGE + 3 * TILE + 256;
  static_assert(SMEM <= 232448, "shared memory");
};

__global__ void __launch_bounds__(320, 1)
    tc_gemm_p_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmU,
                     const __grid_constant__ CUtensorMap tmDu, const TcGemmPArgs args) {
  using Cfg = TcGemmPCfg;
  constexpr int STAGES = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned by pointer arithmetic on the shared array
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* d_tile = smem + STAGES * Cfg::STAGE;  // dv, then du (bf16, swizzled)
  uint8_t* s_tile = d_tile + Cfg::TILE;          // S_s
  uint8_t* u_tile = s_tile + Cfg::TILE;          // u tile of the current token tile
  uint64_t* full = reinterpret_cast<uint64_t*>(u_tile + Cfg::TILE);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* s_full = drain + 1;
  uint64_t* u_full = s_full + 1;
  uint64_t* edone = u_full + 1;
  uint64_t* edrain = edone + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(edrain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint64_t tmo = args.timeout_ns;
  const int s = blockIdx.x % args.nsb;
  const int slot = blockIdx.x / args.nsb;
  const int mtiles = (args.M + 127) / 128;
  const int ntiles = (mtiles > slot) ? (mtiles - slot + args.nslots - 1) / args.nslots : 0;
  const int n0 = s * 128;
  const int nk = (args.K + 63) / 64;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 256);
    }
    mbar_init(drain, 1);
    mbar_init(s_full, 1);
    mbar_init(u_full, 1);
    mbar_init(edone, 1);
    mbar_init(edrain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmS);
    tma_prefetch_desc(&tmU);
    tma_prefetch_desc(&tmDu);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);  // [0, 256) accumulators, [256, 384) du, [384, 512) G
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  griddep_enter();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_phase[STAGES];
      bool issued[STAGES];
      for (int i = 0; i < STAGES; ++i) issued[i] = false, issued_phase[i] = 0;
      bool ok = true;
      for (int i = 0; i < ntiles && ok; ++i) {
        const int m0 = (slot + i * args.nslots) * 128;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, tmo, abort_flag)) { ok = false; break; }
          uint8_t* sa = smem + stage * Cfg::STAGE;
          uint8_t* sb = sa + Cfg::BOX;
          mbar_arrive_expect_tx(&full[stage], Cfg::STAGE);
          tma_load_2d(sa, &tmA, &full[stage], kb * 64, m0);
          tma_load_2d(sb, &tmB, &full[stage], n0, kb * 64);
          tma_load_2d(sb + 64 * 128, &tmB, &full[stage], n0 + 64, kb * 64);
          issued[stage] = true;
          issued_phase[stage] = phase;
          if (++stage == STAGES) stage = 0, phase ^= 1u;
        }
      }
      for (int i = 0; i < STAGES; ++i)
        if (issued[i]) {
          volatile int never = 0;
          mbar_wait(&full[i], issued_phase[i], tmo, &never);
        }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- main-loop MMAs
      constexpr uint32_t idesc = idesc_bf16_f32(128, 128, false, true);  // B MN-major
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int i = 0; i < ntiles && ok; ++i) {
        const int acc = i & 1;
        const uint32_t acc_phase = (i >> 1) & 1;
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, tmo, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * 128;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(&full[stage], phase, tmo, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * Cfg::STAGE);
          const uint32_t sb = sa + Cfg::BOX;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16_f32(d_tmem, smem_desc_sw128(sa + kk * 32, 16, 1024),
                         smem_desc_sw128(sb + kk * 2048, 64 * 128, 1024), idesc, (kb | kk) != 0 ? 1u : 0u);
          mma_commit(&empty[stage]);
          if (++stage == STAGES) stage = 0, phase ^= 1u;
        }
        if (!ok) break;
        mma_commit(&tfull[acc]);
      }
      mma_commit(drain);
      volatile int never = 0;
      mbar_wait(drain, 0, tmo, &never);
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int g = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row = g * 32 + lane;
    const bool leader = (warp == 2 && lane == 0);
    const uint32_t du_cols = tmem_base + 256, g_cols = tmem_base + 384;
    int u_loads = 0, u_landed = 0;  // leader's counts of u tile loads issued / waited for
    bool s_pending = false;
    auto load_u = [&](int i) {
      const int m0 = (slot + i * args.nslots) * 128;
      mbar_arrive_expect_tx(u_full, Cfg::TILE);
      tma_load_2d(u_tile, &tmU, u_full, n0, m0);
      tma_load_2d(u_tile + Cfg::BOX, &tmU, u_full, n0 + 64, m0);
      ++u_loads;
    };
    auto stage_bf16 = [&](const uint32_t (&r)[2][32]) {
      uint8_t* box = d_tile + half * Cfg::BOX;
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
    };
    if (leader && ntiles > 0) {
      mbar_arrive_expect_tx(s_full, Cfg::TILE);
      tma_load_2d(s_tile, &tmS, s_full, 0, n0);
      tma_load_2d(s_tile + Cfg::BOX, &tmS, s_full, 64, n0);
      s_pending = true;
      load_u(0);
    }
    int done = 0;  // tiles whose epilogue MMAs completed
    for (int i = 0; i < ntiles; ++i) {
      const int m0 = (slot + i * args.nslots) * 128;
      const int acc = i & 1;
      const uint32_t acc_phase = (i >> 1) & 1;
      const bool waited = mbar_wait(&tfull[acc], acc_phase, tmo, abort_flag);
      // leave together: the named barriers below have no deadline
      if (named_barrier_any(1, 256, !waited)) break;
      tc_fence_after();
      uint32_t r[2][32];
      const uint32_t col = tmem_base + acc * 128 + half * 64 + (static_cast<uint32_t>(g * 32) << 16);
      tmem_ld_32x32b_x32(col, r[0]);
      tmem_ld_32x32b_x32(col + 32, r[1]);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      if (leader) bulk_wait_read_all();  // the previous du store has read the tile
      named_barrier(1, 256);
      stage_bf16(r);
      fence_proxy_async_smem();
      named_barrier(1, 256);
      bool fail = false;
      if (leader) {
        if (s_pending) {
          fail = !mbar_wait(s_full, 0, tmo, abort_flag);
          if (!fail) s_pending = false;
        }
        if (!fail) {
          fail = !mbar_wait(u_full, static_cast<uint32_t>(i & 1), tmo, abort_flag);
          if (!fail) ++u_landed;
        }
        if (!fail) {
          tc_fence_after();
          const uint32_t sd = smem_u32(d_tile), ss = smem_u32(s_tile), su = smem_u32(u_tile);
          constexpr uint32_t idesc_t = idesc_bf16_f32(128, 128, false, false);  // dv S^T
          constexpr uint32_t idesc_g = idesc_bf16_f32(128, 128, true, true);    // dv^T u
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * Cfg::BOX + (kk & 3) * 32;
            mma_bf16_f32(du_cols, smem_desc_sw128(sd + off, 16, 1024), smem_desc_sw128(ss + off, 16, 1024),
                         idesc_t, kk != 0 ? 1u : 0u);
          }
#pragma unroll
          for (int kt = 0; kt < 8; ++kt) {
            const uint32_t off = kt * 16 * 128;
            mma_bf16_f32(g_cols, smem_desc_sw128(sd + off, Cfg::BOX, 1024),
                         smem_desc_sw128(su + off, Cfg::BOX, 1024), idesc_g, (i | kt) != 0 ? 1u : 0u);
          }
          mma_commit(edone);
        }
      }
      if (named_barrier_any(1, 256, fail)) break;
      const bool eok = mbar_wait(edone, static_cast<uint32_t>(i & 1), tmo, abort_flag);
      if (named_barrier_any(1, 256, !eok)) break;
      ++done;
      tc_fence_after();
      const uint32_t dc = du_cols + half * 64 + (static_cast<uint32_t>(g * 32) << 16);
      tmem_ld_32x32b_x32(dc, r[0]);
      tmem_ld_32x32b_x32(dc + 32, r[1]);
      tmem_ld_wait();
      tc_fence_before();
      if (leader && i + 1 < ntiles) load_u(i + 1);  // the reduction MMAs have read the u tile
      named_barrier(1, 256);  // every du value is in registers; the dv tile is free
      stage_bf16(r);
      fence_proxy_async_smem();
      named_barrier(1, 256);
      if (leader) {
        tma_store_2d(&tmDu, d_tile, n0, m0);
        if (n0 + 64 < args.N) tma_store_2d(&tmDu, d_tile + Cfg::BOX, n0 + 64, m0);
        bulk_commit();
      }
    }
    if (leader) bulk_wait_all();
    // reduction partial of this CTA (zeros when it had no tile or stopped
    // early); only the diagonal b x b blocks are read downstream
    const bool have = (ntiles > 0) && (done == ntiles);
    float* out = args.partial + (static_cast<int64_t>(slot) * args.nsb + s) * 128 * 128 +
                 static_cast<int64_t>(row) * 128;
#pragma unroll 1
    for (int c = 0; c < 2; ++c) {
      const int c0 = half * 64 + c * 32;
      if (c0 / args.b != row / args.b) continue;
      uint32_t r[32];
      if (have) {
        tmem_ld_32x32b_x32(g_cols + c0 + (static_cast<uint32_t>(g * 32) << 16), r);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int q = 0; q < 32; ++q) r[q] = 0u;
      }
#pragma unroll
      for (int q = 0; q < 8; ++q)
        reinterpret_cast<uint4*>(out + c0)[q] = make_uint4(r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
    }
    if (leader) {
      // every epilogue MMA is complete before TMEM is released, and loads
      // still in flight land before the CTA exits
      mma_commit(edrain);
      volatile int never = 0;
      mbar_wait(edrain, 0, tmo, &never);
      if (s_pending) mbar_wait(s_full, 0, tmo, &never);
      if (u_loads > u_landed) mbar_wait(u_full, static_cast<uint32_t>((u_loads - 1) & 1), tmo, &never);
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
