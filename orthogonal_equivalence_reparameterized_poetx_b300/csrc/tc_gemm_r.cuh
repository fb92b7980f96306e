// Forward GEMM with the R block transform in its epilogue (blocks of at most
// 128, i.e. 128-wide super-blocks):
//   h = v W0'^T                 main loop, 128 x 128 output tiles, full K
//   z[:, s] = h[:, s] S_s^T     epilogue: a second MMA on the bf16 h tile
// A 128-column output tile [n0, n0 + 128) is exactly super-block s = n0 / 128
// of the R side ("POET-X: Memory-efficient LLM Training by Scaling
// Orthogonal Transformation", Methodologie §1 and §3: the layer evaluated as
// maps on the input, the blocks as independent small matrices).  The h tile
// is rounded to bf16 and staged in 128-byte-swizzled shared memory; that
// buffer is both the TMA-store source of h (when the caller keeps h) and the
// K-major A operand of the transform MMA.  The super-block matrix S_s is
// loaded by TMA once per tile into its own buffer.  The separate pass that
// reads h back to form z disappears.
//
// Warps: 0 TMA producer, 1 TMEM allocator and main-loop MMA issuer, 2..9
// epilogue; warp 2 lane 0 also issues the transform MMAs and the S_s loads.
// TMEM: two 128-column accumulators for the main loop, 128 columns for z.
// Every wait is bounded; after a timeout the CTA drains what it issued.
#pragma once

#include "ptx.cuh"

namespace poetx {

struct TcGemmRArgs {
  int M;          // tokens
  int N;          // output features (m)
  int K;          // input features (n)
  int num_tiles;  // ceil(M / 128) * ceil(N / 128)
  int store_h;    // also write h
  uint64_t timeout_ns;
};

struct TcGemmRCfg {
  static constexpr int BOX = 128 * 64 * 2;  // 128 rows x 64 bf16 (16 KB)
  static constexpr int STAGE = 2 * BOX;     // A and B boxes of one 64-wide K step
  static constexpr int STAGES = 5;
  static constexpr int TILE = 2 * BOX;      // 128 x 128 bf16
  static constexpr int SMEM = 1024 + STAGES * STAGE + 2 * TILE + 256;
  static_assert(SMEM <= 232448, "shared memory");
};

__global__ void __launch_bounds__(320, 1)
    tc_gemm_r_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmH,
                     const __grid_constant__ CUtensorMap tmZ, const TcGemmRArgs args) {
  using Cfg = TcGemmRCfg;
  constexpr int STAGES = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned by pointer arithmetic on the shared array
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* hz_tile = smem + STAGES * Cfg::STAGE;  // h, then z (bf16, swizzled)
  uint8_t* s_tile = hz_tile + Cfg::TILE;          // S_s
  uint64_t* full = reinterpret_cast<uint64_t*>(s_tile + Cfg::TILE);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* s_full = drain + 1;
  uint64_t* zdone = s_full + 1;
  uint64_t* zdrain = zdone + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(zdrain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint64_t tmo = args.timeout_ns;
  const int ntn = (args.N + 127) / 128;
  const int nk = (args.K + 63) / 64;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 256);
    }
    mbar_init(drain, 1);
    mbar_init(s_full, 1);
    mbar_init(zdone, 1);
    mbar_init(zdrain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmS);
    tma_prefetch_desc(&tmH);
    tma_prefetch_desc(&tmZ);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);  // [0, 256): accumulators, [256, 384): z
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
      for (int s = 0; s < STAGES; ++s) issued[s] = false, issued_phase[s] = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < args.num_tiles && ok; tile += gridDim.x) {
        const int m0 = (tile / ntn) * 128, n0 = (tile % ntn) * 128;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, tmo, abort_flag)) { ok = false; break; }
          uint8_t* sa = smem + stage * Cfg::STAGE;
          mbar_arrive_expect_tx(&full[stage], Cfg::STAGE);
          tma_load_2d(sa, &tmA, &full[stage], kb * 64, m0);
          tma_load_2d(sa + Cfg::BOX, &tmB, &full[stage], kb * 64, n0);
          issued[stage] = true;
          issued_phase[stage] = phase;
          if (++stage == STAGES) stage = 0, phase ^= 1u;
        }
      }
      for (int s = 0; s < STAGES; ++s)
        if (issued[s]) {
          volatile int never = 0;
          mbar_wait(&full[s], issued_phase[s], tmo, &never);
        }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- main-loop MMAs
      constexpr uint32_t idesc = idesc_bf16_f32(128, 128, false, false);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < args.num_tiles && ok; tile += gridDim.x, ++it) {
        const int acc = it & 1;
        const uint32_t acc_phase = (it >> 1) & 1;
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
                         smem_desc_sw128(sb + kk * 32, 16, 1024), idesc, (kb | kk) != 0 ? 1u : 0u);
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
    const uint32_t zcols = tmem_base + 256;
    int s_loads = 0, s_landed = 0;  // leader's count of S_s loads issued / waited for
    auto load_s = [&](int tile) {
      const int n0 = (tile % ntn) * 128;
      mbar_arrive_expect_tx(s_full, Cfg::TILE);
      tma_load_2d(s_tile, &tmS, s_full, 0, n0);
      tma_load_2d(s_tile + Cfg::BOX, &tmS, s_full, 64, n0);
      ++s_loads;
    };
    // rounds a 64-column half-row of fp32 values to bf16 into the swizzled tile
    auto stage_bf16 = [&](const uint32_t (&r)[2][32]) {
      uint8_t* box = hz_tile + half * Cfg::BOX;
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
    if (leader && static_cast<int>(blockIdx.x) < args.num_tiles) load_s(blockIdx.x);
    int it = 0;
    for (int tile = blockIdx.x; tile < args.num_tiles; tile += gridDim.x, ++it) {
      const int m0 = (tile / ntn) * 128, n0 = (tile % ntn) * 128;
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      const bool waited = mbar_wait(&tfull[acc], acc_phase, tmo, abort_flag);
      // leave together: the named barriers below have no deadline
      if (named_barrier_any(1, 256, !waited)) break;
      tc_fence_after();
      uint32_t r[2][32];
      const uint32_t hcol = tmem_base + acc * 128 + half * 64 + (static_cast<uint32_t>(g * 32) << 16);
      tmem_ld_32x32b_x32(hcol, r[0]);
      tmem_ld_32x32b_x32(hcol + 32, r[1]);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      if (leader) bulk_wait_read_all();  // the previous tile's z store has read the tile
      named_barrier(1, 256);
      stage_bf16(r);
      fence_proxy_async_smem();
      named_barrier(1, 256);
      bool fail = false;
      if (leader) {
        if (args.store_h) {
          tma_store_2d(&tmH, hz_tile, n0, m0);
          if (n0 + 64 < args.N) tma_store_2d(&tmH, hz_tile + Cfg::BOX, n0 + 64, m0);
          bulk_commit();
        }
        fail = !mbar_wait(s_full, static_cast<uint32_t>(it & 1), tmo, abort_flag);
        if (!fail) {
          ++s_landed;
          tc_fence_after();
          constexpr uint32_t idesc_r = idesc_bf16_f32(128, 128, false, false);  // h S^T
          const uint32_t sa = smem_u32(hz_tile), ss = smem_u32(s_tile);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * Cfg::BOX + (kk & 3) * 32;
            mma_bf16_f32(zcols, smem_desc_sw128(sa + off, 16, 1024), smem_desc_sw128(ss + off, 16, 1024),
                         idesc_r, kk != 0 ? 1u : 0u);
          }
          mma_commit(zdone);
        }
      }
      if (named_barrier_any(1, 256, fail)) break;
      const bool zok = mbar_wait(zdone, static_cast<uint32_t>(it & 1), tmo, abort_flag);
      if (named_barrier_any(1, 256, !zok)) break;
      tc_fence_after();
      const uint32_t zc = zcols + half * 64 + (static_cast<uint32_t>(g * 32) << 16);
      tmem_ld_32x32b_x32(zc, r[0]);
      tmem_ld_32x32b_x32(zc + 32, r[1]);
      tmem_ld_wait();
      tc_fence_before();
      if (leader) {
        // the transform MMAs are complete: S_s of the next tile may land
        const int next = tile + static_cast<int>(gridDim.x);
        if (next < args.num_tiles) load_s(next);
        bulk_wait_read_all();  // the h store has read the tile
      }
      named_barrier(1, 256);   // every z value is in registers: the tile and z columns are free
      stage_bf16(r);
      fence_proxy_async_smem();
      named_barrier(1, 256);
      if (leader) {
        tma_store_2d(&tmZ, hz_tile, n0, m0);
        if (n0 + 64 < args.N) tma_store_2d(&tmZ, hz_tile + Cfg::BOX, n0 + 64, m0);
        bulk_commit();
      }
    }
    if (leader) {
      bulk_wait_all();
      // every transform MMA is complete before TMEM is released, and an S_s
      // load still in flight lands before the CTA exits
      mma_commit(zdrain);
      volatile int never = 0;
      mbar_wait(zdrain, 0, tmo, &never);
      if (s_loads > s_landed) mbar_wait(s_full, static_cast<uint32_t>((s_loads - 1) & 1), tmo, &never);
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
