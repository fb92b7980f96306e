// Forward GEMM on CTA pairs (tcgen05 .cta_group::2) with the R block
// transform in its epilogue (blocks of at most 128, i.e. 128-wide
// super-blocks):
//   h = v W0'^T                 main loop, 256 x 256 output tiles per pair
//   z[:, s] = h[:, s] S_s^T     epilogue: two more pair MMAs per tile, one for
//                               each of the tile's two super-blocks
// ("POET-X: Memory-efficient LLM Training by Scaling Orthogonal
// Transformation", Methodologie §1 and §3).  The main loop is the one of
// tc_gemm_pair_kernel with B K-major and five stages.  The epilogue runs the
// tile's two super-blocks in turn: each CTA rounds its 128 accumulator rows
// of one super-block of h to bf16 into a 128 x 128 swizzled shared tile,
// which is the TMA-store source of h (when h is kept) and, in both CTAs at
// the same offset, the A operand of the transform; each CTA also loads its
// 64-row half of both super-block matrices (the B operand split of an M =
// 256, N = 128 pair MMA).  The even CTA's epilogue leader issues the
// super-block's transform MMAs into its own accumulator columns (both CTAs
// have read h from them by then), so no TMEM beyond the two 256-column
// accumulators is needed; z goes out through the same shared tile, and the
// accumulator goes back to the main loop once both halves of z are read.
// Staging one super-block at a time (32 KB instead of 64) leaves room for
// the fifth main-loop stage.
//
// Warps (both CTAs): 0 TMA producer, 1 TMEM allocator (even CTA: main-loop
// MMA issuer), 2..9 epilogue.  Barriers beyond the pair GEMM's:
//   s_full    each CTA's: its super-block halves of the current tile landed
//   hstaged   even CTA's: both CTAs' h tiles are staged and S halves landed
//             (twice per tile, once per super-block)
//   zdone     each CTA's: a super-block's transform MMAs are complete
//             (multicast commit; twice per tile)
//   zdrain    even CTA's: every transform MMA is complete (before TMEM is freed)
// Every wait is bounded; on a timeout a CTA records it and winds down, and
// the pair meets at a cluster barrier before freeing TMEM and exiting.
#pragma once

#include "ptx.cuh"

namespace poetx {

struct TcPairRArgs {
  int M, N, K;
  int num_tiles;  // ceil(M / 256) * ceil(N / 256)
  int store_h;
  uint64_t timeout_ns;
};

struct TcPairRCfg {
  static constexpr int BOX = 128 * 64 * 2;     // 128 rows x 64 bf16 (16 KB)
  static constexpr int STAGE_BYTES = 2 * BOX;  // this CTA's A rows and B columns of one K step
  static constexpr int STAGES = 5;
  static constexpr int HZ_BYTES = 2 * BOX;     // 128 rows x 128 features (one super-block)
  static constexpr int SBOX = 64 * 64 * 2;     // 64 rows x 64 bf16 (8 KB)
  static constexpr int S_BYTES = 4 * SBOX;     // two super-blocks x (64 rows x 128)
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + HZ_BYTES + S_BYTES + 256;
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(320, 1)
    tc_gemm_pair_r_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                          const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmH,
                          const __grid_constant__ CUtensorMap tmZ, const TcPairRArgs args) {
  using Cfg = TcPairRCfg;
  constexpr int STAGES = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned by pointer arithmetic on the shared array
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* hz_tile = smem + STAGES * Cfg::STAGE_BYTES;
  uint8_t* s_tile = hz_tile + Cfg::HZ_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(s_tile + Cfg::S_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* s_full = drain + 1;
  uint64_t* hstaged = s_full + 1;
  uint64_t* zdone = hstaged + 1;
  uint64_t* zdrain = zdone + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(zdrain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs
  const int pair = blockIdx.x / 2, npairs = gridDim.x / 2;
  const int ntn = (args.N + 255) / 256;
  const int nk = (args.K + 63) / 64;
  const uint64_t tmo = args.timeout_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 512);
    }
    mbar_init(drain, 1);
    mbar_init(s_full, 1);
    mbar_init(hstaged, 2);
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
    tmem_alloc_pair(tmem_slot, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  // both CTAs' barriers are initialised before either CTA signals the other's
  cluster_sync();
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
      for (int tile = pair; tile < args.num_tiles && ok; tile += npairs) {
        const int m0 = (tile / ntn) * 256 + 128 * static_cast<int>(rank);
        const int nb = (tile % ntn) * 256 + 128 * static_cast<int>(rank);
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, tmo, abort_flag)) { ok = false; break; }
          uint8_t* sa = smem + stage * Cfg::STAGE_BYTES;
          const uint32_t fbar = dsmem_addr(&full[stage], 0);  // the even CTA's barrier
          if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * Cfg::STAGE_BYTES);
          tma_load_2d_pair(sa, &tmA, fbar, kb * 64, m0);
          tma_load_2d_pair(sa + Cfg::BOX, &tmB, fbar, kb * 64, nb);
          issued[stage] = true;
          issued_phase[stage] = phase;
          if (++stage == STAGES) stage = 0, phase ^= 1u;
        }
      }
      // this CTA's copies in flight land before the pair may exit: wait for
      // the matching empty phase (the MMAs that consumed them), bounded
      for (int s = 0; s < STAGES; ++s)
        if (issued[s]) {
          volatile int never = 0;
          mbar_wait(&empty[s], issued_phase[s], tmo, &never);
        }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------------------------------------------------- main-loop MMAs
      constexpr uint32_t idesc = idesc_bf16_f32(256, 256, false, false);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int tile = pair; tile < args.num_tiles && ok; tile += npairs, ++it) {
        const int acc = it & 1;
        const uint32_t acc_phase = (it >> 1) & 1;
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, tmo, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * 256;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(&full[stage], phase, tmo, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * Cfg::STAGE_BYTES);
          const uint32_t sb = sa + Cfg::BOX;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16_f32_pair(d_tmem, smem_desc_sw128(sa + kk * 32, 16, 1024),
                              smem_desc_sw128(sb + kk * 32, 16, 1024), idesc, (kb | kk) != 0 ? 1u : 0u);
          mma_commit_pair(&empty[stage], 0x3);
          if (++stage == STAGES) stage = 0, phase ^= 1u;
        }
        if (!ok) break;
        mma_commit_pair(&tfull[acc], 0x3);
      }
      mma_commit_pair(drain, 0x3);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int g = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row = g * 32 + lane;
    const bool leader = (warp == 2 && lane == 0);
    int s_loads = 0, s_landed = 0;  // leader's count of S loads issued / waited for
    auto load_s = [&](int tile) {
      const int n0 = (tile % ntn) * 256;
      mbar_arrive_expect_tx(s_full, Cfg::S_BYTES);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int r0 = n0 + j * 128 + 64 * static_cast<int>(rank);  // this CTA's 64 output features
        tma_load_2d(s_tile + (2 * j) * Cfg::SBOX, &tmS, s_full, 0, r0);
        tma_load_2d(s_tile + (2 * j + 1) * Cfg::SBOX, &tmS, s_full, 64, r0);
      }
      ++s_loads;
    };
    // fp32 accumulator columns [sl * 128 + half * 64, + 64) of this thread's row
    // to bf16 into box `half` of the swizzled tile
    auto tmem_to_tile = [&](uint32_t base, int sl) {
      uint32_t r[2][32];
      const uint32_t c = base + sl * 128 + half * 64;
      tmem_ld_32x32b_x32(c, r[0]);
      tmem_ld_32x32b_x32(c + 32, r[1]);
      tmem_ld_wait();
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
    // the staged super-block (features [x, x + 128)) to global memory
    auto store_tile = [&](const CUtensorMap* map, int x, int m0) {
      if (m0 >= args.M || x >= args.N) return;
      tma_store_2d(map, hz_tile, x, m0);
      if (x + 64 < args.N) tma_store_2d(map, hz_tile + Cfg::BOX, x + 64, m0);
      bulk_commit();
    };
    if (leader && pair < args.num_tiles) load_s(pair);
    int it = 0;
    for (int tile = pair; tile < args.num_tiles; tile += npairs, ++it) {
      const int m0 = (tile / ntn) * 256 + 128 * static_cast<int>(rank);
      const int n0 = (tile % ntn) * 256;
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      const bool waited = mbar_wait(&tfull[acc], acc_phase, tmo, abort_flag);
      // leave together: the named barriers below have no deadline
      if (named_barrier_any(1, 256, !waited)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + acc * 256 + (static_cast<uint32_t>(g * 32) << 16);
      bool quit = false;
#pragma unroll 1
      for (int sl = 0; sl < 2 && !quit; ++sl) {
        // round sl: super-block sl of the tile (features n0 + 128 sl ...)
        const int x = n0 + sl * 128;
        if (leader) bulk_wait_read_all();  // the previous z store has read the tile
        named_barrier(1, 256);
        tmem_to_tile(taddr, sl);
        tc_fence_before();
        fence_proxy_async_smem();
        named_barrier(1, 256);
        bool fail = false;
        if (leader) {
          if (args.store_h) store_tile(&tmH, x, m0);
          if (sl == 0) {
            fail = !mbar_wait(s_full, static_cast<uint32_t>(s_landed & 1), tmo, abort_flag);
            if (!fail) ++s_landed;
          }
          if (!fail) mbar_arrive_remote(dsmem_addr(hstaged, 0));
          if (!fail && rank == 0) {
            // hstaged and zdone complete twice per tile: round sl is phase sl
            fail = !mbar_wait(hstaged, static_cast<uint32_t>(sl), tmo, abort_flag);
            if (!fail) {
              tc_fence_after();
              constexpr uint32_t idesc_r = idesc_bf16_f32(256, 128, false, false);  // h S^T
              const uint32_t sa = smem_u32(hz_tile), ss = smem_u32(s_tile);
              const uint32_t d = tmem_base + acc * 256 + sl * 128;
#pragma unroll
              for (int kk = 0; kk < 8; ++kk) {
                const uint32_t a_off = (kk >> 2) * Cfg::BOX + (kk & 3) * 32;
                const uint32_t b_off = (2 * sl + (kk >> 2)) * Cfg::SBOX + (kk & 3) * 32;
                mma_bf16_f32_pair(d, smem_desc_sw128(sa + a_off, 16, 1024),
                                  smem_desc_sw128(ss + b_off, 16, 1024), idesc_r, kk != 0 ? 1u : 0u);
              }
              mma_commit_pair(zdone, 0x3);
            }
          }
        }
        if (named_barrier_any(1, 256, fail)) { quit = true; break; }
        const bool zok = mbar_wait(zdone, static_cast<uint32_t>(sl), tmo, abort_flag);
        if (named_barrier_any(1, 256, !zok)) { quit = true; break; }
        tc_fence_after();
        if (leader) bulk_wait_read_all();  // the h store has read the tile
        named_barrier(1, 256);
        tmem_to_tile(taddr, sl);
        tc_fence_before();
        // both halves of z are read: the accumulator is free
        if (sl == 1) mbar_arrive_remote(dsmem_addr(&tempty[acc], 0));
        fence_proxy_async_smem();
        named_barrier(1, 256);
        if (leader) {
          store_tile(&tmZ, x, m0);
          // the tile's transform MMAs are complete: the next tile's S halves may land
          const int next = tile + npairs;
          if (sl == 1 && next < args.num_tiles) load_s(next);
        }
      }
      if (quit) break;
    }
    if (leader) {
      bulk_wait_all();
      volatile int never = 0;
      if (s_loads > s_landed) mbar_wait(s_full, static_cast<uint32_t>(s_landed & 1), tmo, &never);
      if (rank == 0) {  // every transform MMA is complete before TMEM is freed
        mma_commit_pair(zdrain, 0x1);
        mbar_wait(zdrain, 0, tmo, &never);
      }
    }
  }

  // every main-loop MMA of the pair must be complete before TMEM is freed
  if (warp == 1 && lane == 0) {
    volatile int never = 0;
    mbar_wait(drain, 0, tmo, &never);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA frees TMEM or exits while the other may still use it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, 512);
  }
}

}  // namespace poetx
