// Column permutation fused into the block-diagonal transform (and, for the
// backward, into the token reduction), for 128-wide super-blocks (b <= 128)
// and rows of a few KB.
//
// For a row-major activation src (T x d), a permutation perm of its d
// columns, the super-block matrices S_s (rows = output features, K-major) and
// an optional second activation C (T x d):
//   A          = src[:, perm]                      (the gather, never in HBM
//                                                   unless store_a)
//   out[:, s]  = A[:, s] S_s^T                     (block transform)
//   G[slot][s] = sum over this CTA's tokens of A[:, s]^T C[:, s]   (REDUCE)
// ("POET-X: Memory-efficient LLM Training by Scaling Orthogonal
// Transformation", Methodologie §1 and §2: the layer applied to the input,
// the permutations as index maps on the feature axis.)  The forward uses it
// for X -> u -> v (store_a writes u for the backward); the backward for
// dY -> dz -> dh with the dz^T h partials, where dz never reaches HBM.
//
// CTA b owns super-block s = b % nsb and token tiles slot, slot + nslots, ...
// with slot = b / nsb (the schedule of the fused transform + reduction).  For
// each 128-token tile, whole rows of src are staged in shared memory by TMA
// (boxes of 256 columns x `chunk_rows` rows, unswizzled) through a ring of
// two to four chunk slots (at d = 512: 96 or 128 rows in flight); the gather
// warps read the 128 columns perm[128 s + k] of each staged row and write
// them as the 128-byte-swizzled K-major A tile.  The two half-warps of a gather warp work
// on consecutive rows with their column chunks rotated by eight, so that
// they do not read the same offset of two rows (the same bank).  A
// super-block uses only 128 of the d columns of a row, so every row is
// staged by the nsb CTAs of its tile (served from L2): this pays only where
// launches, not bytes, bound the separate gather pass (small d).  The A and C
// tiles are single-buffered to leave the shared memory to the row staging.
//
// Warps: 0 producer (S_s once, row chunks), 1 TMEM allocator + MMA issuer,
// 2..9 epilogue, 10..13 gather (their first thread also loads the C tiles).  Every wait is bounded; after a
// timeout every role stops and the CTA drains what it issued.
#pragma once

#include "ptx.cuh"

namespace poetx {

struct GbdArgs {
  int M;            // tokens
  int N;            // features d
  int nsb;          // super-blocks
  int nslots;       // CTAs per super-block
  int b;            // block size (32, 64 or 128): only diagonal b x b blocks of a partial are written
  int chunk_rows;   // rows per staged chunk (a power of two, at most 128)
  int nbox;         // 256-column boxes per staged row, ceil(N / 256)
  int nstg;         // chunk slots in the ring (2..4)
  int store_a;      // also write A (the gathered activation) through tmA
  const int32_t* perm;   // A[:, c] = src[:, perm[c]]
  float* partial;   // REDUCE: [nslots][nsb][128][128]
  uint64_t timeout_ns;
};

template <bool REDUCE>
struct GbdCfg {
  static constexpr int BOX = 128 * 64 * 2;  // 16 KB
  static constexpr int TILE = 2 * BOX;      // 32 KB (128 x 128 bf16)
  static constexpr int STAGES = 1;
  static constexpr int A_BYTES = STAGES * TILE;
  static constexpr int C_BYTES = REDUCE ? STAGES * TILE : 0;
  static constexpr int FIXED = A_BYTES + C_BYTES + TILE /* S */ + TILE /* out */;
  static constexpr int BAR = 256;
  static constexpr int MAX_SLOTS = 4;
  static constexpr int STG_BYTES = (232448 - 1024 - FIXED - BAR) / 1024 * 1024;  // row-staging ring
  static constexpr int SMEM = 1024 + FIXED + STG_BYTES + BAR;
  static constexpr int THREADS = 448;
  static_assert(SMEM <= 232448, "shared memory");
};

template <bool REDUCE>
__global__ void __launch_bounds__(448, 1)
    tc_gbd_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmS,
                  const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmOut,
                  const __grid_constant__ CUtensorMap tmA, const GbdArgs args) {
  using Cfg = GbdCfg<REDUCE>;
  constexpr int STAGES = Cfg::STAGES;
  constexpr int MAX_SLOTS = Cfg::MAX_SLOTS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* a_tiles = smem;                           // STAGES x 32 KB
  uint8_t* c_tiles = a_tiles + Cfg::A_BYTES;         // STAGES x 32 KB (REDUCE)
  uint8_t* s_tile = c_tiles + Cfg::C_BYTES;          // 32 KB
  uint8_t* out_stage = s_tile + Cfg::TILE;           // 32 KB
  uint8_t* rows_stage = out_stage + Cfg::TILE;       // nstg x slot_bytes
  uint64_t* full = reinterpret_cast<uint64_t*>(rows_stage + Cfg::STG_BYTES);  // C tile landed
  uint64_t* afull = full + STAGES;                   // A tile gathered
  uint64_t* empty = afull + STAGES;                  // stage consumed by the MMAs
  uint64_t* rfull = empty + STAGES;                  // row chunk landed
  uint64_t* rempty = rfull + MAX_SLOTS;              // row chunk read by the gather warps
  uint64_t* tfull = rempty + MAX_SLOTS;
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
  const int f0 = s * 128;
  const int CR = args.chunk_rows;
  const int NSTG = args.nstg;
  const uint32_t box_bytes = static_cast<uint32_t>(CR) * 512u;   // 256 bf16 x CR rows
  const uint32_t slot_bytes = box_bytes * static_cast<uint32_t>(args.nbox);

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&afull[i], 128);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < MAX_SLOTS; ++i) {
      mbar_init(&rfull[i], 1);
      mbar_init(&rempty[i], 128);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 256);
    }
    mbar_init(gdone, 1);
    mbar_init(sfull, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmS);
    if (REDUCE) tma_prefetch_desc(&tmC);
    tma_prefetch_desc(&tmOut);
    if (args.store_a) tma_prefetch_desc(&tmA);
  }
  if (warp == 1) {
    // [0,256): transform accumulators x2, [256,384): reduction
    tmem_alloc(tmem_slot, REDUCE ? 512 : 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  griddep_enter();

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      mbar_arrive_expect_tx(sfull, Cfg::TILE);
      tma_load_2d(s_tile, &tmS, sfull, 0, f0);
      tma_load_2d(s_tile + Cfg::BOX, &tmS, sfull, 64, f0);
      int rs = 0;
      uint32_t rphase = 0;
      uint32_t r_phase_issued[MAX_SLOTS] = {};
      bool r_issued[MAX_SLOTS] = {};
      bool ok = true;
      for (int i = 0; i < ntiles && ok; ++i) {
        const int m0 = (slot + i * args.nslots) * 128;
        const int rows = min(128, args.M - m0);
        for (int r0 = 0; r0 < rows; r0 += CR) {
          if (!mbar_wait(&rempty[rs], rphase ^ 1u, tmo, abort_flag)) {
            ok = false;
            break;
          }
          // whole boxes land (rows past T and columns past d as zeros)
          mbar_arrive_expect_tx(&rfull[rs], slot_bytes);
          uint8_t* dst = rows_stage + rs * slot_bytes;
          for (int k = 0; k < args.nbox; ++k) tma_load_2d(dst + k * box_bytes, &tmX, &rfull[rs], 256 * k, m0 + r0);
          r_issued[rs] = true;
          r_phase_issued[rs] = rphase;
          if (++rs == NSTG) rs = 0, rphase ^= 1u;
        }
      }
      // nothing of ours may still be landing when the CTA exits
      volatile int never = 0;
      mbar_wait(sfull, 0, tmo, &never);
      for (int q = 0; q < NSTG; ++q)
        if (r_issued[q]) mbar_wait(&rfull[q], r_phase_issued[q], tmo, &never);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_t = idesc_bf16_f32(128, 128, false, false);  // A S^T
      constexpr uint32_t idesc_g = idesc_bf16_f32(128, 128, true, true);    // A^T C
      const uint32_t d_g = tmem_base + 256;
      const uint32_t ss = smem_u32(s_tile);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = (ntiles == 0) || mbar_wait(sfull, 0, tmo, abort_flag);
      int done = 0;
      for (int i = 0; i < ntiles && ok; ++i) {
        const int acc = i & 1;
        const uint32_t acc_phase = (i >> 1) & 1;
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, tmo, abort_flag)) break;
        if (!mbar_wait(&afull[stage], phase, tmo, abort_flag)) break;
        if (REDUCE && !mbar_wait(&full[stage], phase, tmo, abort_flag)) break;
        tc_fence_after();
        const uint32_t sa = smem_u32(a_tiles + stage * Cfg::TILE);
        const uint32_t d_t = tmem_base + acc * 128;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * Cfg::BOX + (kk & 3) * 32;
          mma_bf16_f32(d_t, smem_desc_sw128(sa + off, 16, 1024), smem_desc_sw128(ss + off, 16, 1024),
                       idesc_t, kk != 0 ? 1u : 0u);
        }
        if (REDUCE) {
          const uint32_t sc = smem_u32(c_tiles + stage * Cfg::TILE);
#pragma unroll
          for (int kt = 0; kt < 8; ++kt) {
            const uint32_t off = kt * 16 * 128;
            mma_bf16_f32(d_g, smem_desc_sw128(sa + off, Cfg::BOX, 1024),
                         smem_desc_sw128(sc + off, Cfg::BOX, 1024), idesc_g, (i | kt) != 0 ? 1u : 0u);
          }
        }
        mma_commit(&empty[stage]);
        mma_commit(&tfull[acc]);
        ++done;
        if (++stage == STAGES) stage = 0, phase ^= 1u;
      }
      if (REDUCE) {
        mma_commit(gdone);  // the reduction accumulator is complete
        volatile int never = 0;
        if (done > 0) mbar_wait(gdone, 0, tmo, &never);
      }
    }
  } else if (warp < 10) {
    // ---------------------------------------------------------------- epilogue
    const int g = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row = g * 32 + lane;
    const bool leader = (warp == 2 && lane == 0);
    int done = 0;
    for (int i = 0; i < ntiles; ++i) {
      const int m0 = (slot + i * args.nslots) * 128;
      const int acc = i & 1;
      const uint32_t acc_phase = (i >> 1) & 1;
      const bool waited = mbar_wait(&tfull[acc], acc_phase, tmo, abort_flag);
      if (named_barrier_any(1, 256, !waited)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + acc * 128 + half * 64 + (static_cast<uint32_t>(g * 32) << 16);
      uint32_t r[2][32];
      tmem_ld_32x32b_x32(taddr, r[0]);
      tmem_ld_32x32b_x32(taddr + 32, r[1]);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      if (leader) bulk_wait_read_all();
      named_barrier(1, 256);
      uint8_t* box = out_stage + half * Cfg::BOX;
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
        tma_store_2d(&tmOut, out_stage, f0, m0);
        if (f0 + 64 < args.N) tma_store_2d(&tmOut, out_stage + Cfg::BOX, f0 + 64, m0);
        bulk_commit();
      }
      ++done;
    }
    if (leader) bulk_wait_all();
    if (REDUCE) {
      // the CTA's partial (rows = features of A, columns = of C); zeros when
      // it had no token tile; a timed-out CTA leaves it unwritten (the host
      // reads the status word)
      const bool have = (ntiles > 0) && (done == ntiles) && mbar_wait(gdone, 0, tmo, abort_flag);
      if (have || ntiles == 0) {
        if (have) tc_fence_after();
        float* out = args.partial + (static_cast<int64_t>(slot) * args.nsb + s) * 128 * 128 +
                     static_cast<int64_t>(row) * 128;
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          const int col = half * 64 + c * 32;
          if (col / args.b != row / args.b) continue;  // only the diagonal b x b blocks are read
          uint32_t r[32];
          if (have) {
            tmem_ld_32x32b_x32(tmem_base + 256 + col + (static_cast<uint32_t>(g * 32) << 16), r);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int q = 0; q < 32; ++q) r[q] = 0u;
          }
#pragma unroll
          for (int q = 0; q < 8; ++q)
            reinterpret_cast<uint4*>(out + col)[q] =
                make_uint4(r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
        }
      }
    }
  } else {
    // ---------------------------------------------------------------- gather
    const int gt = threadIdx.x - 320;  // 0..127
    const int rg = gt >> 4;                 // row phase 0..7
    const int j = (gt + 8 * (rg & 1)) & 15;  // 16-byte chunk (8 columns) of the tile row
    const bool gleader = (gt == 0);
    // byte offsets in a staged chunk of the chunk's 8 source columns (row 0;
    // row r adds 512 r), -1 past d
    int off[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int c = f0 + 8 * j + e;
      const int p = c < args.N ? __ldg(args.perm + c) : -1;
      off[e] = p >= 0 ? (p >> 8) * static_cast<int>(box_bytes) + (p & 255) * 2 : -1;
    }
    int stage = 0, rs = 0;
    uint32_t phase = 0, rphase = 0;
    uint32_t c_phase_issued[STAGES] = {};
    bool c_issued[STAGES] = {};
    for (int i = 0; i < ntiles; ++i) {
      const int m0 = (slot + i * args.nslots) * 128;
      const int rows = min(128, args.M - m0);
      // the MMAs of this stage's previous tile are done: A and C are free
      const bool w = mbar_wait(&empty[stage], phase ^ 1u, tmo, abort_flag);
      if (gleader && w) {
        // the TMA store of u from this stage's previous tile must have read it
        if (args.store_a) {
          if (STAGES == 1) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
          else asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
        }
        // the C tile lands while the A tile is gathered
        if (REDUCE) {
          uint8_t* sc = c_tiles + stage * Cfg::TILE;
          mbar_arrive_expect_tx(&full[stage], Cfg::TILE);
          tma_load_2d(sc, &tmC, &full[stage], f0, m0);
          tma_load_2d(sc + Cfg::BOX, &tmC, &full[stage], f0 + 64, m0);
          c_issued[stage] = true;
          c_phase_issued[stage] = phase;
        }
      }
      if (named_barrier_any(2, 128, !w)) break;
      uint8_t* A = a_tiles + stage * Cfg::TILE;
      bool failed = false;
      for (int r0 = 0; r0 < rows; r0 += CR) {
        const int nr = min(CR, rows - r0);
        const bool wr = mbar_wait(&rfull[rs], rphase, tmo, abort_flag);
        if (named_barrier_any(2, 128, !wr)) {
          failed = true;
          break;
        }
        const uint8_t* chunk = rows_stage + rs * slot_bytes;
        for (int rr = rg; rr < nr; rr += 8) {
          const uint8_t* sr = chunk + rr * 512;
          uint32_t h[8];
#pragma unroll
          for (int e = 0; e < 8; ++e)
            h[e] = off[e] >= 0 ? static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(sr + off[e])) : 0u;
          const int tr = r0 + rr;
          *reinterpret_cast<uint4*>(A + (j >> 3) * Cfg::BOX + tr * 128 + (((j & 7) ^ (tr & 7)) << 4)) =
              make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16), h[6] | (h[7] << 16));
        }
        mbar_arrive(&rempty[rs]);
        if (++rs == NSTG) rs = 0, rphase ^= 1u;
      }
      if (failed) break;
      // token rows past T are zero (they meet zero-filled rows of C in the reduction)
      for (int tr = rows + rg; tr < 128; tr += 8)
        *reinterpret_cast<uint4*>(A + (j >> 3) * Cfg::BOX + tr * 128 + (((j & 7) ^ (tr & 7)) << 4)) =
            make_uint4(0u, 0u, 0u, 0u);
      fence_proxy_async_smem();
      mbar_arrive(&afull[stage]);
      if (args.store_a) {
        named_barrier(2, 128);
        if (gleader) {
          tma_store_2d(&tmA, A, f0, m0);
          if (f0 + 64 < args.N) tma_store_2d(&tmA, A + Cfg::BOX, f0 + 64, m0);
          bulk_commit();
        }
      }
      if (++stage == STAGES) stage = 0, phase ^= 1u;
    }
    if (gleader) {
      bulk_wait_all();
      // nothing of ours may still be landing when the CTA exits
      volatile int never = 0;
      for (int q = 0; q < STAGES; ++q)
        if (c_issued[q]) mbar_wait(&full[q], c_phase_issued[q], tmo, &never);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, REDUCE ? 512 : 256);
  }
}

}  // namespace poetx
