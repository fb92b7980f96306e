// bf16 GEMMs on CTA pairs (tcgen05 .cta_group::2).
//
// Dense: C (M x N, bf16, row-major) = A (M x K, K-major) * B^T, with B stored
// N x K (K-major: the forward h = v W0'^T) or K x N (MN-major: the dgrad
// dv = dh W0').
// GradRed: partial[p][s] = sum over the tokens of split p of A[t, s]^T B[t, s]
// for super-blocks of sb >= 256 (both operands MN-major, K = tokens), as
// 256 x 256 fp32 tiles of each sb x sb product, stored directly.
// ("POET-X: Memory-efficient LLM Training by Scaling Orthogonal
// Transformation", Methodologie §3: the blocks as independent matrices.)  A cluster of two CTAs owns 256 x 256 output tiles
// (persistent over tiles): CTA r stages rows [128 r, 128 r + 128) of the A
// tile and columns [128 r, 128 r + 128) of the B tile, the even CTA issues
// M = 256, N = 256 MMAs that read both CTAs' shared memory, and each CTA's
// TMEM receives its own 128 accumulator rows for all 256 columns.  Compared
// with one CTA per 128 x 256 tile, every SM stages and feeds the tensor core
// half the B bytes per MMA, which is what bounds the single-CTA kernel.
//
// Warps (both CTAs): 0 TMA producer, 1 TMEM allocator (even CTA: also the MMA
// issuer), 2..9 epilogue (TMEM -> bf16 -> swizzled shared memory -> TMA
// store of this CTA's 128 rows).  Barriers:
//   full[s]    even CTA's: both CTAs' TMA bytes of stage s (one expect_tx)
//   empty[s]   each CTA's: the MMAs reading stage s are done (multicast commit)
//   tfull[a]   each CTA's: accumulator a is complete (multicast commit)
//   tempty[a]  even CTA's: both CTAs' epilogues have read accumulator a
//   drain      each CTA's: every MMA has completed (before TMEM is freed)
// Every wait is bounded; on a timeout a CTA records it and winds down, and
// the pair meets at a cluster barrier before freeing TMEM and exiting.
#pragma once

#include "ptx.cuh"

namespace poetx {

enum class PairMode : int { Dense = 0, GradRed = 1 };

struct TcPairArgs {
  int M, N, K;            // Dense: C is M x N, contraction K
  int num_tiles;          // Dense: ceil(M / 256) * ceil(N / 256);
                          // GradRed: splits * nsb * (sb / 256)^2
  int sb;                 // GradRed: super-block size (multiple of 256)
  int nsb;                // GradRed: super-blocks
  int tokens, chunk;      // GradRed: tokens, tokens per split (multiple of 64)
  float* C;               // GradRed: partials [split][nsb][sb][sb]
  int64_t split_stride;   // GradRed: floats between split partials
  uint64_t timeout_ns;
};

// One output tile as CTA `rank` of the pair sees it.
struct PairTile {
  int m0;    // this CTA's A origin: rows (Dense) or features (GradRed)
  int nb;    // this CTA's B origin (features)
  int n0;    // Dense: the tile's first output column
  int ky0;   // GradRed: first token of the split
  int nk;    // k-iterations of 64
  int p, s, i, j, row0;  // GradRed: split, super-block, tile indices, local row origin
};

template <PairMode MODE>
__device__ __forceinline__ PairTile decode_pair(int tile, const TcPairArgs& a, uint32_t rank) {
  PairTile t{};
  if constexpr (MODE == PairMode::GradRed) {
    const int tps = a.sb / 256;
    const int per_split = a.nsb * tps * tps;
    t.p = tile / per_split;
    int r = tile % per_split;
    t.s = r / (tps * tps);
    r %= tps * tps;
    t.i = r / tps;
    t.j = r % tps;
    t.row0 = t.i * 256 + 128 * static_cast<int>(rank);
    t.m0 = t.s * a.sb + t.row0;
    t.nb = t.s * a.sb + t.j * 256 + 128 * static_cast<int>(rank);
    t.ky0 = t.p * a.chunk;
    const int len = min(a.chunk, a.tokens - t.ky0);
    t.nk = len > 0 ? (len + 63) / 64 : 0;
  } else {
    const int ntn = (a.N + 255) / 256;
    t.m0 = (tile / ntn) * 256 + 128 * static_cast<int>(rank);
    t.n0 = (tile % ntn) * 256;
    t.nb = t.n0 + 128 * static_cast<int>(rank);
    t.nk = (a.K + 63) / 64;
  }
  return t;
}

struct TcPairCfg {
  static constexpr int A_BYTES = 128 * 64 * 2;  // this CTA's 128 rows x 64 k
  static constexpr int B_BYTES = 128 * 64 * 2;  // this CTA's 128 columns x 64 k
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = 6;
  static constexpr int OUT_BYTES = 128 * 128 * 2;  // one 128 x 128 bf16 slice
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + OUT_BYTES + 256;
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

template <bool B_MN, PairMode MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(320, 1)
    tc_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC, const TcPairArgs args) {
  using Cfg = TcPairCfg;
  constexpr int STAGES = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned by pointer arithmetic on the shared array, so that the
  // compiler keeps shared-memory instructions for the accesses through it
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* out_stage = smem + STAGES * Cfg::STAGE_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(out_stage + Cfg::OUT_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs
  const int pair = blockIdx.x / 2, npairs = gridDim.x / 2;
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
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if constexpr (MODE != PairMode::GradRed) tma_prefetch_desc(&tmC);
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
        const PairTile t = decode_pair<MODE>(tile, args, rank);
        for (int kb = 0; kb < t.nk; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, tmo, abort_flag)) { ok = false; break; }
          uint8_t* sa = smem + stage * Cfg::STAGE_BYTES;
          uint8_t* sb = sa + Cfg::A_BYTES;
          const uint32_t fbar = dsmem_addr(&full[stage], 0);  // the even CTA's barrier
          if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * Cfg::STAGE_BYTES);
          if constexpr (MODE == PairMode::GradRed) {
            // both operands MN-major: 64-feature x 64-token boxes
            const int ky = t.ky0 + kb * 64;
            tma_load_2d_pair(sa, &tmA, fbar, t.m0, ky);
            tma_load_2d_pair(sa + 64 * 128, &tmA, fbar, t.m0 + 64, ky);
            tma_load_2d_pair(sb, &tmB, fbar, t.nb, ky);
            tma_load_2d_pair(sb + 64 * 128, &tmB, fbar, t.nb + 64, ky);
          } else {
            tma_load_2d_pair(sa, &tmA, fbar, kb * 64, t.m0);
            if constexpr (B_MN) {
              tma_load_2d_pair(sb, &tmB, fbar, t.nb, kb * 64);
              tma_load_2d_pair(sb + 64 * 128, &tmB, fbar, t.nb + 64, kb * 64);
            } else {
              tma_load_2d_pair(sb, &tmB, fbar, kb * 64, t.nb);
            }
          }
          issued[stage] = true;
          issued_phase[stage] = phase;
          if (++stage == STAGES) stage = 0, phase ^= 1u;
        }
      }
      // this CTA's copies in flight must land before the pair may exit: they
      // count on the even CTA's barrier, which that CTA's MMA thread drains;
      // here wait for the matching empty phase instead (bounded)
      for (int s = 0; s < STAGES; ++s)
        if (issued[s]) {
          volatile int never = 0;
          mbar_wait(&empty[s], issued_phase[s], tmo, &never);
        }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------------------------------------------------- MMA issuer
      constexpr bool A_MN = MODE == PairMode::GradRed;
      constexpr bool BM = B_MN || MODE == PairMode::GradRed;
      constexpr uint32_t idesc = idesc_bf16_f32(256, 256, A_MN, BM);
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
        const int nk = decode_pair<MODE>(tile, args, rank).nk;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(&full[stage], phase, tmo, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * Cfg::STAGE_BYTES);
          const uint32_t sb = sa + Cfg::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            uint64_t ad, bd;
            if constexpr (A_MN) ad = smem_desc_sw128(sa + kk * 2048, 64 * 128, 1024);
            else ad = smem_desc_sw128(sa + kk * 32, 16, 1024);
            if constexpr (BM) bd = smem_desc_sw128(sb + kk * 2048, 64 * 128, 1024);
            else bd = smem_desc_sw128(sb + kk * 32, 16, 1024);
            mma_bf16_f32_pair(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
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
    int it = 0;
    for (int tile = pair; tile < args.num_tiles; tile += npairs, ++it) {
      const PairTile t = decode_pair<MODE>(tile, args, rank);
      const int m0 = t.m0, n0 = t.n0;
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      const bool waited = mbar_wait(&tfull[acc], acc_phase, tmo, abort_flag);
      // leave together: the named barriers below have no deadline
      if (named_barrier_any(1, 256, !waited)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + acc * 256 + (static_cast<uint32_t>(g * 32) << 16);
#pragma unroll 1
      for (int sl = 0; sl < 2; ++sl) {
        const int c0 = sl * 128 + half * 64;
        uint32_t r[2][32];
        tmem_ld_32x32b_x32(taddr + c0, r[0]);
        tmem_ld_32x32b_x32(taddr + c0 + 32, r[1]);
        tmem_ld_wait();
        if (sl == 1) {  // accumulator fully read: release it to the MMA thread
          tc_fence_before();
          mbar_arrive_remote(dsmem_addr(&tempty[acc], 0));
        }
        if constexpr (MODE == PairMode::GradRed) {
          // fp32 partial rows straight to global memory: local feature row
          // t.row0 + row of super-block t.s, columns t.j * 256 + c0 ..
          if (t.nk == 0) {  // no MMA wrote this accumulator (an empty split)
#pragma unroll
            for (int q = 0; q < 32; ++q) r[0][q] = r[1][q] = 0u;
          }
          float* out = args.C + t.p * args.split_stride + static_cast<int64_t>(t.s) * args.sb * args.sb +
                       static_cast<int64_t>(t.row0 + row) * args.sb + t.j * 256 + c0;
#pragma unroll
          for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int q = 0; q < 8; ++q)
              reinterpret_cast<uint4*>(out + 32 * hh)[q] =
                  make_uint4(r[hh][4 * q], r[hh][4 * q + 1], r[hh][4 * q + 2], r[hh][4 * q + 3]);
          continue;
        }
        if (leader) bulk_wait_read_all();
        named_barrier(1, 256);
        uint8_t* box = out_stage + half * (128 * 128);
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
        if (leader && n0 + sl * 128 < args.N && m0 < args.M) {
          const int x = n0 + sl * 128;
          tma_store_2d(&tmC, out_stage, x, m0);
          if (x + 64 < args.N) tma_store_2d(&tmC, out_stage + 128 * 128, x + 64, m0);
          bulk_commit();
        }
      }
    }
    if constexpr (MODE != PairMode::GradRed) {
      if (leader) bulk_wait_all();
    }
  }

  // every MMA of the pair must be complete before TMEM is freed
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
