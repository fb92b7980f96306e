// tcgen05 GEMM engine for the bf16 layer path.
//
// C = A * B^T with bf16 operands staged by TMA into 128-byte-swizzled shared
// memory, fp32 accumulation in tensor memory (TMEM), and an epilogue that
// reads TMEM with tcgen05.ld and stores bf16 or fp32.
//
// One CTA per SM (persistent), 10 warps:
//   warp 0      TMA producer (one elected lane)
//   warp 1      TMEM allocator and single-thread MMA issuer
//   warps 2..9  epilogue; warp w reads TMEM lanes 32*(w%4) .. 32*(w%4)+31 and
//               64-column half (w-2)/4 of every 128-column slice of the tile
// The accumulator is double-buffered in TMEM (2 x BN columns) so the
// epilogue of one tile overlaps the main loop of the next.  bf16 results are
// staged per 128-column slice in a 128-byte-swizzled shared buffer and
// written with TMA bulk tensor stores (whole lines, clipped at the edges);
// fp32 partials of the token reductions are stored directly.
//
// Three tile schedules cover every contraction of the layer:
//   Dense      h = v W0'^T (B K-major) and dv = dh W0' (B MN-major): tiles of
//              128 rows x BN columns, full K.
//   BlockDiag  out[:, s] = in[:, s] * S_s^T for a block-diagonal matrix stored
//              as "super-blocks" S_s of sb x sb (sb = max(b, 128); smaller
//              blocks sit on the diagonal of a super-block): K = sb per tile.
//              This is "Methodologie §3" of the POET-X summary (blocks handled
//              as independent matrices, batch-parallel).
//   GradRed    partial[p][s] = sum over tokens in split p of
//              A[t, s]^T B[t, s]: both operands MN-major (features contiguous),
//              K = tokens; a deterministic reduction over p follows.
#pragma once

#include "ptx.cuh"

namespace poetx {

enum class TileMode : int { Dense = 0, BlockDiag = 1, GradRed = 2 };

struct TcGemmArgs {
  int M;        // Dense/BlockDiag: rows of C (tokens)
  int N;        // Dense/BlockDiag: columns of C (features)
  int K;        // Dense: contraction length
  int sb;       // BlockDiag/GradRed: super-block size (multiple of 128)
  int nsb;      // GradRed: number of super-blocks
  int tokens;   // GradRed: token count
  int chunk;    // GradRed: tokens per split (multiple of 64)
  int num_tiles;
  void* C;
  int64_t ldc;             // Dense/BlockDiag: elements between rows of C
  int64_t split_stride;    // GradRed: floats between split partials
  uint64_t timeout_ns;
};

template <int BN, bool STAGED>
struct TcGemmCfg {
  static constexpr int BM = 128;
  static constexpr int BK = 64;
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = (BN >= 256) ? 4 : 6;
  static constexpr int TMEM_COLS = 2 * BN;
  static constexpr int OUT_BYTES = STAGED ? 128 * 128 * 2 : 0;  // one 128 x 128 bf16 slice
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + OUT_BYTES + 256;
  static_assert(BN == 128 || BN == 256, "BN");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

struct TileInfo {
  int m0, n0;      // Dense/BlockDiag: C tile origin.  GradRed: feature origins
  int kx0, ky0;    // operand coordinate bases
  int nk;          // k-iterations of 64
  int p, s, i, j;  // GradRed indices
};

template <int BN, TileMode MODE>
__device__ __forceinline__ TileInfo decode_tile(int tile, const TcGemmArgs& a) {
  TileInfo t{};
  if constexpr (MODE == TileMode::Dense || MODE == TileMode::BlockDiag) {
    const int ntn = (a.N + BN - 1) / BN;
    const int mt = tile / ntn, nt = tile % ntn;
    t.m0 = mt * 128;
    t.n0 = nt * BN;
    if constexpr (MODE == TileMode::Dense) {
      t.nk = (a.K + 63) / 64;
      t.kx0 = 0;
    } else {
      t.nk = a.sb / 64;
      t.kx0 = (t.n0 / a.sb) * a.sb;  // first input feature of the super-block
    }
  } else {
    const int tps = a.sb / 128;
    const int per_split = a.nsb * tps * tps;
    t.p = tile / per_split;
    int r = tile % per_split;
    t.s = r / (tps * tps);
    r %= tps * tps;
    t.i = r / tps;
    t.j = r % tps;
    t.m0 = t.s * a.sb + t.i * 128;
    t.n0 = t.s * a.sb + t.j * 128;
    t.ky0 = t.p * a.chunk;
    const int len = min(a.chunk, a.tokens - t.ky0);
    t.nk = (len + 63) / 64;
  }
  return t;
}

template <int BN, bool A_MN, bool B_MN, TileMode MODE, typename OutT>
__global__ void __launch_bounds__(320, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const TcGemmArgs args) {
  constexpr bool STAGED = (MODE != TileMode::GradRed);
  using Cfg = TcGemmCfg<BN, STAGED>;
  constexpr int STAGES = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned by pointer arithmetic on the shared array, so that the
  // compiler keeps shared-memory instructions for the accesses through it
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* out_stage = smem + STAGES * Cfg::STAGE_BYTES;  // 1024-aligned
  uint64_t* full = reinterpret_cast<uint64_t*>(out_stage + Cfg::OUT_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint64_t tmo = args.timeout_ns;

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
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if constexpr (STAGED) tma_prefetch_desc(&tmC);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
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
        const TileInfo t = decode_tile<BN, MODE>(tile, args);
        for (int kb = 0; kb < t.nk; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, tmo, abort_flag)) { ok = false; break; }
          uint8_t* sa = smem + stage * Cfg::STAGE_BYTES;
          uint8_t* sb = sa + Cfg::A_BYTES;
          mbar_arrive_expect_tx(&full[stage], Cfg::STAGE_BYTES);
          if constexpr (MODE == TileMode::GradRed) {
            const int ky = t.ky0 + kb * 64;
            tma_load_2d(sa, &tmA, &full[stage], t.m0, ky);
            tma_load_2d(sa + 64 * 128, &tmA, &full[stage], t.m0 + 64, ky);
#pragma unroll
            for (int h = 0; h < BN / 64; ++h)
              tma_load_2d(sb + h * 64 * 128, &tmB, &full[stage], t.n0 + 64 * h, ky);
          } else {
            const int kx = t.kx0 + kb * 64;
            tma_load_2d(sa, &tmA, &full[stage], kx, t.m0);
            if constexpr (MODE == TileMode::BlockDiag) {
              tma_load_2d(sb, &tmB, &full[stage], kb * 64, t.n0);
            } else if constexpr (B_MN) {
#pragma unroll
              for (int h = 0; h < BN / 64; ++h)
                tma_load_2d(sb + h * 64 * 128, &tmB, &full[stage], t.n0 + 64 * h, kb * 64);
            } else {
              tma_load_2d(sb, &tmB, &full[stage], kb * 64, t.n0);
            }
          }
          issued[stage] = true;
          issued_phase[stage] = phase;
          if (++stage == STAGES) stage = 0, phase ^= 1u;
        }
      }
      // Copies in flight must land before the CTA may exit.
      for (int s = 0; s < STAGES; ++s)
        if (issued[s]) {
          volatile int never = 0;
          mbar_wait(&full[s], issued_phase[s], tmo, &never);
        }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      constexpr uint32_t idesc = idesc_bf16_f32(128, BN, A_MN, B_MN);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < args.num_tiles && ok; tile += gridDim.x, ++it) {
        const TileInfo t = decode_tile<BN, MODE>(tile, args);
        const int acc = it & 1;
        const uint32_t acc_phase = (it >> 1) & 1;
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, tmo, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < t.nk; ++kb) {
          if (!mbar_wait(&full[stage], phase, tmo, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * Cfg::STAGE_BYTES);
          const uint32_t sb = sa + Cfg::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            uint64_t ad, bd;
            if constexpr (A_MN) ad = smem_desc_sw128(sa + kk * 2048, 64 * 128, 1024);
            else ad = smem_desc_sw128(sa + kk * 32, 16, 1024);
            if constexpr (B_MN) bd = smem_desc_sw128(sb + kk * 2048, 64 * 128, 1024);
            else bd = smem_desc_sw128(sb + kk * 32, 16, 1024);
            mma_bf16_f32(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          mma_commit(&empty[stage]);
          if (++stage == STAGES) stage = 0, phase ^= 1u;
        }
        if (!ok) break;
        mma_commit(&tfull[acc]);
      }
      // Every MMA this thread issued must finish before TMEM is released.
      mma_commit(drain);
      volatile int never = 0;
      mbar_wait(drain, 0, tmo, &never);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int g = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row = g * 32 + lane;
    const bool leader = (warp == 2 && lane == 0);
    int it = 0;
    for (int tile = blockIdx.x; tile < args.num_tiles; tile += gridDim.x, ++it) {
      const TileInfo t = decode_tile<BN, MODE>(tile, args);
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      const bool waited = mbar_wait(&tfull[acc], acc_phase, tmo, abort_flag);
      // leave together: the named barriers below have no deadline
      if (named_barrier_any(1, 256, !waited)) break;
      tc_fence_after();
      const bool empty_tile = t.nk <= 0;  // no MMA wrote this accumulator: store zeros
      const uint32_t taddr = tmem_base + acc * BN + (static_cast<uint32_t>(g * 32) << 16);
#pragma unroll 1
      for (int sl = 0; sl < BN / 128; ++sl) {
        // this warp's 64 columns of the 128-column slice: two loads, one wait
        const int c0 = sl * 128 + half * 64;
        uint32_t r[2][32];
        tmem_ld_32x32b_x32(taddr + c0, r[0]);
        tmem_ld_32x32b_x32(taddr + c0 + 32, r[1]);
        tmem_ld_wait();
        if (sl == BN / 128 - 1) {  // accumulator fully read: release it to the MMA warp
          tc_fence_before();
          mbar_arrive(&tempty[acc]);
        }
        if (empty_tile) {
#pragma unroll
          for (int q = 0; q < 32; ++q) r[0][q] = r[1][q] = 0u;
        }
        if constexpr (MODE == TileMode::GradRed) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            float* out = reinterpret_cast<float*>(args.C) + t.p * args.split_stride +
                         static_cast<int64_t>(t.s) * args.sb * args.sb +
                         static_cast<int64_t>(t.i * 128 + row) * args.sb + t.j * 128 + c0 + 32 * hh;
#pragma unroll
            for (int q = 0; q < 8; ++q)
              reinterpret_cast<uint4*>(out)[q] =
                  make_uint4(r[hh][4 * q], r[hh][4 * q + 1], r[hh][4 * q + 2], r[hh][4 * q + 3]);
          }
        } else {
          // the previous slice's TMA stores must have read the staging buffer
          if (leader) bulk_wait_read_all();
          named_barrier(1, 256);
          // 128-byte-swizzled box `half` (64 columns x 128 rows): 16-byte chunk q
          // of row `row` sits at chunk (q ^ (row % 8)).
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
          if (leader && t.n0 + sl * 128 < args.N) {
            const int x = t.n0 + sl * 128;
            tma_store_2d(&tmC, out_stage, x, t.m0);
            if (x + 64 < args.N) tma_store_2d(&tmC, out_stage + 128 * 128, x + 64, t.m0);
            bulk_commit();
          }
        }
      }
    }
    if constexpr (STAGED) {
      if (leader) bulk_wait_all();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
  }
}

}  // namespace poetx
