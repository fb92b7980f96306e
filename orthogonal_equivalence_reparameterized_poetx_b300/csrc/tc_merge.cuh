// Tensor-core merge pass (tcgen05): one right-multiplication by a
// block-diagonal near-identity matrix, in fp32-grade precision from bf16
// operands, with the result written transposed.
//
// The merge W <- R W P ("POET-X: Memory-efficient LLM Training by Scaling
// Orthogonal Transformation", Methodologie §1) multiplies the weight by two
// block-diagonal orthogonal matrices whose blocks are close to the identity.
// Each pass here computes, for a row-major A (M x N) split as A = A_hi + A_lo
// (two bf16 arrays, A_lo optional) and super-blocks D_s = B_s - I split the
// same way (D_hi + D_lo, both bf16, rows = output features, K-major):
//   C[:, s] = A[:, s] + A_hi[:, s] D_hi,s^T + A_hi[:, s] D_lo,s^T (+ A_lo[:, s] D_hi,s^T)
// i.e. C = A B^T per super-block with the identity part added exactly in the
// epilogue and only the small correction A (B - I)^T taken on the tensor
// cores.  The dropped terms (A_lo D_lo, and the splitting residues) are below
// 2^-16 of |A| |B - I|, so one pass loses nothing a later bf16 rounding
// would keep.  The epilogue writes C^T (N x M, row-major) as a hi/lo pair
// (or hi only), which serves directly as the next pass's A.  Two passes
// therefore apply one block-diagonal factor from the right and the other from
// the left, and the second transposition restores the original orientation:
// pass 1 maps W to (W B_P)^T, pass 2 maps that to B_R W B_P.
//
// Warps: 0 TMA producer, 1 TMEM allocator + MMA issuer, 2..9 epilogue.
// Tile: 128 rows x 128 output columns; K = the super-block (sb) of those
// columns in 64-wide steps.  Persistent over tiles, accumulator double-
// buffered in TMEM (2 x 128 columns).
#pragma once

#include "ptx.cuh"

namespace poetx {

struct MergeArgs {
  int M;                          // rows of A
  int N;                          // columns of A (and of C)
  int sb;                         // super-block size (multiple of 128)
  int num_tiles;                  // ceil(M / 128) * ceil(N / 128)
  const __nv_bfloat16* res_hi;    // A_hi, row-major M x N (the exact identity part)
  const __nv_bfloat16* res_lo;    // A_lo or nullptr
  __nv_bfloat16* out_hi;          // C^T rounded to bf16, row-major N x M
  __nv_bfloat16* out_lo;          // bf16(C^T - out_hi) or nullptr
  uint64_t timeout_ns;
};

template <bool A_SPLIT>
struct MergeCfg {
  static constexpr int BOX = 128 * 64 * 2;        // 128 rows x 64 k, bf16: 16 KB
  static constexpr int NBOX = A_SPLIT ? 4 : 3;    // A_hi, [A_lo], D_hi, D_lo
  static constexpr int STAGE = NBOX * BOX;
  static constexpr int STAGES = A_SPLIT ? 3 : 4;
  static constexpr int SMEM = 1024 + STAGES * STAGE + 256;
  static_assert(SMEM <= 232448, "shared memory");
};

template <bool A_SPLIT>
__global__ void __launch_bounds__(320, 1)
    tc_merge_kernel(const __grid_constant__ CUtensorMap tmAhi, const __grid_constant__ CUtensorMap tmAlo,
                    const __grid_constant__ CUtensorMap tmDhi, const __grid_constant__ CUtensorMap tmDlo,
                    const MergeArgs args) {
  using Cfg = MergeCfg<A_SPLIT>;
  constexpr int STAGES = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned by pointer arithmetic on the shared array, so that the
  // compiler keeps shared-memory instructions for the accesses through it
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * Cfg::STAGE);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint64_t tmo = args.timeout_ns;
  const int ntn = (args.N + 127) / 128;
  const int nk = args.sb / 64;

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
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmAhi);
    if constexpr (A_SPLIT) tma_prefetch_desc(&tmAlo);
    tma_prefetch_desc(&tmDhi);
    tma_prefetch_desc(&tmDlo);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_phase[STAGES];
      bool issued[STAGES];
      for (int i = 0; i < STAGES; ++i) issued[i] = false, issued_phase[i] = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < args.num_tiles && ok; tile += gridDim.x) {
        const int m0 = (tile / ntn) * 128, n0 = (tile % ntn) * 128;
        const int kx0 = (n0 / args.sb) * args.sb;  // first input column of the super-block
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, tmo, abort_flag)) { ok = false; break; }
          uint8_t* st = smem + stage * Cfg::STAGE;
          mbar_arrive_expect_tx(&full[stage], Cfg::STAGE);
          int b = 0;
          tma_load_2d(st + (b++) * Cfg::BOX, &tmAhi, &full[stage], kx0 + kb * 64, m0);
          if constexpr (A_SPLIT) tma_load_2d(st + (b++) * Cfg::BOX, &tmAlo, &full[stage], kx0 + kb * 64, m0);
          tma_load_2d(st + (b++) * Cfg::BOX, &tmDhi, &full[stage], kb * 64, n0);
          tma_load_2d(st + (b++) * Cfg::BOX, &tmDlo, &full[stage], kb * 64, n0);
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
      // ------------------------------------------------------------ MMA issuer
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
        const uint32_t d = tmem_base + acc * 128;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(&full[stage], phase, tmo, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t s0 = smem_u32(smem + stage * Cfg::STAGE);
          const uint32_t a_hi = s0;
          const uint32_t a_lo = s0 + Cfg::BOX;                       // A_SPLIT only
          const uint32_t d_hi = s0 + (A_SPLIT ? 2 : 1) * Cfg::BOX;
          const uint32_t d_lo = d_hi + Cfg::BOX;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t o = kk * 32;
            const uint64_t ah = smem_desc_sw128(a_hi + o, 16, 1024);
            mma_bf16_f32(d, ah, smem_desc_sw128(d_hi + o, 16, 1024), idesc, (kb | kk) != 0 ? 1u : 0u);
            mma_bf16_f32(d, ah, smem_desc_sw128(d_lo + o, 16, 1024), idesc, 1u);
            if constexpr (A_SPLIT)
              mma_bf16_f32(d, smem_desc_sw128(a_lo + o, 16, 1024), smem_desc_sw128(d_hi + o, 16, 1024),
                           idesc, 1u);
          }
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
    // warp w: TMEM lanes (rows) 32*(w%4).., columns 64*half .. +63 of the tile
    const int g = warp & 3;
    const int half = (warp - 2) >> 2;
    int it = 0;
    for (int tile = blockIdx.x; tile < args.num_tiles; tile += gridDim.x, ++it) {
      const int m0 = (tile / ntn) * 128, n0 = (tile % ntn) * 128;
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      if (!mbar_wait(&tfull[acc], acc_phase, tmo, abort_flag)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + acc * 128 + half * 64 + (static_cast<uint32_t>(g * 32) << 16);
      uint32_t r[2][32];
      tmem_ld_32x32b_x32(taddr, r[0]);
      tmem_ld_32x32b_x32(taddr + 32, r[1]);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      const int row = m0 + g * 32 + lane;
      if (row >= args.M) continue;
      const int64_t rin = static_cast<int64_t>(row) * args.N;
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8) {
        const int col = n0 + half * 64 + c8 * 8;
        if (col >= args.N) break;  // N is a multiple of 8: a chunk is all in or all out
        const uint4 rh = *reinterpret_cast<const uint4*>(args.res_hi + rin + col);
        uint4 rl = make_uint4(0u, 0u, 0u, 0u);
        if (args.res_lo) rl = *reinterpret_cast<const uint4*>(args.res_lo + rin + col);
        const __nv_bfloat16* eh = reinterpret_cast<const __nv_bfloat16*>(&rh);
        const __nv_bfloat16* el = reinterpret_cast<const __nv_bfloat16*>(&rl);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int c = c8 * 8 + e;
          const float v = __uint_as_float(r[c >> 5][c & 31]) + __bfloat162float(eh[e]) +
                          __bfloat162float(el[e]);
          const __nv_bfloat16 hi = __float2bfloat16_rn(v);
          const int64_t o = static_cast<int64_t>(col + e) * args.M + row;  // transposed
          args.out_hi[o] = hi;
          if (args.out_lo) args.out_lo[o] = __float2bfloat16_rn(v - __bfloat162float(hi));
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 256);
  }
}

}  // namespace poetx
