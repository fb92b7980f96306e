// Batched fp32-grade GEMM on the tensor cores (tcgen05), for the small dense
// per-block products of the bf16 layer path: the Cayley backward
// 2 M^T G M^T (b >= 256), the batched Neumann chain rule (b >= 256) and the
// Neumann builder products of small blocks.
//
//   C[z] = alpha * A[z] B[z]^T + beta * C[z],   z = 0 .. batch-1
//
// A (M x K) and B (N x K) are fp32 in global memory, each contiguous along
// K ("K-contiguous") or along its rows ("row-contiguous"); both are read by
// TMA as 3-D tensors (contiguous index, other index, batch).  Every staged
// value v is split into two bf16 terms hi = bf16(v), lo = bf16(v - hi), and
// each 16-wide K step issues three MMAs, A_hi B_hi + A_hi B_lo + A_lo B_hi,
// accumulating in fp32 in TMEM.  The dropped A_lo B_lo term and the split
// residues are below 2^-16 of |A| |B| per product (about 1e-5 relative), far
// inside the bf16 path's tolerance though not fp32 round-off, which is why
// the fp32 layer path keeps its CUDA-core products.
//
// One 128 x 128 output tile per CTA (grid: tiles x batch), 10 warps:
//   warp 0      TMA producer: 64-wide K chunks of A and B as fp32, two stages
//   warp 1      TMEM allocator; one thread issues the MMAs of each chunk
//   warps 2..9  convert each fp32 chunk into 128-byte-swizzled bf16 hi/lo
//               tiles, then (after the last chunk) read the accumulator,
//               stage it in shared memory and write C with coalesced stores
// Every wait is bounded; on a timeout the kernel records it and returns.
#pragma once

#include "ptx.cuh"

namespace poetx {

struct F32GemmArgs {
  int M, N, K;
  float* c;           // C(i, j) of batch z: c[z * c_bs + i * c_rs + j]
  int64_t c_rs, c_bs;
  float alpha, beta;
  uint64_t timeout_ns;
};

struct F32GemmCfg {
  static constexpr int F32_TILE = 128 * 64 * 4;   // one operand chunk, fp32: 32 KB
  static constexpr int F32_STAGE = 2 * F32_TILE;  // A and B
  static constexpr int F32_STAGES = 2;
  static constexpr int BOX = 128 * 64 * 2;        // 128 rows x 64 k, bf16: 16 KB
  static constexpr int BF_TILES = 4 * BOX;        // A_hi, A_lo, B_hi, B_lo (64 KB; later the C tile)
  static constexpr int SMEM = 1024 + F32_STAGES * F32_STAGE + BF_TILES + 128;
  static_assert(SMEM <= 232448, "shared memory");
};

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int32_t x,
                                            int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

__device__ __forceinline__ uint32_t split_bf16x2(float a0, float a1, uint32_t& lo) {
  const __nv_bfloat16 h0 = __float2bfloat16_rn(a0), h1 = __float2bfloat16_rn(a1);
  lo = pack_bf16x2(a0 - __bfloat162float(h0), a1 - __bfloat162float(h1));
  return static_cast<uint32_t>(__bfloat16_as_ushort(h0)) |
         (static_cast<uint32_t>(__bfloat16_as_ushort(h1)) << 16);
}

// Converts one staged fp32 chunk (128 rows x 64 k) into the hi and lo bf16
// boxes (K-major, 128-byte swizzle: 16-byte chunk c of row r at c ^ (r % 8)).
// t: converter thread 0..255.  K-contiguous staging is [row][k] (256-byte
// rows); row-contiguous staging is [k][row] (512-byte rows).
template <bool KCONTIG>
__device__ __forceinline__ void f32gemm_convert(const float* src, uint8_t* hi, uint8_t* lo, int t) {
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    int r, c;
    float v[8];
    if constexpr (KCONTIG) {
      // lanes along k: 8 lanes cover one row's 64 values, a warp 4 rows
      const int e = t + 256 * u;
      r = e / 8;
      c = e % 8;
      const float4 a = *reinterpret_cast<const float4*>(src + r * 64 + 8 * c);
      const float4 b = *reinterpret_cast<const float4*>(src + r * 64 + 8 * c + 4);
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
      v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
      // lanes along rows: consecutive words of each staged k row
      r = t % 128;
      c = 4 * (t / 128) + u;
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = src[(8 * c + e) * 128 + r];
    }
    uint32_t h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) h[e] = split_bf16x2(v[2 * e], v[2 * e + 1], l[e]);
    const int off = r * 128 + ((c ^ (r & 7)) << 4);
    *reinterpret_cast<uint4*>(hi + off) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(lo + off) = make_uint4(l[0], l[1], l[2], l[3]);
  }
}

template <bool A_KCONTIG, bool B_KCONTIG>
__global__ void __launch_bounds__(320, 1)
    tc_f32gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const F32GemmArgs args) {
  using Cfg = F32GemmCfg;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned by pointer arithmetic on the shared array, so that the
  // compiler keeps shared-memory instructions for the accesses through it
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* bf = smem + Cfg::F32_STAGES * Cfg::F32_STAGE;  // bf16 tiles, then the C tile
  uint64_t* full = reinterpret_cast<uint64_t*>(bf + Cfg::BF_TILES);
  uint64_t* fempty = full + Cfg::F32_STAGES;
  uint64_t* cvt = fempty + Cfg::F32_STAGES;
  uint64_t* mdone = cvt + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mdone + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int ntn = (args.N + 127) / 128;
  const int m0 = (blockIdx.x / ntn) * 128, n0 = (blockIdx.x % ntn) * 128;
  const int z = blockIdx.y;
  const int nk = (args.K + 63) / 64;
  const uint64_t tmo = args.timeout_ns;

  if (threadIdx.x == 0) {
    for (int i = 0; i < Cfg::F32_STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&fempty[i], 256);
    }
    mbar_init(cvt, 256);
    mbar_init(mdone, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_enter();

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      bool issued[Cfg::F32_STAGES] = {false, false};
      uint32_t issued_par[Cfg::F32_STAGES] = {0, 0};
      for (int kb = 0; kb < nk; ++kb) {
        const int s = kb % Cfg::F32_STAGES;
        const uint32_t par = static_cast<uint32_t>((kb / Cfg::F32_STAGES) & 1);
        if (!mbar_wait(&fempty[s], par ^ 1u, tmo, abort_flag)) break;
        uint8_t* st = smem + s * Cfg::F32_STAGE;
        mbar_arrive_expect_tx(&full[s], Cfg::F32_STAGE);
        // A: K-contiguous boxes are {64 k, 128 rows}, row-contiguous {128 rows, 64 k}
        if constexpr (A_KCONTIG) tma_load_3d(st, &tmA, &full[s], kb * 64, m0, z);
        else tma_load_3d(st, &tmA, &full[s], m0, kb * 64, z);
        if constexpr (B_KCONTIG) tma_load_3d(st + Cfg::F32_TILE, &tmB, &full[s], kb * 64, n0, z);
        else tma_load_3d(st + Cfg::F32_TILE, &tmB, &full[s], n0, kb * 64, z);
        issued[s] = true;
        issued_par[s] = par;
      }
      for (int i = 0; i < Cfg::F32_STAGES; ++i)
        if (issued[i]) {
          volatile int never = 0;
          mbar_wait(&full[i], issued_par[i], tmo, &never);
        }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t idesc = idesc_bf16_f32(128, 128, false, false);
      const uint32_t a_hi = smem_u32(bf), a_lo = a_hi + Cfg::BOX;
      const uint32_t b_hi = a_hi + 2 * Cfg::BOX, b_lo = a_hi + 3 * Cfg::BOX;
      for (int kb = 0; kb < nk; ++kb) {
        if (!mbar_wait(cvt, static_cast<uint32_t>(kb & 1), tmo, abort_flag)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint32_t o = kk * 32;
          const uint64_t ah = smem_desc_sw128(a_hi + o, 16, 1024), bh = smem_desc_sw128(b_hi + o, 16, 1024);
          mma_bf16_f32(tmem, ah, bh, idesc, (kb | kk) != 0 ? 1u : 0u);
          mma_bf16_f32(tmem, ah, smem_desc_sw128(b_lo + o, 16, 1024), idesc, 1u);
          mma_bf16_f32(tmem, smem_desc_sw128(a_lo + o, 16, 1024), bh, idesc, 1u);
        }
        mma_commit(mdone);
      }
    }
  } else {
    // -------------------------------------------------- converters, epilogue
    const int t = threadIdx.x - 64;
    bool ok = true;
    for (int kb = 0; kb < nk && ok; ++kb) {
      const int s = kb % Cfg::F32_STAGES;
      ok = mbar_wait(&full[s], static_cast<uint32_t>((kb / Cfg::F32_STAGES) & 1), tmo, abort_flag);
      // the previous chunk's MMAs must be done with the bf16 tiles
      if (ok && kb > 0) ok = mbar_wait(mdone, static_cast<uint32_t>((kb - 1) & 1), tmo, abort_flag);
      if (!ok) break;
      const float* st = reinterpret_cast<const float*>(smem + s * Cfg::F32_STAGE);
      f32gemm_convert<A_KCONTIG>(st, bf, bf + Cfg::BOX, t);
      f32gemm_convert<B_KCONTIG>(st + Cfg::F32_TILE / 4, bf + 2 * Cfg::BOX, bf + 3 * Cfg::BOX, t);
      mbar_arrive(&fempty[s]);
      fence_proxy_async_smem();  // generic-proxy stores -> visible to the tensor cores
      mbar_arrive(cvt);
    }
    if (ok && nk > 0) ok = mbar_wait(mdone, static_cast<uint32_t>((nk - 1) & 1), tmo, abort_flag);
    tc_fence_after();
    // every converter thread reaches this barrier exactly once
    named_barrier(1, 256);
    if (ok && nk > 0) {
      // accumulator -> shared C tile [128][128] fp32; 16-byte chunk q of row r at q ^ (r % 8)
      const int g = warp & 3, half = (warp - 2) >> 2;
      const int r = g * 32 + lane;
      uint32_t v[2][32];
      const uint32_t taddr = tmem + half * 64 + (static_cast<uint32_t>(g * 32) << 16);
      tmem_ld_32x32b_x32(taddr, v[0]);
      tmem_ld_32x32b_x32(taddr + 32, v[1]);
      tmem_ld_wait();
      float* ct = reinterpret_cast<float*>(bf);
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const int chunk = half * 16 + q;
        *reinterpret_cast<uint4*>(ct + r * 128 + 4 * (chunk ^ (r & 7))) =
            make_uint4(v[q >> 3][4 * (q & 7)], v[q >> 3][4 * (q & 7) + 1], v[q >> 3][4 * (q & 7) + 2],
                       v[q >> 3][4 * (q & 7) + 3]);
      }
    }
    named_barrier(1, 256);
    if (ok && nk > 0) {
      // coalesced: a warp writes 128 consecutive floats of one row per step
      const float* ct = reinterpret_cast<const float*>(bf);
      float* cz = args.c + z * args.c_bs;
      for (int e = t; e < 128 * 32; e += 256) {
        const int r = e / 32, chunk = e % 32;
        const int row = m0 + r, col = n0 + 4 * chunk;
        if (row >= args.M || col >= args.N) continue;
        const float4 a = *reinterpret_cast<const float4*>(ct + r * 128 + 4 * (chunk ^ (r & 7)));
        float* cp = cz + static_cast<int64_t>(row) * args.c_rs + col;
        float o[4] = {args.alpha * a.x, args.alpha * a.y, args.alpha * a.z, args.alpha * a.w};
        const int nv = min(4, args.N - col);
        if (nv == 4 && (reinterpret_cast<uintptr_t>(cp) & 15) == 0) {
          if (args.beta != 0.f) {
            const float4 old = *reinterpret_cast<const float4*>(cp);
            o[0] += args.beta * old.x; o[1] += args.beta * old.y;
            o[2] += args.beta * old.z; o[3] += args.beta * old.w;
          }
          *reinterpret_cast<float4*>(cp) = make_float4(o[0], o[1], o[2], o[3]);
        } else {
          for (int q = 0; q < nv; ++q) cp[q] = o[q] + (args.beta != 0.f ? args.beta * cp[q] : 0.f);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

}  // namespace poetx
