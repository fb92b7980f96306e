// Truncated-Neumann blocks of size 128, 256 or 512 in one launch, with the
// products on the tensor cores.
//
// "POET-X: Memory-efficient LLM Training by Scaling Orthogonal
// Transformation", Methodologie §4, replaces the Cayley inverse by its
// truncated series; with k terms B = (I + Q)(I + Q + ... + Q^k).  Horner:
//   S_1 = I + Q,  S_{s+1} = I + Q S_s  (s < k),  B = S_k + Q S_k,
// k products of b x b matrices per block.
//
// One cluster per block, one CTA per 128-row x NT-column tile of the block
// (NT = min(b, 256)): 1, 2 or 8 CTAs.  Each product P = Q S_s is computed in
// 64-wide K chunks with fp32-grade operands: converter warps read Q (rows of
// this tile, K-major) and S_s (K rows, MN-major) from global memory through
// L2, split every value v into bf16 hi = bf16(v) and lo = bf16(v - hi) and
// stage them in 128-byte-swizzled tiles; one thread issues
// hi*hi + hi*lo + lo*hi per 16-wide K step (tcgen05, fp32 accumulator in
// TMEM).  The epilogue adds I (or S_k) and writes the tile of S_{s+1} (or B)
// to global memory; a cluster barrier orders those writes before the next
// product's reads.  The iterates alternate between two b x b scratch
// matrices per block.
//
// Warps 0-7: unpack, converters (double-buffered bf16 tiles), epilogue.
// Warp 8: TMEM allocation; lane 0 issues the MMAs.  Every mbarrier wait is
// bounded; after a timeout the kernel skips its remaining work but still
// takes every cluster barrier, so the cluster never waits on it.
#pragma once

#include "ptx.cuh"
#include "simt.cuh"
#include "tc_f32gemm.cuh"

namespace poetx {

struct NeumannSide {
  const float* gen;
  SideGeom s;
  float* B;
  float* Q;
  float* S0;  // two b x b fp32 scratch matrices per block
  float* S1;
  int sb;
  __nv_bfloat16* Bsb;
  __nv_bfloat16* BsbT;
};

// Converts 64 K values of `ROWS` rows of a row-major fp32 matrix (row r at
// src + r * ld, K contiguous) into K-major 128-byte-swizzled bf16 hi / lo
// tiles: 16-byte chunk c of row r at r * 128 + ((c ^ (r % 8)) * 16).  Each of
// the 256 converter threads issues all its loads before it converts any, so
// the operand chunk costs one L2 round trip.
template <int ROWS>
__device__ __forceinline__ void nb_convert_kmajor(const float* src, int64_t ld, uint8_t* hi, uint8_t* lo,
                                                  int t) {
  constexpr int U = ROWS / 32;
  float4 x[U], y[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int e = t + 256 * u, r = e / 8, c = e % 8;
    const float* p = src + static_cast<int64_t>(r) * ld + 8 * c;
    x[u] = __ldcg(reinterpret_cast<const float4*>(p));
    y[u] = __ldcg(reinterpret_cast<const float4*>(p + 4));
  }
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int e = t + 256 * u, r = e / 8, c = e % 8;
    uint32_t h[4], l[4];
    h[0] = split_bf16x2(x[u].x, x[u].y, l[0]);
    h[1] = split_bf16x2(x[u].z, x[u].w, l[1]);
    h[2] = split_bf16x2(y[u].x, y[u].y, l[2]);
    h[3] = split_bf16x2(y[u].z, y[u].w, l[3]);
    const int off = r * 128 + ((c ^ (r & 7)) << 4);
    *reinterpret_cast<uint4*>(hi + off) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(lo + off) = make_uint4(l[0], l[1], l[2], l[3]);
  }
}

// Converts 64 K rows of `COLS` consecutive columns of a row-major fp32
// matrix (K row kk at src + kk * ld) into MN-major 128-byte-swizzled bf16
// hi / lo tiles: atoms of 64 columns x 8 K rows, column chunk nc at
// nc * 8 KB, K row kk at kk * 128, 16-byte chunk c at (c ^ (kk % 8)) * 16.
// All loads of a thread are issued before any conversion, as above.
template <int COLS>
__device__ __forceinline__ void nb_convert_mnmajor(const float* src, int64_t ld, uint8_t* hi,
                                                   uint8_t* lo, int t) {
  constexpr int U = COLS / 32;
  float4 x[U], y[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int e = t + 256 * u;
    const int c = e % 8, nc = (e / 8) % (COLS / 64), kk = e / (COLS / 8);
    const float* p = src + static_cast<int64_t>(kk) * ld + nc * 64 + 8 * c;
    x[u] = __ldcg(reinterpret_cast<const float4*>(p));
    y[u] = __ldcg(reinterpret_cast<const float4*>(p + 4));
  }
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int e = t + 256 * u;
    const int c = e % 8, nc = (e / 8) % (COLS / 64), kk = e / (COLS / 8);
    uint32_t h[4], l[4];
    h[0] = split_bf16x2(x[u].x, x[u].y, l[0]);
    h[1] = split_bf16x2(x[u].z, x[u].w, l[1]);
    h[2] = split_bf16x2(y[u].x, y[u].y, l[2]);
    h[3] = split_bf16x2(y[u].z, y[u].w, l[3]);
    const int off = nc * 8192 + kk * 128 + ((c ^ (kk & 7)) << 4);
    *reinterpret_cast<uint4*>(hi + off) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(lo + off) = make_uint4(l[0], l[1], l[2], l[3]);
  }
}

template <int BS>
struct NeuCfg {
  static constexpr int NT = BS < 256 ? BS : 256;     // tile columns
  static constexpr int RS = BS / 128;                 // row tiles per block
  static constexpr int C = RS * (BS / NT);            // CTAs per block (one cluster)
  static constexpr int NK = BS / 64;                  // K chunks per product
  static constexpr int A_BOX = 128 * 64 * 2;          // bf16, K-major: 16 KB
  static constexpr int B_BOX = 64 * NT * 2;           // bf16, MN-major: 16 or 32 KB
  static constexpr int BUF = 2 * A_BOX + 2 * B_BOX;   // hi and lo of A and B
  static constexpr int SMEM = 1024 + 2 * BUF + 128;
  static constexpr int THREADS = 288;
  static_assert(SMEM <= 232448, "shared memory");
};

template <int BS>
__global__ void __cluster_dims__(NeuCfg<BS>::C, 1, 1) __launch_bounds__(288, 1)
    tc_neumann_kernel(const NeumannSide first, const NeumannSide second, int k, uint64_t timeout_ns) {
  using Cfg = NeuCfg<BS>;
  constexpr int NT = Cfg::NT, RS = Cfg::RS, C = Cfg::C, NK = Cfg::NK;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned by pointer arithmetic on the shared array, so that the
  // compiler keeps shared-memory instructions for the accesses through it
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* cvt_full = reinterpret_cast<uint64_t*>(smem + 2 * Cfg::BUF);  // [2]
  uint64_t* mma_done = cvt_full + 2;                                       // [2]
  uint64_t* acc_full = mma_done + 2;
  uint64_t* drain = acc_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = static_cast<int>(threadIdx.x) / 32, lane = static_cast<int>(threadIdx.x) % 32;
  const int kg = static_cast<int>(blockIdx.x) / C;
  const bool is_first = kg < first.s.nblk;
  const NeumannSide& ns = is_first ? first : second;
  const int kb = is_first ? kg : kg - first.s.nblk;
  const int rank = static_cast<int>(cluster_ctarank());
  const int row0 = 128 * (rank % RS), col0 = NT * (rank / RS);
  const int sz = block_size(ns.s, kb);
  const int64_t base = static_cast<int64_t>(kb) * BS * BS;
  const float* g = ns.gen + static_cast<int64_t>(kb) * BS * (BS - 1) / 2;
  float* const Qk = ns.Q + base;
  float* const S0 = ns.S0 + base;
  float* const S1 = ns.S1 + base;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&cvt_full[i], 256);
      mbar_init(&mma_done[i], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 8) {
    tmem_alloc(tmem_slot, NT);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // 1. this CTA's tile of Q (strict upper triangle unpacked, entry (i, j),
  //    i < j, at i*sz - i(i+1)/2 + (j-i-1); zero beyond the block's size)
  //    and of S_1 = I + Q; eight loads in flight per thread
  if (warp < 8) {
    const int t = static_cast<int>(threadIdx.x);
    for (int e0 = t; e0 < 128 * NT; e0 += 256 * 8) {
      float q[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int e = e0 + 256 * u;
        const int i = row0 + e / NT, j = col0 + e % NT;
        q[u] = 0.f;
        if (e < 128 * NT && i < sz && j < sz && i != j)
          q[u] = i < j ? g[i * sz - i * (i + 1) / 2 + (j - i - 1)]
                       : -g[j * sz - j * (j + 1) / 2 + (i - j - 1)];
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int e = e0 + 256 * u;
        if (e >= 128 * NT) continue;
        const int i = row0 + e / NT, j = col0 + e % NT;
        Qk[i * BS + j] = q[u];
        S0[i * BS + j] = (i == j ? 1.f : 0.f) + q[u];
      }
    }
  }
  cluster_sync();  // every tile of Q and S_1 is written

  // 2. k products P = Q S_s
  int gc = 0;  // K chunks issued so far (over all products): buffer and phase
  bool ok = true;
  for (int s = 1; s <= k; ++s) {
    const float* Scur = (s & 1) ? S0 : S1;   // S_s
    float* Snext = (s & 1) ? S1 : S0;        // S_{s+1}
    if (warp < 8) {
      const int t = static_cast<int>(threadIdx.x);
      // ---------------------------------------------------------- converters
      for (int kc = 0; kc < NK; ++kc, ++gc) {
        const int buf = gc & 1;
        if (ok && gc >= 2)
          ok = mbar_wait(&mma_done[buf], static_cast<uint32_t>(((gc >> 1) - 1) & 1), timeout_ns,
                         abort_flag);
        if (ok) {
          uint8_t* ah = smem + buf * Cfg::BUF;
          uint8_t* al = ah + Cfg::A_BOX;
          uint8_t* bh = al + Cfg::A_BOX;
          uint8_t* bl = bh + Cfg::B_BOX;
          // A = rows [row0, row0 + 128) of Q, K chunk kc (K-major); B(n, kk) =
          // S_s[kc*64 + kk][col0 + n] (MN-major)
          nb_convert_kmajor<128>(Qk + static_cast<int64_t>(row0) * BS + kc * 64, BS, ah, al, t);
          nb_convert_mnmajor<NT>(Scur + static_cast<int64_t>(kc * 64) * BS + col0, BS, bh, bl, t);
          fence_proxy_async_smem();  // generic-proxy stores -> visible to the tensor cores
        }
        mbar_arrive(&cvt_full[buf]);
      }
      // ------------------------------------------------------------ epilogue
      if (ok) ok = mbar_wait(acc_full, static_cast<uint32_t>((s - 1) & 1), timeout_ns, abort_flag);
      tc_fence_after();
      if (ok) {
        const int gq = warp & 3, hh = warp >> 2;
        constexpr int HC = NT / 2;  // columns per warp
        const int i = row0 + gq * 32 + lane;
#pragma unroll 1
        for (int c32 = 0; c32 < HC / 32; ++c32) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(gq * 32) << 16) + hh * HC + c32 * 32, v);
          tmem_ld_wait();
          const int j0 = col0 + hh * HC + c32 * 32;
          if (s < k) {
            float* dst = Snext + static_cast<int64_t>(i) * BS + j0;
#pragma unroll
            for (int q = 0; q < 32; q += 4) {
              float4 o;
              o.x = __uint_as_float(v[q]) + (i == j0 + q ? 1.f : 0.f);
              o.y = __uint_as_float(v[q + 1]) + (i == j0 + q + 1 ? 1.f : 0.f);
              o.z = __uint_as_float(v[q + 2]) + (i == j0 + q + 2 ? 1.f : 0.f);
              o.w = __uint_as_float(v[q + 3]) + (i == j0 + q + 3 ? 1.f : 0.f);
              *reinterpret_cast<float4*>(dst + q) = o;
            }
          } else {
            const float* sk = Scur + static_cast<int64_t>(i) * BS + j0;
            float bv[32];
#pragma unroll
            for (int q = 0; q < 32; q += 4) {
              const float4 a = __ldcg(reinterpret_cast<const float4*>(sk + q));
              bv[q] = a.x + __uint_as_float(v[q]);
              bv[q + 1] = a.y + __uint_as_float(v[q + 1]);
              bv[q + 2] = a.z + __uint_as_float(v[q + 2]);
              bv[q + 3] = a.w + __uint_as_float(v[q + 3]);
            }
            float* bd = ns.B + base + static_cast<int64_t>(i) * BS + j0;
#pragma unroll
            for (int q = 0; q < 32; q += 4)
              *reinterpret_cast<float4*>(bd + q) = make_float4(bv[q], bv[q + 1], bv[q + 2], bv[q + 3]);
            if (ns.Bsb) {
              // super-block = block: row kb*BS + i of Bsb is row i of B
              __nv_bfloat16* d = ns.Bsb + (static_cast<int64_t>(kb) * BS + i) * ns.sb + j0;
#pragma unroll
              for (int q = 0; q < 32; q += 8)
                *reinterpret_cast<uint4*>(d + q) =
                    make_uint4(pack_bf16x2(bv[q], bv[q + 1]), pack_bf16x2(bv[q + 2], bv[q + 3]),
                               pack_bf16x2(bv[q + 4], bv[q + 5]), pack_bf16x2(bv[q + 6], bv[q + 7]));
            }
            if (ns.BsbT) {
              // row kb*BS + j of BsbT is column j of B: the warp's 32 rows i
              // are 32 consecutive entries of it
#pragma unroll
              for (int q = 0; q < 32; ++q)
                ns.BsbT[(static_cast<int64_t>(kb) * BS + j0 + q) * ns.sb + i] = __float2bfloat16_rn(bv[q]);
            }
          }
        }
      }
      tc_fence_before();
    } else {
      if (warp == 8 && lane == 0) {
        // -------------------------------------------------------- MMA issuer
        constexpr uint32_t idesc = idesc_bf16_f32(128, NT, false, true);
        for (int kc = 0; kc < NK; ++kc, ++gc) {
          const int buf = gc & 1;
          if (ok) ok = mbar_wait(&cvt_full[buf], static_cast<uint32_t>((gc >> 1) & 1), timeout_ns, abort_flag);
          if (ok) {
            tc_fence_after();
            const uint32_t a_hi = smem_u32(smem + buf * Cfg::BUF), a_lo = a_hi + Cfg::A_BOX;
            const uint32_t b_hi = a_lo + Cfg::A_BOX, b_lo = b_hi + Cfg::B_BOX;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ahd = smem_desc_sw128(a_hi + kk * 32, 16, 1024);
              const uint64_t ald = smem_desc_sw128(a_lo + kk * 32, 16, 1024);
              const uint64_t bhd = smem_desc_sw128(b_hi + kk * 2048, 8192, 1024);
              const uint64_t bld = smem_desc_sw128(b_lo + kk * 2048, 8192, 1024);
              mma_bf16_f32(tmem, ahd, bhd, idesc, (kc | kk) != 0 ? 1u : 0u);
              mma_bf16_f32(tmem, ahd, bld, idesc, 1u);
              mma_bf16_f32(tmem, ald, bhd, idesc, 1u);
            }
          }
          mma_commit(&mma_done[buf]);
        }
        mma_commit(acc_full);
      } else {
        gc += NK;
      }
    }
    // the next product reads every CTA's tile of S_{s+1}
    if (s < k) {
      cluster_sync();
      tc_fence_after();
    }
  }

  // every MMA has completed before TMEM is freed
  if (warp == 8 && lane == 0) {
    mma_commit(drain);
    volatile int never = 0;
    mbar_wait(drain, 0, timeout_ns, &never);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, NT);
  }
}

}  // namespace poetx
