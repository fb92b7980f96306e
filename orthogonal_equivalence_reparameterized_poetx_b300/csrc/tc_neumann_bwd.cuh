// Backward of the truncated-Neumann blocks in one launch, with the products
// on the tensor cores (used for 128-wide blocks; written for 128, 256, 512).
//
// With B = sum_p c_p Q^p (c_0 = 1, c_1..c_k = 2, c_{k+1} = 1; the Horner
// form of "POET-X: Memory-efficient LLM Training by Scaling Orthogonal
// Transformation", Methodologie §4) and G = dL/dB, the chain rule gives
//   dL/dQ = sum_{p=1}^{k+1} c_p F_p,   F_p = sum_{a+c=p-1} P^a G P^c,  P = Q^T.
// The terms obey F_1 = G, F_{s+1} = P F_s + G P^s, so with M_s = G P^{s-1}:
//   stage s = 1..k:  M_{s+1} = M_s P,  F_{s+1} = P F_s + M_{s+1},
// two products per stage and k stages.  The packed gradient of the strict
// upper triangle is then g_ij = dL/dQ[i][j] - dL/dQ[j][i].
//
// Same organisation as the Neumann builder: one cluster per block, one CTA
// per 128 x NT tile (NT = min(b, 256)), fp32-grade split-bf16 tcgen05
// products with the operands split by converter warps straight from L2, and
// a cluster barrier after every stage.  M_s P reads M_s (K-major) and Q
// (K-major, since P = Q^T); P F_s reads Q (MN-major) and F_s (MN-major).
// Each CTA keeps its tile of dL/dQ in global scratch and packs the entries
// i < j of its tile at the end, reading the transposed entries of the other
// tiles after a cluster barrier.
#pragma once

#include "ptx.cuh"
#include "simt.cuh"
#include "tc_f32gemm.cuh"
#include "tc_neumann.cuh"

namespace poetx {

struct NeumannBwdSide {
  const float* G;  // dL/dB per block, b x b fp32
  const float* Q;  // the unpacked skew matrices (params)
  float* scratch;  // five b x b fp32 matrices per block: F (2), M (2), dL/dQ
  int64_t scratch_stride;  // floats between the five scratch matrices
  SideGeom s;
  float* dGen;
};

template <int BS>
__global__ void __cluster_dims__(NeuCfg<BS>::C, 1, 1) __launch_bounds__(288, 1)
    tc_neumann_bwd_kernel(const NeumannBwdSide first, const NeumannBwdSide second, int k,
                          int accumulate, uint64_t timeout_ns) {
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
  const NeumannBwdSide& ns = is_first ? first : second;
  const int kb = is_first ? kg : kg - first.s.nblk;
  const int rank = static_cast<int>(cluster_ctarank());
  const int row0 = 128 * (rank % RS), col0 = NT * (rank / RS);
  const int sz = block_size(ns.s, kb);
  const int64_t base = static_cast<int64_t>(kb) * BS * BS;
  const float* const Gk = ns.G + base;
  const float* const Qk = ns.Q + base;
  float* const F0 = ns.scratch + base;
  float* const F1 = F0 + ns.scratch_stride;
  float* const M0 = F1 + ns.scratch_stride;
  float* const M1 = M0 + ns.scratch_stride;
  float* const GQ = M1 + ns.scratch_stride;

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
  griddep_enter();

  // epilogue thread mapping: row i of the tile, columns hh * NT/2 + [0, NT/2)
  const int gq = warp & 3, hh = warp >> 2;
  constexpr int HC = NT / 2;
  const int ei = row0 + gq * 32 + lane;

  // dL/dQ tile = c_1 F_1 = 2 G
  if (warp < 8) {
#pragma unroll 1
    for (int c32 = 0; c32 < HC / 32; ++c32) {
      const int j0 = col0 + hh * HC + c32 * 32;
      const float* g = Gk + static_cast<int64_t>(ei) * BS + j0;
      float* o = GQ + static_cast<int64_t>(ei) * BS + j0;
#pragma unroll
      for (int q = 0; q < 32; q += 4) {
        const float4 a = __ldcg(reinterpret_cast<const float4*>(g + q));
        *reinterpret_cast<float4*>(o + q) = make_float4(2.f * a.x, 2.f * a.y, 2.f * a.z, 2.f * a.w);
      }
    }
  }

  int gc = 0;  // K chunks issued so far: buffer and phase
  int pi = 0;  // products completed so far: accumulator phase
  bool ok = true;
  for (int s = 1; s <= k; ++s) {
    const float* Fs = (s == 1) ? Gk : ((s & 1) ? F1 : F0);   // F_s
    const float* Ms = (s == 1) ? Gk : ((s & 1) ? M1 : M0);   // M_s
    float* Fn = (s & 1) ? F0 : F1;                            // F_{s+1}
    float* Mn = (s & 1) ? M0 : M1;                            // M_{s+1}
    const float cn = (s == k) ? 1.f : 2.f;                    // c_{s+1}
    // two products: y = 0: M_{s+1} = M_s P; y = 1: F_{s+1} = P F_s + M_{s+1}
#pragma unroll 1
    for (int y = 0; y < 2; ++y, ++pi) {
      if (warp < 8) {
        const int t = static_cast<int>(threadIdx.x);
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
            if (y == 0) {
              // A(m, j) = M_s[row0 + m][kc*64 + j], B(n, j) = P[j][n] = Q[col0 + n][kc*64 + j]
              nb_convert_kmajor<128>(Ms + static_cast<int64_t>(row0) * BS + kc * 64, BS, ah, al, t);
              nb_convert_kmajor<NT>(Qk + static_cast<int64_t>(col0) * BS + kc * 64, BS, bh, bl, t);
            } else {
              // A(m, j) = P[m][j] = Q[kc*64 + j][row0 + m], B(n, j) = F_s[kc*64 + j][col0 + n]
              nb_convert_mnmajor<128>(Qk + static_cast<int64_t>(kc * 64) * BS + row0, BS, ah, al, t);
              nb_convert_mnmajor<NT>(Fs + static_cast<int64_t>(kc * 64) * BS + col0, BS, bh, bl, t);
            }
            fence_proxy_async_smem();  // generic-proxy stores -> visible to the tensor cores
          }
          mbar_arrive(&cvt_full[buf]);
        }
        // ---------------------------------------------------------- epilogue
        if (ok) ok = mbar_wait(acc_full, static_cast<uint32_t>(pi & 1), timeout_ns, abort_flag);
        tc_fence_after();
        if (ok) {
#pragma unroll 1
          for (int c32 = 0; c32 < HC / 32; ++c32) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(gq * 32) << 16) + hh * HC + c32 * 32, v);
            tmem_ld_wait();
            const int64_t off = static_cast<int64_t>(ei) * BS + col0 + hh * HC + c32 * 32;
            if (y == 0) {
#pragma unroll
              for (int q = 0; q < 32; q += 4)
                *reinterpret_cast<float4*>(Mn + off + q) =
                    make_float4(__uint_as_float(v[q]), __uint_as_float(v[q + 1]),
                                __uint_as_float(v[q + 2]), __uint_as_float(v[q + 3]));
            } else {
              // this thread wrote the same entries of M_{s+1} in the first product
#pragma unroll
              for (int q = 0; q < 32; q += 4) {
                const float4 m = *reinterpret_cast<const float4*>(Mn + off + q);
                const float4 a = *reinterpret_cast<const float4*>(GQ + off + q);
                float4 f;
                f.x = __uint_as_float(v[q]) + m.x;
                f.y = __uint_as_float(v[q + 1]) + m.y;
                f.z = __uint_as_float(v[q + 2]) + m.z;
                f.w = __uint_as_float(v[q + 3]) + m.w;
                if (s < k) *reinterpret_cast<float4*>(Fn + off + q) = f;
                *reinterpret_cast<float4*>(GQ + off + q) =
                    make_float4(fmaf(cn, f.x, a.x), fmaf(cn, f.y, a.y), fmaf(cn, f.z, a.z),
                                fmaf(cn, f.w, a.w));
              }
            }
          }
        }
        tc_fence_before();
      } else {
        if (warp == 8 && lane == 0) {
          // ------------------------------------------------------ MMA issuer
          const uint32_t idesc = (y == 0) ? idesc_bf16_f32(128, NT, false, false)
                                          : idesc_bf16_f32(128, NT, true, true);
          for (int kc = 0; kc < NK; ++kc, ++gc) {
            const int buf = gc & 1;
            if (ok) ok = mbar_wait(&cvt_full[buf], static_cast<uint32_t>((gc >> 1) & 1), timeout_ns, abort_flag);
            if (ok) {
              tc_fence_after();
              const uint32_t a_hi = smem_u32(smem + buf * Cfg::BUF), a_lo = a_hi + Cfg::A_BOX;
              const uint32_t b_hi = a_lo + Cfg::A_BOX, b_lo = b_hi + Cfg::B_BOX;
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                uint64_t ahd, ald, bhd, bld;
                if (y == 0) {  // both K-major
                  ahd = smem_desc_sw128(a_hi + kk * 32, 16, 1024);
                  ald = smem_desc_sw128(a_lo + kk * 32, 16, 1024);
                  bhd = smem_desc_sw128(b_hi + kk * 32, 16, 1024);
                  bld = smem_desc_sw128(b_lo + kk * 32, 16, 1024);
                } else {       // both MN-major: 16 K rows = 2 KB per step
                  ahd = smem_desc_sw128(a_hi + kk * 2048, 8192, 1024);
                  ald = smem_desc_sw128(a_lo + kk * 2048, 8192, 1024);
                  bhd = smem_desc_sw128(b_hi + kk * 2048, 8192, 1024);
                  bld = smem_desc_sw128(b_lo + kk * 2048, 8192, 1024);
                }
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
    }
    // the next stage reads every CTA's tiles of F_{s+1} and M_{s+1}; the
    // pack reads every CTA's tile of dL/dQ
    cluster_sync();
    tc_fence_after();
  }

  // packed gradient: entries (i, j), i < j < sz, of this tile; eight entries'
  // loads in flight per thread
  if (warp < 8) {
    float* out = ns.dGen + static_cast<int64_t>(kb) * BS * (BS - 1) / 2;
    const int t = static_cast<int>(threadIdx.x);
    for (int e0 = t; e0 < 128 * NT; e0 += 256 * 8) {
      float v[8], old[8];
      int64_t o[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int e = e0 + 256 * u;
        const int i = row0 + e / NT, j = col0 + e % NT;
        o[u] = -1;
        v[u] = old[u] = 0.f;
        if (e < 128 * NT && i < j && j < sz) {
          o[u] = i * sz - i * (i + 1) / 2 + (j - i - 1);
          v[u] = __ldcg(GQ + static_cast<int64_t>(i) * BS + j) - __ldcg(GQ + static_cast<int64_t>(j) * BS + i);
          if (accumulate) old[u] = out[o[u]];
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (o[u] >= 0) out[o[u]] = old[u] + v[u];
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
