// CUDA-core kernels of the POET-X layer: the fp32 path, the block builder,
// gradient reduction/packing, permutation gathers and the merge.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

#include "ptx.cuh"

namespace poetx {

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// ------------------------------------------------------------------ SIMT GEMM
// C[z](i,j) = alpha * sum_k A[z](i,k) B[z](k,j) + beta * C[z](i,j), fp32 accumulation.
// Element (i,k) of A[z] is at A[z*bsA + i*sAm + k*sAk]; likewise B and C, so
// any operand may be a transposed or strided view.
struct SimtGemmArgs {
  int M, N, K, batch;
  const void* A;
  int64_t sAm, sAk, bsA;
  const void* B;
  int64_t sBk, sBn, bsB;
  void* C;
  int64_t sCm, sCn, bsC;
  float alpha, beta;
};

template <typename TA, typename TB, typename TC>
__global__ void __launch_bounds__(256) simt_gemm_kernel(const SimtGemmArgs g) {
  griddep_enter();
  __shared__ __align__(16) float As[16][68];
  __shared__ __align__(16) float Bs[16][68];
  const int z = blockIdx.z;
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  const TA* A = reinterpret_cast<const TA*>(g.A) + z * g.bsA;
  const TB* B = reinterpret_cast<const TB*>(g.B) + z * g.bsB;
  TC* C = reinterpret_cast<TC*>(g.C) + z * g.bsC;
  const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
  const bool a_k_contig = (g.sAk == 1);
  const bool b_n_contig = (g.sBn == 1);
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  for (int k0 = 0; k0 < g.K; k0 += 16) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int idx = tid + 256 * e;
      int mm, kk;
      if (a_k_contig) mm = idx / 16, kk = idx % 16;
      else mm = idx % 64, kk = idx / 64;
      const int gm = m0 + mm, gk = k0 + kk;
      float v = 0.f;
      if (gm < g.M && gk < g.K) v = to_f32(A[gm * g.sAm + gk * g.sAk]);
      As[kk][mm] = v;
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int idx = tid + 256 * e;
      int kk, nn;
      if (b_n_contig) kk = idx / 64, nn = idx % 64;
      else kk = idx % 16, nn = idx / 16;
      const int gk = k0 + kk, gn = n0 + nn;
      float v = 0.f;
      if (gk < g.K && gn < g.N) v = to_f32(B[gk * g.sBk + gn * g.sBn]);
      Bs[kk][nn] = v;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      const float4 a = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
      const float4 b = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
      const float av[4] = {a.x, a.y, a.z, a.w};
      const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int gm = m0 + ty * 4 + i;
    if (gm >= g.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int gn = n0 + tx * 4 + j;
      if (gn >= g.N) continue;
      TC* c = C + gm * g.sCm + gn * g.sCn;
      float v = g.alpha * acc[i][j];
      if (g.beta != 0.f) v = fmaf(g.beta, to_f32(*c), v);
      *c = from_f32<TC>(v);
    }
  }
}

// Same contraction with 128 x 128 output tiles for large M and N: 256 threads,
// each owning an 8 x 8 sub-tile (rows ty*4 + {0..3} and 64 + ty*4 + {0..3},
// columns likewise), k-slices of 8 double-buffered in shared memory, so every
// 64 FMAs cost four 16-byte shared loads.
template <typename TA, typename TB, typename TC>
__global__ void __launch_bounds__(256) simt_gemm128_kernel(const SimtGemmArgs g) {
  griddep_enter();
  __shared__ __align__(16) float As[2][8][128];
  __shared__ __align__(16) float Bs[2][8][128];
  const int z = blockIdx.z;
  const int m0 = blockIdx.y * 128, n0 = blockIdx.x * 128;
  const TA* A = reinterpret_cast<const TA*>(g.A) + z * g.bsA;
  const TB* B = reinterpret_cast<const TB*>(g.B) + z * g.bsB;
  TC* C = reinterpret_cast<TC*>(g.C) + z * g.bsC;
  const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
  const bool a_k_contig = (g.sAk == 1);
  const bool b_n_contig = (g.sBn == 1);
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
  float ra[4], rb[4];
  auto load = [&](int k0) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int idx = tid + 256 * e;  // 0..1023 over 128 x 8
      int mm, kk;
      if (a_k_contig) mm = idx / 8, kk = idx % 8;
      else mm = idx % 128, kk = idx / 128;
      const int gm = m0 + mm, gk = k0 + kk;
      ra[e] = (gm < g.M && gk < g.K) ? to_f32(A[gm * g.sAm + gk * g.sAk]) : 0.f;
      int kb, nn;
      if (b_n_contig) kb = idx / 128, nn = idx % 128;
      else kb = idx % 8, nn = idx / 8;
      const int gk2 = k0 + kb, gn = n0 + nn;
      rb[e] = (gk2 < g.K && gn < g.N) ? to_f32(B[gk2 * g.sBk + gn * g.sBn]) : 0.f;
    }
  };
  auto store = [&](int buf) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int idx = tid + 256 * e;
      int mm, kk;
      if (a_k_contig) mm = idx / 8, kk = idx % 8;
      else mm = idx % 128, kk = idx / 128;
      As[buf][kk][mm] = ra[e];
      int kb, nn;
      if (b_n_contig) kb = idx / 128, nn = idx % 128;
      else kb = idx % 8, nn = idx / 8;
      Bs[buf][kb][nn] = rb[e];
    }
  };
  load(0);
  store(0);
  __syncthreads();
  int buf = 0;
  for (int k0 = 0; k0 < g.K; k0 += 8) {
    const bool more = k0 + 8 < g.K;
    if (more) load(k0 + 8);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 4]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][kk][64 + ty * 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * 4]);
      const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][kk][64 + tx * 4]);
      const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    if (more) {
      store(buf ^ 1);
      __syncthreads();
      buf ^= 1;
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int gm = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
    if (gm >= g.M) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int gn = n0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + (j - 4));
      if (gn >= g.N) continue;
      TC* c = C + gm * g.sCm + gn * g.sCn;
      float v = g.alpha * acc[i][j];
      if (g.beta != 0.f) v = fmaf(g.beta, to_f32(*c), v);
      *c = from_f32<TC>(v);
    }
  }
}

// ------------------------------------------------------------------ gathers
// out[r][j] = in[r][idx[j]] for `rows` rows of d elements (row-local feature
// permutation).  A CTA stages `rows_per_iter` consecutive rows (one
// contiguous span) in shared memory with 16-byte loads, then writes each
// permuted row with 16-byte stores; the index vector of an output chunk is
// loaded once and reused for every staged row.  Global traffic is one
// coalesced read and one coalesced write per element.  d must be a multiple
// of 16 / sizeof(T) (checked by the caller).
template <typename T>
__global__ void __launch_bounds__(256) gather_cols_kernel(const T* __restrict__ in,
                                                          T* __restrict__ out,
                                                          const int32_t* __restrict__ idx,
                                                          int64_t rows, int d, int rows_per_iter) {
  griddep_enter();
  extern __shared__ __align__(16) uint8_t gsm[];
  T* buf = reinterpret_cast<T*>(gsm);
  uint4* buf4 = reinterpret_cast<uint4*>(gsm);
  constexpr int VEC = 16 / sizeof(T);
  const int vpr = d / VEC;
  for (int64_t r0 = static_cast<int64_t>(blockIdx.x) * rows_per_iter; r0 < rows;
       r0 += static_cast<int64_t>(gridDim.x) * rows_per_iter) {
    const int nr = static_cast<int>(min(static_cast<int64_t>(rows_per_iter), rows - r0));
    const uint4* src = reinterpret_cast<const uint4*>(in + r0 * d);
    for (int v = threadIdx.x; v < nr * vpr; v += blockDim.x) buf4[v] = src[v];
    __syncthreads();
    for (int c = threadIdx.x; c < vpr; c += blockDim.x) {
      int id[VEC];
#pragma unroll
      for (int q = 0; q < VEC; ++q) id[q] = __ldg(idx + c * VEC + q);
      for (int rr = 0; rr < nr; ++rr) {
        uint4 o;
        if constexpr (sizeof(T) == 2) {
          const uint16_t* row = reinterpret_cast<const uint16_t*>(buf) + rr * d;
          uint32_t w[4];
#pragma unroll
          for (int q = 0; q < 4; ++q)
            w[q] = static_cast<uint32_t>(row[id[2 * q]]) |
                   (static_cast<uint32_t>(row[id[2 * q + 1]]) << 16);
          o = make_uint4(w[0], w[1], w[2], w[3]);
        } else {
          const uint32_t* row = reinterpret_cast<const uint32_t*>(buf) + rr * d;
          o = make_uint4(row[id[0]], row[id[1]], row[id[2]], row[id[3]]);
        }
        reinterpret_cast<uint4*>(out + (r0 + rr) * d)[c] = o;
      }
    }
    __syncthreads();
  }
}

// bf16 gather on persistent CTAs with rows staged by bulk copies:
// out[r][j] = in[r][idx[j]].  CTA c takes blocks of `rb` rows c, c + G, ...
// (G = gridDim.x) and keeps two blocks in flight: while its 256 threads
// gather block k from one shared buffer (random 2-byte reads, 16-byte
// coalesced stores), block k + 1 is landing in the other.  Thread t always
// produces the 16-byte output chunks t, t + 256, ... of a row, so it keeps
// their indices in registers when a row has at most KREG * 256 chunks.
// NARROW (rows of fewer than 256 chunks that divide 256: d = 8, 16, ...,
// 1024; KREG = 1) takes 256 / vpr rows at a time: thread t produces chunk
// t % vpr of rows t / vpr, t / vpr + 256 / vpr, ... of the block.
// Waits are bounded; on a timeout the CTA records it and returns.
template <int KREG, bool NARROW>
__global__ void __launch_bounds__(256, 3) gather_rows_pipelined_kernel(const uint16_t* __restrict__ in,
                                                                    uint4* __restrict__ out,
                                                                    const int32_t* __restrict__ idx,
                                                                    int64_t rows, int d, int rb,
                                                                    uint64_t timeout_ns) {
  extern __shared__ __align__(16) uint8_t gsm[];
  const size_t buf_bytes = static_cast<size_t>(rb) * d * 2;
  uint64_t* full = reinterpret_cast<uint64_t*>(gsm + 2 * buf_bytes);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(full + 2);
  const int vpr = d / 8;  // 16-byte output chunks per row
  const int64_t nblocks = (rows + rb - 1) / rb;
  const int tid = threadIdx.x;
  if (tid == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  griddep_enter();
  auto issue = [&](int64_t k, int s) {
    const int64_t b = blockIdx.x + k * gridDim.x;
    if (b >= nblocks) return;
    const int nr = static_cast<int>(min(static_cast<int64_t>(rb), rows - b * rb));
    const uint32_t rowb = static_cast<uint32_t>(d) * 2;
    // the block's rows are contiguous in memory: one copy for all of them
    mbar_arrive_expect_tx(&full[s], rowb * nr);
    bulk_load(gsm + s * buf_bytes, in + b * rb * static_cast<int64_t>(d), rowb * nr, &full[s]);
  };
  if (tid == 0) {
    issue(0, 0);
    issue(1, 1);
  }
  // rows per pass (narrow rows) and this thread's chunk indices
  static_assert(!NARROW || KREG == 1, "narrow rows: one chunk per thread");
  const int rpp = NARROW ? 256 / vpr : 1;
  const bool in_regs = NARROW || vpr <= KREG * 256;
  int4 ia[KREG], ib[KREG];
#pragma unroll
  for (int q = 0; q < KREG; ++q) {
    const int c = NARROW ? tid % vpr : tid + 256 * q;
    if (in_regs && c < vpr) {
      ia[q] = __ldg(reinterpret_cast<const int4*>(idx) + 2 * c);
      ib[q] = __ldg(reinterpret_cast<const int4*>(idx) + 2 * c + 1);
    } else {
      ia[q] = ib[q] = make_int4(0, 0, 0, 0);
    }
  }
  int64_t kfail = -1;
  for (int64_t k = 0;; ++k) {
    const int64_t b = blockIdx.x + k * gridDim.x;
    if (b >= nblocks) break;
    const int s = static_cast<int>(k & 1);
    const bool ok = mbar_wait(&full[s], static_cast<uint32_t>((k >> 1) & 1), timeout_ns, abort_flag);
    if (__syncthreads_or(!ok)) {  // every thread leaves at the same block
      kfail = k;
      break;
    }
    const int nr = static_cast<int>(min(static_cast<int64_t>(rb), rows - b * rb));
    const uint16_t* buf = reinterpret_cast<const uint16_t*>(gsm + s * buf_bytes);
    if constexpr (NARROW) {
      const int c = tid % vpr;
      const int4 i0 = ia[0], i1 = ib[0];
      for (int r = tid / vpr; r < nr; r += rpp) {
        const uint16_t* row = buf + static_cast<size_t>(r) * d;
        out[(b * rb + r) * static_cast<int64_t>(vpr) + c] =
            make_uint4(row[i0.x] | (static_cast<uint32_t>(row[i0.y]) << 16),
                       row[i0.z] | (static_cast<uint32_t>(row[i0.w]) << 16),
                       row[i1.x] | (static_cast<uint32_t>(row[i1.y]) << 16),
                       row[i1.z] | (static_cast<uint32_t>(row[i1.w]) << 16));
      }
    }
    for (int r = 0; r < (NARROW ? 0 : nr); ++r) {
      const uint16_t* row = buf + static_cast<size_t>(r) * d;
      uint4* orow = out + (b * rb + r) * static_cast<int64_t>(vpr);
      if (in_regs) {
#pragma unroll
        for (int q = 0; q < KREG; ++q) {
          const int c = tid + 256 * q;
          if (c < vpr) {
            const int4 i0 = ia[q], i1 = ib[q];
            orow[c] = make_uint4(row[i0.x] | (static_cast<uint32_t>(row[i0.y]) << 16),
                                 row[i0.z] | (static_cast<uint32_t>(row[i0.w]) << 16),
                                 row[i1.x] | (static_cast<uint32_t>(row[i1.y]) << 16),
                                 row[i1.z] | (static_cast<uint32_t>(row[i1.w]) << 16));
          }
        }
      } else {
        for (int c = tid; c < vpr; c += 256) {
          const int4 i0 = __ldg(reinterpret_cast<const int4*>(idx) + 2 * c);
          const int4 i1 = __ldg(reinterpret_cast<const int4*>(idx) + 2 * c + 1);
          orow[c] = make_uint4(row[i0.x] | (static_cast<uint32_t>(row[i0.y]) << 16),
                               row[i0.z] | (static_cast<uint32_t>(row[i0.w]) << 16),
                               row[i1.x] | (static_cast<uint32_t>(row[i1.y]) << 16),
                               row[i1.z] | (static_cast<uint32_t>(row[i1.w]) << 16));
        }
      }
    }
    __syncthreads();  // every thread is done with buffer s
    if (tid == 0) issue(k + 2, s);
  }
  // after a timeout, blocks kfail and kfail + 1 may still be landing: wait
  // for them (bounded) before the CTA's shared memory is released
  if (tid == 0 && kfail >= 0) {
    volatile int never = 0;
    for (int64_t k = kfail; k < kfail + 2; ++k)
      if (blockIdx.x + k * gridDim.x < nblocks)
        mbar_wait(&full[k & 1], static_cast<uint32_t>((k >> 1) & 1), timeout_ns, &never);
  }
  __syncthreads();
}

// bf16 version with rows staged in interleaved pairs: shared word c of pair p
// holds (row 2p)[c] in its low half and (row 2p+1)[c] in its high half, so one
// random 4-byte shared-memory read serves both rows (half the bank-conflicted
// reads of a per-row gather).  `pairs_per_iter` pairs (2 rows each) are
// staged per iteration; an odd last row pairs with zeros and is not stored.
__global__ void __launch_bounds__(256) gather_cols_bf16x2_kernel(const uint4* __restrict__ in,
                                                                 uint4* __restrict__ out,
                                                                 const int32_t* __restrict__ idx,
                                                                 int64_t rows, int d,
                                                                 int pairs_per_iter) {
  griddep_enter();
  extern __shared__ __align__(16) uint8_t gsm[];
  uint32_t* w = reinterpret_cast<uint32_t*>(gsm);
  const int vpr = d / 8;  // 16-byte vectors per row
  const int64_t rows_per_iter = 2 * static_cast<int64_t>(pairs_per_iter);
  for (int64_t r0 = blockIdx.x * rows_per_iter; r0 < rows; r0 += gridDim.x * rows_per_iter) {
    const int nr = static_cast<int>(min(rows_per_iter, rows - r0));
    const int np = (nr + 1) / 2;
    // four iterations' loads in flight before any shared-memory store
    const int total = np * vpr;
    for (int v0 = threadIdx.x; v0 < total; v0 += 4 * blockDim.x) {
      uint4 a[4], b[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int v = v0 + u * blockDim.x;
        a[u] = b[u] = make_uint4(0, 0, 0, 0);
        if (v < total) {
          const int p = v / vpr, c = v - p * vpr;
          const int64_t ra = r0 + 2 * p;
          a[u] = in[ra * vpr + c];
          if (2 * p + 1 < nr) b[u] = in[(ra + 1) * vpr + c];
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int v = v0 + u * blockDim.x;
        if (v < total) {
          const int p = v / vpr, c = v - p * vpr;
          uint4* dst = reinterpret_cast<uint4*>(w + static_cast<int64_t>(p) * d + 8 * c);
          dst[0] = make_uint4(__byte_perm(a[u].x, b[u].x, 0x5410), __byte_perm(a[u].x, b[u].x, 0x7632),
                              __byte_perm(a[u].y, b[u].y, 0x5410), __byte_perm(a[u].y, b[u].y, 0x7632));
          dst[1] = make_uint4(__byte_perm(a[u].z, b[u].z, 0x5410), __byte_perm(a[u].z, b[u].z, 0x7632),
                              __byte_perm(a[u].w, b[u].w, 0x5410), __byte_perm(a[u].w, b[u].w, 0x7632));
        }
      }
    }
    __syncthreads();
    for (int c = threadIdx.x; c < vpr; c += blockDim.x) {
      const int4 i0 = __ldg(reinterpret_cast<const int4*>(idx) + 2 * c);
      const int4 i1 = __ldg(reinterpret_cast<const int4*>(idx) + 2 * c + 1);
      for (int p = 0; p < np; ++p) {
        const uint32_t* pw = w + static_cast<int64_t>(p) * d;
        const uint32_t q0 = pw[i0.x], q1 = pw[i0.y], q2 = pw[i0.z], q3 = pw[i0.w];
        const uint32_t q4 = pw[i1.x], q5 = pw[i1.y], q6 = pw[i1.z], q7 = pw[i1.w];
        const int64_t ra = r0 + 2 * p;
        out[ra * vpr + c] = make_uint4(__byte_perm(q0, q1, 0x5410), __byte_perm(q2, q3, 0x5410),
                                       __byte_perm(q4, q5, 0x5410), __byte_perm(q6, q7, 0x5410));
        if (2 * p + 1 < nr)
          out[(ra + 1) * vpr + c] =
              make_uint4(__byte_perm(q0, q1, 0x7632), __byte_perm(q2, q3, 0x7632),
                         __byte_perm(q4, q5, 0x7632), __byte_perm(q6, q7, 0x7632));
      }
    }
    __syncthreads();
  }
}

// Scalar version for widths that are not a multiple of 16 bytes.
template <typename T>
__global__ void __launch_bounds__(256) gather_cols_scalar_kernel(const T* __restrict__ in,
                                                                 T* __restrict__ out,
                                                                 const int32_t* __restrict__ idx,
                                                                 int64_t rows, int d) {
  griddep_enter();
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x)
    for (int c = threadIdx.x; c < d; c += blockDim.x) out[r * d + c] = in[r * d + __ldg(idx + c)];
}

// out[i][j] = convert(in[ridx[i]][cidx[j]]), both row-major with `cols`
// elements per row.  Used for the weight pre-merge (W0' = W0[pi_R][:, pi_P])
// and for re-basing the merged weight under new permutations.
template <typename TI, typename TO>
__global__ void __launch_bounds__(256) gather2d_kernel(const TI* __restrict__ in, TO* __restrict__ out,
                                                       const int32_t* __restrict__ ridx,
                                                       const int32_t* __restrict__ cidx, int rows,
                                                       int cols) {
  for (int i = blockIdx.x; i < rows; i += gridDim.x) {
    const TI* src = in + static_cast<int64_t>(__ldg(ridx + i)) * cols;
    TO* dst = out + static_cast<int64_t>(i) * cols;
    for (int j = threadIdx.x; j < cols; j += blockDim.x)
      dst[j] = from_f32<TO>(to_f32(src[__ldg(cidx + j)]));
  }
}

// ------------------------------------------------------------------ builder
// Geometry of one side (R on the m side, P on the n side): nblk blocks of b,
// the last of size `last` (= b unless b does not divide d).
struct SideGeom {
  int d, b, nblk, last;
};

__device__ __forceinline__ int block_size(const SideGeom& s, int k) {
  return (k == s.nblk - 1) ? s.last : s.b;
}

// Unpacks the strict upper triangle of block k = blockIdx.x into Q (b x b,
// zero padded beyond the block's size) and writes A = I - Q (identity on the
// padding).  One warp per row i (grid.y covers rows 8 at a time); entry
// (i, j), i < j, of a block of size sz sits at i*sz - i(i+1)/2 + (j-i-1).
__global__ void __launch_bounds__(256) unpack_kernel(const float* __restrict__ gen, SideGeom s,
                                                     float* __restrict__ Q, float* __restrict__ A) {
  const int k = blockIdx.x;
  const int i = blockIdx.y * 8 + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (i >= s.b) return;
  const int sz = block_size(s, k);
  const float* g = gen + static_cast<int64_t>(k) * s.b * (s.b - 1) / 2;
  float* Qr = Q + (static_cast<int64_t>(k) * s.b + i) * s.b;
  float* Ar = A ? A + (static_cast<int64_t>(k) * s.b + i) * s.b : nullptr;
  const int row_base = i * sz - i * (i + 1) / 2 - i - 1;  // + j for j > i
  for (int j = lane; j < s.b; j += 32) {
    float q = 0.f;
    if (i < sz && j < sz) {
      if (i < j) q = g[row_base + j];
      else if (j < i) q = -g[j * sz - j * (j + 1) / 2 - j - 1 + i];
    }
    Qr[j] = q;
    if (Ar) Ar[j] = (i == j ? 1.f : 0.f) - q;
  }
}

// Register Gauss-Jordan inversion of a P x P matrix (P <= 128) by one CTA of
// P * R threads, R = min(P, 1024 / P): thread (ty, tx) owns column j = tx and
// rows i = ty + R*r (r < NR = ceil(P / R) <= 16) in registers.  No pivoting:
// the matrices inverted here are I - Q for skew Q and pivot blocks of its
// block elimination, whose symmetric parts are >= I, so every pivot has
// magnitude >= 1.  The pivot row and column are published through a
// double-buffered shared array, one barrier per pivot.  PT > 0 fixes P at
// compile time (the index arithmetic folds away); PT == 0 reads P at run time.
constexpr int kGjMaxRows = 16;

template <int PT>
struct GjShape {
  int P, R, NR;
  __device__ __forceinline__ explicit GjShape(int p_runtime)
      : P(PT > 0 ? PT : p_runtime),
        R(PT > 0 ? (PT < 1024 / PT ? PT : 1024 / PT) : min(p_runtime, 1024 / p_runtime)),
        NR((P + R - 1) / R) {}
};

template <int PT>
__device__ __forceinline__ void gj_register_invert(float (&a)[kGjMaxRows], const GjShape<PT>& sh,
                                                   int tx, int ty, float* rowbuf, float* colbuf) {
  const int P = sh.P, R = sh.R, NR = sh.NR;
#pragma unroll
  for (int r = 0; r < kGjMaxRows; ++r) {
    const int i = ty + R * r;
    if (r < NR && i < P) {
      if (i == 0) rowbuf[tx] = a[r];
      if (tx == 0) colbuf[i] = a[r];
    }
  }
  __syncthreads();
  for (int k = 0; k < P; ++k) {
    const int cur = (k & 1) * 128, nxt = 128 - cur;
    const float p = 1.0f / rowbuf[cur + k];
    const float rj = rowbuf[cur + tx] * p;
    const bool col_k = (tx == k), col_k1 = (tx == k + 1);
#pragma unroll
    for (int r = 0; r < kGjMaxRows; ++r) {
      const int i = ty + R * r;
      if (r < NR && i < P) {
        float v = a[r];
        if (i == k) v = col_k ? p : v * p;
        else if (col_k) v = -v * p;
        else v = fmaf(-colbuf[cur + i], rj, v);
        a[r] = v;
        if (i == k + 1) rowbuf[nxt + tx] = v;
        if (col_k1) colbuf[nxt + i] = v;
      }
    }
    __syncthreads();
  }
}

__device__ __forceinline__ float sel4(const float (&v)[4], int q) {
  return q == 0 ? v[0] : q == 1 ? v[1] : q == 2 ? v[2] : v[3];
}

// Same inversion with pivots taken four at a time (P % 4 == 0).  For the
// panel K = {k0..k0+3} with pivot block D = A_KK:
//   A_ij -= (A_iK D^-1) A_Kj     (i, j outside K)
//   A_Kj  = D^-1 A_Kj,  A_iK = -A_iK D^-1,  A_KK = D^-1.
// D's symmetric part stays >= I (Schur complements of I - Q), so its
// unpivoted inverse is well conditioned.  Each round: the P threads of row
// group ty = 0 invert D in registers and publish, for their row / column
// tx, c_tx = A_txK D^-1 and the new pivot-row entries D^-1 A_K,tx (and one
// of them D^-1 itself); then every element takes a rank-4 update (one
// 16-byte shared load, four FMAs).  Two barriers per four pivots.  `sm`
// holds kGj4SmemFloats floats.
constexpr int kGj4SmemFloats = 2560 + 512 + 32;

template <int PT>
__device__ __forceinline__ void gj_register_invert4(float (&a)[kGjMaxRows], const GjShape<PT>& sh,
                                                    int tx, int ty, float* sm) {
  const int P = sh.P, R = sh.R, NR = sh.NR;
  float* rowK0 = sm;          // [2][4][128]: panel rows A_Kj
  float* colK0 = sm + 1024;   // [2][128][4]: panel columns A_iK
  float* cK = sm + 2048;      // [128][4]: c_i = A_iK D^-1
  float* nrK = sm + 2560;     // [4][128]: new pivot rows D^-1 A_K*
  float* dK = sm + 3072;      // [4][4]: D^-1
#pragma unroll
  for (int r = 0; r < kGjMaxRows; ++r) {
    const int i = ty + R * r;
    if (r < NR && i < P) {
      if (i < 4) rowK0[i * 128 + tx] = a[r];
      if (tx < 4) colK0[i * 4 + tx] = a[r];
    }
  }
  __syncthreads();
  for (int k0 = 0, buf = 0; k0 < P; k0 += 4, buf ^= 1) {
    const float* rk = rowK0 + buf * 512;
    const float* ck = colK0 + buf * 512;
    const float rj[4] = {rk[tx], rk[128 + tx], rk[256 + tx], rk[384 + tx]};
    if (ty == 0) {
      float D[4][4];
#pragma unroll
      for (int p = 0; p < 4; ++p)
#pragma unroll
        for (int q = 0; q < 4; ++q) D[p][q] = rk[p * 128 + k0 + q];
#pragma unroll
      for (int p = 0; p < 4; ++p) {  // in-place unpivoted Gauss-Jordan on the 4 x 4 block
        const float pv = 1.0f / D[p][p];
#pragma unroll
        for (int q = 0; q < 4; ++q) D[p][q] = (q == p) ? pv : D[p][q] * pv;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (i == p) continue;
          const float f = D[i][p];
#pragma unroll
          for (int q = 0; q < 4; ++q) D[i][q] = (q == p) ? -f * pv : fmaf(-f, D[p][q], D[i][q]);
        }
      }
      const float4 ai = *reinterpret_cast<const float4*>(ck + tx * 4);
      float4 c;
      c.x = ai.x * D[0][0] + ai.y * D[1][0] + ai.z * D[2][0] + ai.w * D[3][0];
      c.y = ai.x * D[0][1] + ai.y * D[1][1] + ai.z * D[2][1] + ai.w * D[3][1];
      c.z = ai.x * D[0][2] + ai.y * D[1][2] + ai.z * D[2][2] + ai.w * D[3][2];
      c.w = ai.x * D[0][3] + ai.y * D[1][3] + ai.z * D[2][3] + ai.w * D[3][3];
      *reinterpret_cast<float4*>(cK + tx * 4) = c;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        nrK[q * 128 + tx] = D[q][0] * rj[0] + D[q][1] * rj[1] + D[q][2] * rj[2] + D[q][3] * rj[3];
      if (tx == 0) {
#pragma unroll
        for (int p = 0; p < 4; ++p)
#pragma unroll
          for (int q = 0; q < 4; ++q) dK[p * 4 + q] = D[p][q];
      }
    }
    const int qj = tx - k0;
    const bool colK = (qj >= 0 && qj < 4);
    __syncthreads();  // cK, nrK and dK ready
    const int k1 = k0 + 4;
    float* rkn = rowK0 + (buf ^ 1) * 512;
    float* ckn = colK0 + (buf ^ 1) * 512;
    const int qj1 = tx - k1;
    const bool colK1 = (k1 < P) && (qj1 >= 0 && qj1 < 4);
#pragma unroll
    for (int r = 0; r < kGjMaxRows; ++r) {
      const int i = ty + R * r;
      if (r < NR && i < P) {
        const int qi = i - k0;
        float v;
        if (qi >= 0 && qi < 4) {
          v = colK ? dK[qi * 4 + qj] : nrK[qi * 128 + tx];
        } else if (colK) {
          v = -cK[i * 4 + qj];
        } else {
          const float4 c = *reinterpret_cast<const float4*>(cK + i * 4);
          v = fmaf(-c.x, rj[0], fmaf(-c.y, rj[1], fmaf(-c.z, rj[2], fmaf(-c.w, rj[3], a[r]))));
        }
        a[r] = v;
        const int qi1 = i - k1;
        if (k1 < P && qi1 >= 0 && qi1 < 4) rkn[qi1 * 128 + tx] = v;
        if (colK1) ckn[i * 4 + qj1] = v;
      }
    }
    __syncthreads();  // next panel published; cK, nrK and dK free
  }
}

// Exact Cayley blocks for b <= 128, one CTA per block: unpack the packed
// generator into A = I - Q (identity on the padding of a ragged block),
// invert it in registers (M = (I - Q)^-1), and write M, B = 2M - I, Q and,
// when Bsb is given, the bf16 super-block rows of this block (B and B^T on
// the diagonal, zeros elsewhere).
struct CayleySide {
  const float* gen;
  SideGeom s;
  float* B;
  float* M;
  float* Q;
  int sb, nsb;
  __nv_bfloat16* Bsb;
  __nv_bfloat16* BsbT;
};

// Blocks [0, first.s.nblk) belong to `first`, the rest to `second` (the R and
// P sides of a layer built in one launch when their block sizes agree).
template <int PT>
__global__ void __launch_bounds__(1024) cayley_block_kernel(const CayleySide first,
                                                            const CayleySide second) {
  const bool is_first = static_cast<int>(blockIdx.x) < first.s.nblk;
  const CayleySide& cs = is_first ? first : second;
  const float* __restrict__ gen = cs.gen;
  const SideGeom s = cs.s;
  float* __restrict__ Bout = cs.B;
  float* __restrict__ Mout = cs.M;
  float* __restrict__ Qout = cs.Q;
  const int sb = cs.sb, nsb = cs.nsb;
  __nv_bfloat16* __restrict__ Bsb = cs.Bsb;
  __nv_bfloat16* __restrict__ BsbT = cs.BsbT;
  __shared__ float rowbuf[256], colbuf[256];
  __shared__ __align__(16) float gj4_sm[kGj4SmemFloats];
  extern __shared__ float bsm[];  // P x (P + 1) staging of B for the transposed writes
  const GjShape<PT> sh(s.b);
  const int P = sh.P, R = sh.R, NR = sh.NR;
  const int tx = threadIdx.x % P, ty = threadIdx.x / P;
  const int k = is_first ? static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x) - first.s.nblk;
  const int sz = block_size(s, k);
  const float* g = gen + static_cast<int64_t>(k) * P * (P - 1) / 2;
  float* Mk = Mout + static_cast<int64_t>(k) * P * P;
  float* Bk = Bout + static_cast<int64_t>(k) * P * P;
  float* Qk = Qout + static_cast<int64_t>(k) * P * P;
  float a[kGjMaxRows];
#pragma unroll
  for (int r = 0; r < kGjMaxRows; ++r) {
    const int i = ty + R * r, j = tx;
    float q = 0.f;
    if (r < NR && i < P) {
      if (i < sz && j < sz && i != j) {
        if (i < j) q = g[i * sz - i * (i + 1) / 2 + (j - i - 1)];
        else q = -g[j * sz - j * (j + 1) / 2 + (i - j - 1)];
      }
      Qk[i * P + j] = q;
    }
    a[r] = (i == j ? 1.f : 0.f) - q;
  }
  if (P % 4 == 0) gj_register_invert4<PT>(a, sh, tx, ty, gj4_sm);
  else gj_register_invert<PT>(a, sh, tx, ty, rowbuf, colbuf);
#pragma unroll
  for (int r = 0; r < kGjMaxRows; ++r) {
    const int i = ty + R * r;
    if (r < NR && i < P) {
      const float bv = 2.f * a[r] - (i == tx ? 1.f : 0.f);
      Mk[i * P + tx] = a[r];
      Bk[i * P + tx] = bv;
      if (Bsb) bsm[i * (P + 1) + tx] = bv;
    }
  }
  if (!Bsb) return;
  __syncthreads();
  // rows [k*b, k*b + b) of the super-block arrays; the last block also zeroes
  // the rows that no block owns (features beyond nblk * b).
  const int r0 = k * P;
  const int r1 = (k == s.nblk - 1) ? nsb * sb : r0 + P;
  const int c0 = r0 % sb;
  for (int e = threadIdx.x; e < (r1 - r0) * sb; e += blockDim.x) {
    const int rr = e / sb, c = e % sb;
    float v = 0.f, vt = 0.f;
    if (rr < P && c >= c0 && c < c0 + P) {
      v = bsm[rr * (P + 1) + (c - c0)];
      vt = bsm[(c - c0) * (P + 1) + rr];
    }
    const int64_t o = static_cast<int64_t>(r0 + rr) * sb + c;
    Bsb[o] = __float2bfloat16_rn(v);
    BsbT[o] = __float2bfloat16_rn(vt);
  }
}

// Inverse of the 128 x 128 diagonal sub-block of matrix z: read at
// in + z*in_bs with leading dimension in_ld, written to out likewise.
__global__ void __launch_bounds__(1024) gj_invert128_kernel(const float* in, int64_t in_bs, int in_ld,
                                                            float* out, int64_t out_bs, int out_ld) {
  __shared__ __align__(16) float gj4_sm[kGj4SmemFloats];
  const GjShape<128> sh(128);
  const int tx = threadIdx.x % 128, ty = threadIdx.x / 128;
  const float* src = in + blockIdx.x * in_bs;
  float a[kGjMaxRows];
#pragma unroll
  for (int r = 0; r < kGjMaxRows; ++r) a[r] = src[static_cast<int64_t>(ty + 8 * r) * in_ld + tx];
  gj_register_invert4<128>(a, sh, tx, ty, gj4_sm);
  float* dst = out + blockIdx.x * out_bs;
#pragma unroll
  for (int r = 0; r < kGjMaxRows; ++r) dst[static_cast<int64_t>(ty + 8 * r) * out_ld + tx] = a[r];
}

// dst[z](i,j) = alpha * src[z](i,j) (+ beta * I(i,j)) over rows x cols.
__global__ void __launch_bounds__(256) copy2d_kernel(const float* src, int64_t s_bs, int s_ld,
                                                     float* dst, int64_t d_bs, int d_ld, int rows,
                                                     int cols, float alpha, float beta_eye) {
  griddep_enter();
  const int z = blockIdx.y;
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < rows * cols; e += gridDim.x * blockDim.x) {
    const int i = e / cols, j = e % cols;
    float v = alpha * src[z * s_bs + static_cast<int64_t>(i) * s_ld + j];
    if (i == j) v += beta_eye;
    dst[z * d_bs + static_cast<int64_t>(i) * d_ld + j] = v;
  }
}

// dst[e] += alpha * src[e] for e < n.
__global__ void __launch_bounds__(256) axpy_kernel(float* __restrict__ dst, const float* __restrict__ src,
                                                   float alpha, int64_t n) {
  griddep_enter();
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < n;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x)
    dst[e] = fmaf(alpha, src[e], dst[e]);
}

// Super-block arrays for the tensor-core path.  Row r of Bsb (global output
// feature in the permuted basis) holds, in columns c of [0, sb), the entry of
// its block matrix that multiplies input feature s*sb + c (s = r / sb), or 0
// if that feature lies in another block.  BsbT holds the transposed blocks.
__global__ void __launch_bounds__(256) superblock_kernel(const float* __restrict__ B, SideGeom s,
                                                         int sb, int nsb,
                                                         __nv_bfloat16* __restrict__ Bsb,
                                                         __nv_bfloat16* __restrict__ BsbT) {
  const int64_t bb = static_cast<int64_t>(s.b) * s.b;
  const int64_t total = static_cast<int64_t>(nsb) * sb * sb;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int r = static_cast<int>(e / sb), c = static_cast<int>(e % sb);
    const int f = (r / sb) * sb + c;
    const int k = r / s.b;
    float v = 0.f, vt = 0.f;
    if (k < s.nblk && f / s.b == k) {
      const int i = r - k * s.b, j = f - k * s.b;
      v = B[k * bb + static_cast<int64_t>(i) * s.b + j];
      vt = B[k * bb + static_cast<int64_t>(j) * s.b + i];
    }
    Bsb[e] = __float2bfloat16_rn(v);
    BsbT[e] = __float2bfloat16_rn(vt);
  }
}

// Super-block array of the blocks minus the identity, D = B - I (or
// B^T - I with `transpose`), each entry split into two bf16 terms hi + lo
// with hi = bf16(v) and lo = bf16(v - hi), for the tensor-core merge.  The
// layout is that of superblock_kernel; entries outside the d x d matrix are 0.
__global__ void __launch_bounds__(256) delta_superblock_kernel(const float* __restrict__ B, SideGeom s,
                                                               int sb, int nsb, int transpose,
                                                               __nv_bfloat16* __restrict__ hi,
                                                               __nv_bfloat16* __restrict__ lo) {
  const int64_t bb = static_cast<int64_t>(s.b) * s.b;
  const int64_t total = static_cast<int64_t>(nsb) * sb * sb;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int r = static_cast<int>(e / sb), c = static_cast<int>(e % sb);
    const int f = (r / sb) * sb + c;
    const int k = r / s.b;
    float v = 0.f;
    if (r < s.d && f < s.d && f / s.b == k) {
      const int i = r - k * s.b, j = f - k * s.b;
      v = transpose ? B[k * bb + static_cast<int64_t>(j) * s.b + i]
                    : B[k * bb + static_cast<int64_t>(i) * s.b + j];
      if (r == f) v -= 1.f;
    }
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    hi[e] = h;
    lo[e] = __float2bfloat16_rn(v - __bfloat162float(h));
  }
}

// ------------------------------------------------------------------ POET-XQ
// int8 base weights with a float32 scale per row.

// out[i][j] = bf16(scale_i * code_ij), and with `lo` also the remainder
// lo[i][j] = bf16(scale_i * code_ij - out[i][j]) (out + lo is the product to
// 2^-17); eight codes per step (n % 8 == 0, so they share a row).
__global__ void __launch_bounds__(256) dequant_int8_kernel(const int8_t* __restrict__ codes,
                                                           const float* __restrict__ scales,
                                                           __nv_bfloat16* __restrict__ out,
                                                           __nv_bfloat16* __restrict__ lo, int m, int n) {
  const int64_t chunks = static_cast<int64_t>(m) * n / 8;
  for (int64_t c = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; c < chunks;
       c += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t e = c * 8;
    const float sc = scales[e / n];
    const uint2 q = *reinterpret_cast<const uint2*>(codes + e);
    uint32_t w[4], r[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t word = k < 2 ? q.x : q.y;
      const int sh = 16 * (k & 1);
      const float a = sc * static_cast<float>(static_cast<int8_t>((word >> sh) & 0xFFu));
      const float b = sc * static_cast<float>(static_cast<int8_t>((word >> (sh + 8)) & 0xFFu));
      w[k] = pack_bf16x2(a, b);
      const float ah = __bfloat162float(__ushort_as_bfloat16(static_cast<unsigned short>(w[k] & 0xFFFFu)));
      const float bh = __bfloat162float(__ushort_as_bfloat16(static_cast<unsigned short>(w[k] >> 16)));
      r[k] = pack_bf16x2(a - ah, b - bh);
    }
    *reinterpret_cast<uint4*>(out + e) = make_uint4(w[0], w[1], w[2], w[3]);
    if (lo) *reinterpret_cast<uint4*>(lo + e) = make_uint4(r[0], r[1], r[2], r[3]);
  }
}

// Row i of a quantized weight: its values are v_j = S[row_map[i]][col_map[j]]
// of a row-major source S with n columns, S = hi (+ lo when given, in fp32).
// scale_i = max_j |v_j| / 127 and code_ij = round-half-to-even(v_j / scale_i)
// clamped to [-127, 127], in float32 (IEEE division); a zero row gets scale 0
// and codes 0.  One CTA per row; the source row is staged in shared memory
// (its maximum is the maximum of the permuted row).
__global__ void __launch_bounds__(256) quantize_rows_kernel(const __nv_bfloat16* __restrict__ hi,
                                                            const __nv_bfloat16* __restrict__ lo,
                                                            const int32_t* __restrict__ row_map,
                                                            const int32_t* __restrict__ col_map, int n,
                                                            int8_t* __restrict__ codes,
                                                            float* __restrict__ scales) {
  extern __shared__ float qrow[];
  __shared__ float wmax[8];
  const int i = blockIdx.x;
  const int64_t src = static_cast<int64_t>(row_map[i]) * n;
  float mx = 0.f;
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    float v = __bfloat162float(hi[src + j]);
    if (lo) v += __bfloat162float(lo[src + j]);
    qrow[j] = v;
    mx = fmaxf(mx, fabsf(v));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (threadIdx.x % 32 == 0) wmax[threadIdx.x / 32] = mx;
  __syncthreads();
  mx = wmax[0];
  for (int w = 1; w < static_cast<int>(blockDim.x) / 32; ++w) mx = fmaxf(mx, wmax[w]);
  const float sc = mx / 127.f;
  int8_t* out = codes + static_cast<int64_t>(i) * n;
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    int q = 0;
    if (sc > 0.f) q = static_cast<int>(fminf(fmaxf(rintf(qrow[col_map[j]] / sc), -127.f), 127.f));
    out[j] = static_cast<int8_t>(q);
  }
  if (threadIdx.x == 0) scales[i] = sc;
}

// ------------------------------------------------------------------ optimizer
// AdamW on packed generators: see poetx_generator_adamw.  step_size =
// lr / (1 - beta1^t) and inv_sqrt_bc2 = 1 / sqrt(1 - beta2^t) come from the
// host (double, rounded once).
__global__ void __launch_bounds__(256) adamw_kernel(float* __restrict__ gen, const float* __restrict__ grad,
                                                    float* __restrict__ m1, float* __restrict__ m2, int64_t len,
                                                    float beta1, float beta2, float eps, float decay_factor,
                                                    float step_size, float inv_sqrt_bc2) {
  griddep_enter();
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < len;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float g = grad[e];
    const float a = fmaf(beta1, m1[e], (1.f - beta1) * g);
    const float b = fmaf(beta2, m2[e], (1.f - beta2) * g * g);
    m1[e] = a;
    m2[e] = b;
    const float denom = sqrtf(b) * inv_sqrt_bc2 + eps;
    gen[e] = gen[e] * decay_factor - step_size * (a / denom);
  }
}

// ------------------------------------------------------------------ gradients
// G[k](i,j) = sum over splits p of partial[p][s][(a - s*sb)][(c - s*sb)],
// a = k*b + i, c = k*b + j, s = a / sb, in a fixed order (deterministic).
__global__ void __launch_bounds__(256) gradred_reduce_kernel(const float* __restrict__ partial,
                                                             int64_t split_stride, int splits,
                                                             SideGeom s, int sb,
                                                             float* __restrict__ G) {
  griddep_enter();
  const int64_t bb = static_cast<int64_t>(s.b) * s.b;
  const int64_t total = static_cast<int64_t>(s.nblk) * bb;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int k = static_cast<int>(e / bb);
    const int r = static_cast<int>(e % bb);
    const int a = k * s.b + r / s.b, c = k * s.b + r % s.b;
    const int sbi = a / sb;
    const int64_t off = static_cast<int64_t>(sbi) * sb * sb +
                        static_cast<int64_t>(a - sbi * sb) * sb + (c - sbi * sb);
    float v = 0.f;
    for (int p = 0; p < splits; ++p) v += partial[p * split_stride + off];
    G[e] = v;
  }
}

// Packed generator gradient: g[(i,j)] (+)= GQ[k](i,j) - GQ[k](j,i), i < j < size,
// for block k = blockIdx.x; one warp per row i (grid.y covers rows 8 at a
// time), consecutive lanes on consecutive packed entries.
__global__ void __launch_bounds__(256) pack_grad_kernel(const float* __restrict__ GQ, SideGeom s,
                                                        float* __restrict__ out, int accumulate) {
  griddep_enter();
  const int k = blockIdx.x;
  const int i = blockIdx.y * 8 + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int sz = block_size(s, k);
  if (i >= sz - 1) return;
  const float* G = GQ + static_cast<int64_t>(k) * s.b * s.b;
  float* o = out + static_cast<int64_t>(k) * s.b * (s.b - 1) / 2 + (i * sz - i * (i + 1) / 2 - i - 1);
  for (int j = i + 1 + lane; j < sz; j += 32) {
    const float v = G[i * s.b + j] - G[j * s.b + i];
    if (accumulate) o[j] += v;
    else o[j] = v;
  }
}

// One side's operands of the Cayley backward: split partials
// ([split][super-block][128][128] for 128-wide super-blocks), M per block,
// packed output.
struct CbwdSide {
  const float* partial;
  int64_t split_stride;
  int splits;
  SideGeom s;
  const float* M;
  float* out;
};

// Cayley backward of one P x P block per CTA (P in {32, 64}, bf16 path) for
// the blocks of one or two sides (blocks [0, a.s.nblk) of side a, the rest
// of side b), fused:
//   G   = sum over token splits of the reduction partials (fixed order);
//   GQ  = 2 M^T G M^T with M = (I - Q)^-1;
//   g_ij (+)= GQ[i][j] - GQ[j][i] packed row by row (i < j < size).
// Split reduction: every thread owns one float4 of the block and sums a
// contiguous run of the splits (1024 / (P * P / 4) runs per block), eight
// splits' loads in flight; the runs are then added in ascending order.
// Products: (P/4)^2 threads own a 4 x 4 tile each; the matrices live in
// shared memory with rows padded to P + 4 floats so 16-byte loads stay
// aligned, and the second product reads T^T and M^T so both operands are
// contiguous along the loop.  A block lies on the diagonal of its 128-wide
// super-block.
constexpr int kCbwdThreads = 1024;

template <int P>
__host__ __device__ constexpr int cbwd_runs() { return kCbwdThreads / (P * P / 4); }

template <int P>
__host__ __device__ constexpr size_t cbwd_smem() {
  return static_cast<size_t>(3 * P * (P + 4) + (cbwd_runs<P>() - 1) * P * P) * 4;
}

template <int P>
__global__ void __launch_bounds__(kCbwdThreads) cayley_bwd_kernel(const CbwdSide a, const CbwdSide b,
                                                                  int accumulate) {
  griddep_enter();
  constexpr int LD = P + 4;
  constexpr int NT = kCbwdThreads;
  constexpr int E = P * P / 4;           // float4 per block
  constexpr int RUNS = cbwd_runs<P>();
  constexpr int CT = (P / 4) * (P / 4);  // threads of the matrix products
  constexpr int SB = 128;                // super-block width of the partials
  static_assert(RUNS * E == NT && P <= SB, "threads must tile the block");
  extern __shared__ __align__(16) float cbs[];
  float* Gs = cbs;             // G, then T^T
  float* Ms = cbs + P * LD;    // M, then GQ
  float* Mt = Ms + P * LD;     // M^T
  float4* run_sums = reinterpret_cast<float4*>(Mt + P * LD);  // runs 1.. [RUNS - 1][E]
  const int kg = blockIdx.x;
  const bool on_a = kg < a.s.nblk;
  const CbwdSide& side = on_a ? a : b;
  const int k = on_a ? kg : kg - a.s.nblk;
  const SideGeom s = side.s;
  const int tid = threadIdx.x;
  const int e = tid % E, run = tid / E;
  const int i = e / (P / 4), j4 = 4 * (e % (P / 4));
  const float* Mk = side.M + static_cast<int64_t>(k) * P * P;
  float4 mv = make_float4(0.f, 0.f, 0.f, 0.f);
  if (run == 0) mv = *reinterpret_cast<const float4*>(Mk + i * P + j4);
  // block k lies in super-block (k * P) / SB at diagonal offset o0
  const int sbi = (k * P) / SB, o0 = k * P - sbi * SB;
  const float* src = side.partial + static_cast<int64_t>(sbi) * SB * SB +
                     static_cast<int64_t>(o0 + i) * SB + o0 + j4;
  const int per = (side.splits + RUNS - 1) / RUNS;
  const int p0 = min(side.splits, run * per), p1 = min(side.splits, p0 + per);
  float4 g = make_float4(0.f, 0.f, 0.f, 0.f);
  constexpr int SU = 8;
  int p = p0;
  for (; p + SU <= p1; p += SU) {
    float4 w[SU];
#pragma unroll
    for (int q = 0; q < SU; ++q)
      w[q] = *reinterpret_cast<const float4*>(src + static_cast<int64_t>(p + q) * side.split_stride);
#pragma unroll
    for (int q = 0; q < SU; ++q) {
      g.x += w[q].x; g.y += w[q].y; g.z += w[q].z; g.w += w[q].w;
    }
  }
  for (; p < p1; ++p) {
    const float4 w = *reinterpret_cast<const float4*>(src + static_cast<int64_t>(p) * side.split_stride);
    g.x += w.x; g.y += w.y; g.z += w.z; g.w += w.w;
  }
  if (RUNS > 1 && run > 0) run_sums[(run - 1) * E + e] = g;
  __syncthreads();
  if (run == 0) {
#pragma unroll
    for (int r = 1; r < RUNS; ++r) {
      const float4 w = run_sums[(r - 1) * E + e];
      g.x += w.x; g.y += w.y; g.z += w.z; g.w += w.w;
    }
    *reinterpret_cast<float4*>(Gs + i * LD + j4) = g;
    *reinterpret_cast<float4*>(Ms + i * LD + j4) = mv;
    Mt[(j4 + 0) * LD + i] = mv.x;
    Mt[(j4 + 1) * LD + i] = mv.y;
    Mt[(j4 + 2) * LD + i] = mv.z;
    Mt[(j4 + 3) * LD + i] = mv.w;
  }
  __syncthreads();
  const bool mm = tid < CT;  // holds a tile of the products
  const int tr = tid / (P / 4), tc = tid % (P / 4);
  float acc[4][4];
  // T = M^T G: T[i][j] = sum_q M[q][i] G[q][j]
#pragma unroll
  for (int x = 0; x < 4; ++x)
#pragma unroll
    for (int y = 0; y < 4; ++y) acc[x][y] = 0.f;
  if (mm) {
#pragma unroll 4
    for (int q = 0; q < P; ++q) {
      const float4 av4 = *reinterpret_cast<const float4*>(Ms + q * LD + 4 * tr);
      const float4 gv4 = *reinterpret_cast<const float4*>(Gs + q * LD + 4 * tc);
      const float av[4] = {av4.x, av4.y, av4.z, av4.w}, gv[4] = {gv4.x, gv4.y, gv4.z, gv4.w};
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) acc[x][y] = fmaf(av[x], gv[y], acc[x][y]);
    }
  }
  __syncthreads();
  if (mm) {
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
      for (int y = 0; y < 4; ++y) Gs[(4 * tc + y) * LD + 4 * tr + x] = acc[x][y];  // T^T
  }
  __syncthreads();
  // GQ = 2 T M^T: GQ[i][j] = 2 sum_q T^T[q][i] M^T[q][j]
  if (mm) {
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
      for (int y = 0; y < 4; ++y) acc[x][y] = 0.f;
#pragma unroll 4
    for (int q = 0; q < P; ++q) {
      const float4 t4 = *reinterpret_cast<const float4*>(Gs + q * LD + 4 * tr);
      const float4 m4 = *reinterpret_cast<const float4*>(Mt + q * LD + 4 * tc);
      const float tv[4] = {t4.x, t4.y, t4.z, t4.w}, mw[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) acc[x][y] = fmaf(tv[x], mw[y], acc[x][y]);
    }
#pragma unroll
    for (int x = 0; x < 4; ++x)
      *reinterpret_cast<float4*>(Ms + (4 * tr + x) * LD + 4 * tc) =
          make_float4(2.f * acc[x][0], 2.f * acc[x][1], 2.f * acc[x][2], 2.f * acc[x][3]);
  }
  __syncthreads();
  // pack: one warp per row
  const int sz = block_size(s, k);
  float* o = side.out + static_cast<int64_t>(k) * P * (P - 1) / 2;
  const int warp = tid / 32, lane = tid % 32, nwarps = NT / 32;
  for (int r = warp; r < sz - 1; r += nwarps) {
    float* oi = o + (r * sz - r * (r + 1) / 2 - r - 1);
    for (int j = r + 1 + lane; j < sz; j += 32) {
      const float v = Ms[r * LD + j] - Ms[j * LD + r];
      if (accumulate) oi[j] += v;
      else oi[j] = v;
    }
  }
}

// The same computation for 128 x 128 blocks on a cluster of four CTAs per
// block: CTA r owns rows [32r, 32r + 32) of G, T = M^T G and GQ = 2 T M^T.
//   1. reduce its rows of G from the partials; load its rows of M
//   2. cluster barrier; copy the other CTAs' rows of G and M over
//      distributed shared memory; cluster barrier (after it G's storage is
//      reused)
//   3. its rows of T (needs all of G and its columns of M), stored as T^T
//   4. its rows of GQ (needs its rows of T and all of M, read as M^T)
//   5. cluster barrier; pack its rows, reading GQ[j][i] from the CTA that
//      owns row j; cluster barrier so no CTA exits while another reads it.
// Every CTA runs every cluster barrier (no early exit).  256 threads, each
// holding a 4 x 4 tile of the 32 x 128 output rows.
constexpr int kCbwdLD = 132;        // padded row of a 128-wide fp32 matrix
constexpr int kCbwdTLD = 36;        // padded row of T^T (32 wide)
constexpr int kCbwdSmem = (2 * 128 * kCbwdLD + 128 * kCbwdTLD + 32 * kCbwdLD) * 4;

// Clusters [0, a.s.nblk) work on side a, the rest on side b (both sides of a
// layer in one launch).
__global__ void __cluster_dims__(4, 1, 1) __launch_bounds__(256) cayley_bwd_cluster_kernel(
    const CbwdSide a, const CbwdSide b, int accumulate) {
  griddep_enter();
  constexpr int P = 128, LD = kCbwdLD, TLD = kCbwdTLD;
  const int kg = blockIdx.x / 4;
  const bool on_a = kg < a.s.nblk;
  const CbwdSide& side = on_a ? a : b;
  const float* __restrict__ partial = side.partial;
  const int64_t split_stride = side.split_stride;
  const int splits = side.splits;
  const SideGeom s = side.s;
  const float* __restrict__ Mall = side.M;
  float* __restrict__ out = side.out;
  extern __shared__ __align__(16) float cbs[];
  float* Gs = cbs;               // G (all rows), then M^T
  float* Ms = Gs + P * LD;       // M
  float* Tt = Ms + P * LD;       // T^T: Tt[q][i - r0]
  float* Qs = Tt + P * TLD;      // GQ rows [r0, r0 + 32)
  const uint32_t rank = cluster_ctarank();
  const int k = on_a ? kg : kg - a.s.nblk;
  const int r0 = 32 * static_cast<int>(rank);
  const int tid = threadIdx.x;
  const float* Mk = Mall + static_cast<int64_t>(k) * P * P;
  const float* Pk = partial + static_cast<int64_t>(k) * P * P;  // super-block k (sb = 128)

  // 1. own rows of G (summed over splits in a fixed order) and of M: four
  //    float4 of each per thread, all loads of one split in flight together
  {
    constexpr int PER = 32 * P / 4 / 256;  // 4
    float4 g[PER], m[PER];
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int e = tid + 256 * u;
      const int i = r0 + e / (P / 4), j4 = 4 * (e % (P / 4));
      g[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      m[u] = *reinterpret_cast<const float4*>(Mk + i * P + j4);
    }
    // two splits' loads in flight before they are added (ascending split order)
    auto split_ld = [&](int p, int u) {
      const int e = tid + 256 * u;
      const int i = r0 + e / (P / 4), j4 = 4 * (e % (P / 4));
      return *reinterpret_cast<const float4*>(Pk + p * split_stride + i * P + j4);
    };
    int p = 0;
    for (; p + 2 <= splits; p += 2) {
      float4 w[2][PER];
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int u = 0; u < PER; ++u) w[q][u] = split_ld(p + q, u);
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int u = 0; u < PER; ++u) {
          g[u].x += w[q][u].x; g[u].y += w[q][u].y; g[u].z += w[q][u].z; g[u].w += w[q][u].w;
        }
    }
    if (p < splits) {
#pragma unroll
      for (int u = 0; u < PER; ++u) {
        const float4 w = split_ld(p, u);
        g[u].x += w.x; g[u].y += w.y; g[u].z += w.z; g[u].w += w.w;
      }
    }
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int e = tid + 256 * u;
      const int i = r0 + e / (P / 4), j4 = 4 * (e % (P / 4));
      *reinterpret_cast<float4*>(Gs + i * LD + j4) = g[u];
      *reinterpret_cast<float4*>(Ms + i * LD + j4) = m[u];
    }
  }
  cluster_sync();
  // 2. the other CTAs' rows of G and M over distributed shared memory
#pragma unroll 4
  for (int e = tid; e < 3 * 32 * P / 4; e += 256) {
    const uint32_t other = (rank + 1 + e / (32 * P / 4)) & 3u;
    const int f = e % (32 * P / 4);
    const int o = (32 * static_cast<int>(other) + f / (P / 4)) * LD + 4 * (f % (P / 4));
    const float4 gv = dsmem_ld_f4(dsmem_addr(Gs + o, other));
    const float4 mv = dsmem_ld_f4(dsmem_addr(Ms + o, other));
    *reinterpret_cast<float4*>(Gs + o) = gv;
    *reinterpret_cast<float4*>(Ms + o) = mv;
  }
  cluster_sync();
  // 3. T[i][j] = sum_q M[q][i] G[q][j] for i in [r0, r0 + 32)
  const int tr = tid / 32, tc = tid % 32;  // rows 4tr.., columns 4tc..
  float acc[4][4];
#pragma unroll
  for (int x = 0; x < 4; ++x)
#pragma unroll
    for (int y = 0; y < 4; ++y) acc[x][y] = 0.f;
#pragma unroll 4
  for (int q = 0; q < P; ++q) {
    const float4 a = *reinterpret_cast<const float4*>(Ms + q * LD + r0 + 4 * tr);
    const float4 g = *reinterpret_cast<const float4*>(Gs + q * LD + 4 * tc);
    const float av[4] = {a.x, a.y, a.z, a.w}, gv[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
      for (int y = 0; y < 4; ++y) acc[x][y] = fmaf(av[x], gv[y], acc[x][y]);
  }
#pragma unroll
  for (int y = 0; y < 4; ++y)
    *reinterpret_cast<float4*>(Tt + (4 * tc + y) * TLD + 4 * tr) =
        make_float4(acc[0][y], acc[1][y], acc[2][y], acc[3][y]);
  __syncthreads();
  // G is no longer needed (and no other CTA reads it after step 2): M^T in its place
  for (int e = tid; e < P * P; e += 256) {
    const int i = e / P, j = e % P;
    Gs[j * LD + i] = Ms[i * LD + j];
  }
  __syncthreads();
  // 4. GQ[i][j] = 2 sum_q T[i][q] M[j][q] = 2 sum_q T^T[q][i] M^T[q][j]
#pragma unroll
  for (int x = 0; x < 4; ++x)
#pragma unroll
    for (int y = 0; y < 4; ++y) acc[x][y] = 0.f;
#pragma unroll 4
  for (int q = 0; q < P; ++q) {
    const float4 t = *reinterpret_cast<const float4*>(Tt + q * TLD + 4 * tr);
    const float4 m = *reinterpret_cast<const float4*>(Gs + q * LD + 4 * tc);
    const float tv[4] = {t.x, t.y, t.z, t.w}, mv[4] = {m.x, m.y, m.z, m.w};
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
      for (int y = 0; y < 4; ++y) acc[x][y] = fmaf(tv[x], mv[y], acc[x][y]);
  }
#pragma unroll
  for (int x = 0; x < 4; ++x)
    *reinterpret_cast<float4*>(Qs + (4 * tr + x) * LD + 4 * tc) =
        make_float4(2.f * acc[x][0], 2.f * acc[x][1], 2.f * acc[x][2], 2.f * acc[x][3]);
  cluster_sync();
  // 5. pack rows i in [r0, r0 + 32): g_ij = GQ[i][j] - GQ[j][i], j > i
  const int sz = block_size(s, k);
  float* o = out + static_cast<int64_t>(k) * P * (P - 1) / 2;
  const int warp = tid / 32, lane = tid % 32;
  for (int il = warp; il < 32; il += 8) {
    const int i = r0 + il;
    if (i >= sz - 1) continue;
    float* oi = o + (i * sz - i * (i + 1) / 2 - i - 1);
    for (int j = i + 1 + lane; j < sz; j += 32) {
      const uint32_t owner = static_cast<uint32_t>(j / 32);
      const float* src = Qs + (j % 32) * LD + i;
      const float gji = owner == rank ? *src : dsmem_ld_f(dsmem_addr(src, owner));
      const float v = Qs[il * LD + j] - gji;
      if (accumulate) oi[j] += v;
      else oi[j] = v;
    }
  }
  cluster_sync();
}

// ------------------------------------------------------------------ self-test
// Waits on a barrier that nothing completes; must give up after timeout_ns.
__global__ void bounded_wait_selftest_kernel(uint64_t timeout_ns, int* result) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const bool ok = mbar_wait(&bar, 0, timeout_ns, &abort_flag);
    *result = ok ? 1 : 2;
  }
}

}  // namespace poetx
