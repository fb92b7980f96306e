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

// ------------------------------------------------------------------ gathers
// out[r][j] = in[r][idx[j]] for `rows` rows of d elements (row-local feature
// permutation).  A CTA stages whole rows in shared memory with 16-byte loads,
// then writes the permuted row with 16-byte stores, so global traffic is one
// coalesced read and one coalesced write per element.
template <typename T>
__global__ void __launch_bounds__(256) gather_cols_kernel(const T* __restrict__ in,
                                                          T* __restrict__ out,
                                                          const int32_t* __restrict__ idx,
                                                          int64_t rows, int d) {
  extern __shared__ __align__(16) uint8_t gsm[];
  T* row = reinterpret_cast<T*>(gsm);
  constexpr int VEC = 16 / sizeof(T);
  const bool vec_ok = (d % VEC) == 0;
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const T* src = in + r * d;
    T* dst = out + r * d;
    if (vec_ok) {
      for (int c = threadIdx.x; c < d / VEC; c += blockDim.x)
        reinterpret_cast<uint4*>(row)[c] = __ldcs(reinterpret_cast<const uint4*>(src) + c);
    } else {
      for (int c = threadIdx.x; c < d; c += blockDim.x) row[c] = src[c];
    }
    __syncthreads();
    if (vec_ok) {
      for (int c = threadIdx.x; c < d / VEC; c += blockDim.x) {
        alignas(16) T v[VEC];
#pragma unroll
        for (int q = 0; q < VEC; ++q) v[q] = row[__ldg(idx + c * VEC + q)];
        reinterpret_cast<uint4*>(dst)[c] = *reinterpret_cast<const uint4*>(v);
      }
    } else {
      for (int c = threadIdx.x; c < d; c += blockDim.x) dst[c] = row[__ldg(idx + c)];
    }
    __syncthreads();
  }
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

// Unpacks the strict upper triangle of block k into Q (b x b, zero padded
// beyond the block's size) and writes A = I - Q (identity on the padding).
__global__ void __launch_bounds__(256) unpack_kernel(const float* __restrict__ gen, SideGeom s,
                                                     float* __restrict__ Q, float* __restrict__ A) {
  const int k = blockIdx.x;
  const int sz = block_size(s, k);
  const int64_t off = static_cast<int64_t>(k) * s.b * (s.b - 1) / 2;
  const int64_t bb = static_cast<int64_t>(s.b) * s.b;
  for (int e = threadIdx.x; e < s.b * s.b; e += blockDim.x) {
    const int i = e / s.b, j = e % s.b;
    float q = 0.f;
    if (i < sz && j < sz && i != j) {
      if (i < j) q = gen[off + static_cast<int64_t>(i) * sz - i * (i + 1) / 2 + (j - i - 1)];
      else q = -gen[off + static_cast<int64_t>(j) * sz - j * (j + 1) / 2 + (i - j - 1)];
    }
    Q[k * bb + e] = q;
    if (A) A[k * bb + e] = (i == j ? 1.f : 0.f) - q;
  }
}

// In-place Gauss-Jordan inversion of P x P sub-matrices (P <= 128) without
// pivoting: the matrices inverted here are I - Q for skew Q and the pivot
// blocks of its block elimination, whose symmetric parts are >= I, so every
// pivot is >= 1 in magnitude and no exchange is needed.  Matrix z is read
// at in + z*in_bs with leading dimension in_ld and written likewise to out.
__global__ void __launch_bounds__(1024) gj_invert_kernel(const float* in, int64_t in_bs, int in_ld,
                                                         float* out, int64_t out_bs, int out_ld,
                                                         int P) {
  extern __shared__ __align__(16) float gj_sm[];
  float* a = gj_sm;            // P x P
  float* col = a + P * P;      // P
  float* rowv = col + P;       // P
  const int z = blockIdx.x;
  const float* src = in + z * in_bs;
  for (int e = threadIdx.x; e < P * P; e += blockDim.x) a[e] = src[(e / P) * in_ld + (e % P)];
  __syncthreads();
  for (int k = 0; k < P; ++k) {
    if (threadIdx.x < P) {
      col[threadIdx.x] = a[threadIdx.x * P + k];
      rowv[threadIdx.x] = a[k * P + threadIdx.x];
    }
    __syncthreads();
    const float p = 1.0f / rowv[k];
    for (int e = threadIdx.x; e < P * P; e += blockDim.x) {
      const int i = e / P, j = e % P;
      float v;
      if (i == k) v = (j == k) ? p : rowv[j] * p;
      else if (j == k) v = -col[i] * p;
      else v = fmaf(-col[i] * p, rowv[j], a[e]);
      a[e] = v;
    }
    __syncthreads();
  }
  float* dst = out + z * out_bs;
  for (int e = threadIdx.x; e < P * P; e += blockDim.x) dst[(e / P) * out_ld + (e % P)] = a[e];
}

// dst[z](i,j) = alpha * src[z](i,j) (+ beta * I(i,j)) over rows x cols.
__global__ void __launch_bounds__(256) copy2d_kernel(const float* src, int64_t s_bs, int s_ld,
                                                     float* dst, int64_t d_bs, int d_ld, int rows,
                                                     int cols, float alpha, float beta_eye) {
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

// ------------------------------------------------------------------ gradients
// G[k](i,j) = sum over splits p of partial[p][s][(a - s*sb)][(c - s*sb)],
// a = k*b + i, c = k*b + j, s = a / sb, in a fixed order (deterministic).
__global__ void __launch_bounds__(256) gradred_reduce_kernel(const float* __restrict__ partial,
                                                             int64_t split_stride, int splits,
                                                             SideGeom s, int sb,
                                                             float* __restrict__ G) {
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

// Packed generator gradient: g[(i,j)] (+)= GQ[k](i,j) - GQ[k](j,i), i < j < size.
__global__ void __launch_bounds__(256) pack_grad_kernel(const float* __restrict__ GQ, SideGeom s,
                                                        float* __restrict__ out, int accumulate) {
  const int k = blockIdx.x;
  const int sz = block_size(s, k);
  const int64_t off = static_cast<int64_t>(k) * s.b * (s.b - 1) / 2;
  const int64_t bb = static_cast<int64_t>(s.b) * s.b;
  const int npairs = sz * (sz - 1) / 2;
  for (int e = threadIdx.x; e < npairs; e += blockDim.x) {
    // invert e = i*sz - i(i+1)/2 + (j-i-1): walk rows (sz <= 512, cheap)
    int i = 0, rem = e;
    while (rem >= sz - 1 - i) rem -= sz - 1 - i, ++i;
    const int j = i + 1 + rem;
    const float v = GQ[k * bb + static_cast<int64_t>(i) * s.b + j] -
                    GQ[k * bb + static_cast<int64_t>(j) * s.b + i];
    if (accumulate) out[off + e] += v;
    else out[off + e] = v;
  }
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
