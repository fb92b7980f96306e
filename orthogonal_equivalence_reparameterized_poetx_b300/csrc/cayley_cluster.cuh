// Exact Cayley blocks of size 256 or 512 in one launch: one cluster per
// block (two CTAs of 128 rows at b = 256, eight of 64 rows at b = 512).
//
// "POET-X：基于正交变换缩放的内存高效LLM训练方法", 实践 2: B = (I+Q)(I-Q)^-1,
// which equals 2M - I with M = (I - Q)^-1 (the factors commute).  CTA c of a
// block's cluster keeps rows [c*RB, c*RB + RB) of the working matrix
// A = I - Q in shared memory and the cluster inverts A in place
// by Gauss-Jordan, W = 32 pivots per panel K = [k0, k0 + W):
//
//   D = A_KK^-1                          (every CTA, from the owner's rows)
//   R = D A_K*                           (each CTA forms RB of its columns)
//   A_ij -= A_iK R_Kj     i, j outside K
//   A_iK  = -A_iK D       i outside K
//   A_K*  = R,  A_KK = D  (the owner of the pivot rows)
//
// Both kinds of update of a row outside K are one rank-W update with the
// panel column r_j: r_j = R_*j (start A_ij) for j outside K and r_j = D_*j'
// (start 0) for j = k0 + j' in K.  No pivoting: the symmetric part of I - Q
// is I, so every pivot block and every Schur complement has a symmetric
// part >= I, hence an inverse of norm <= 1.
//
// A ragged last block of size sz < b is inverted as the b x b matrix padded
// with the identity, which leaves the padding exactly the identity.
// Per panel: two cluster barriers and W + 1 block barriers; no other waits.
#pragma once

#include "ptx.cuh"
#include "simt.cuh"

namespace poetx {

template <int BS>
struct CcCfg {
  // b = 256: two CTAs of 1024 threads; b = 512: eight CTAs of 512 threads
  // (fewer, wider CTAs hold an SM for less time in total; at b = 512 the
  // 128 KB of rows per CTA allows one CTA per SM and 512 threads keep the
  // per-pivot barriers cheap)
  static constexpr int C = BS == 256 ? 2 : 8;  // CTAs per block (one cluster)
  static constexpr int NT = BS == 256 ? 1024 : 512;  // threads per CTA
  static constexpr int RB = BS / C;           // rows of A per CTA
  static constexpr int TPC = NT / BS;         // threads per column
  static constexpr int RPT = RB / TPC;        // rows per thread
  static constexpr int W = 32;                // pivots per panel
  static constexpr int CS = BS / C;           // columns of R each CTA forms
  static constexpr int NW = NT / 32;          // warps
  static constexpr int U = W / NW;            // pivot-block rows per warp
  static constexpr int DLD = W + 1;           // leading dimension of the inverted pivot block
  static constexpr int RLD = W + 4;           // leading dimension of the transposed R slice
  static constexpr int A_F = RB * BS;
  static constexpr int D_F = W * DLD + 2 * W;  // inverse, then two pivot-row buffers
  static constexpr int CP_F = RB * W;
  static constexpr int AK_F = W * CS;
  static constexpr int RS_F = CS * RLD;
  static constexpr size_t SMEM = static_cast<size_t>(A_F + D_F + CP_F + AK_F + RS_F) * 4;
  static_assert(W % NW == 0 && RPT % W == 0, "pivot-block rows per warp; whole panels per thread");
  static_assert((W * CS) % NT == 0 && (RB * W) % NT == 0 && RB % W == 0, "work split");
  static_assert(D_F % 4 == 0 && A_F % 4 == 0, "16-byte alignment of the buffers");
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

// Blocks [0, first.s.nblk) belong to `first`, the rest to `second`; both
// sides have block size BS.  Grid: C CTAs per block, NT threads each:
// thread t owns column t % BS of the CTA's rows [RPT (t / BS), RPT (t / BS) + RPT).
template <int BS>
__global__ void __cluster_dims__(CcCfg<BS>::C, 1, 1) __launch_bounds__(CcCfg<BS>::NT, 1)
    cayley_cluster_kernel(const CayleySide first, const CayleySide second) {
  using Cfg = CcCfg<BS>;
  constexpr int C = Cfg::C, RB = Cfg::RB, W = Cfg::W, CS = Cfg::CS, NT = Cfg::NT;
  constexpr int RPT = Cfg::RPT, DLD = Cfg::DLD, RLD = Cfg::RLD, NW = Cfg::NW, U = Cfg::U;
  constexpr int E_AK = W * CS / NT, E_CP = RB * W / NT;
  extern __shared__ __align__(16) float ccs[];
  float* A = ccs;                 // own rows of the working matrix, RB x BS
  float* Dinv = A + Cfg::A_F;     // the inverted pivot block, W x DLD
  float* rowbuf = Dinv + W * DLD; // two pivot-row buffers of W
  float* Cp = rowbuf + 2 * W;     // own rows of the pivot columns, RB x W
  float* AK = Cp + Cfg::CP_F;     // pivot rows, this CTA's column slice, W x CS
  float* RS = AK + Cfg::AK_F;     // this CTA's columns of R, transposed: RS[jj * RLD + p]

  const int kg = static_cast<int>(blockIdx.x) / C;
  const bool is_first = kg < first.s.nblk;
  const CayleySide& cs = is_first ? first : second;
  const int k = is_first ? kg : kg - first.s.nblk;
  const uint32_t rank = cluster_ctarank();
  const int r0 = RB * static_cast<int>(rank);
  const int c0 = CS * static_cast<int>(rank);
  const int tid = static_cast<int>(threadIdx.x);
  const int j = tid % BS;                 // column
  const int i0 = RPT * (tid / BS);        // first of this thread's rows (within the CTA)
  const int warp = tid / 32, lane = tid % 32;
  const int sz = block_size(cs.s, k);
  const int64_t base = static_cast<int64_t>(k) * BS * BS;
  const float* g = cs.gen + static_cast<int64_t>(k) * BS * (BS - 1) / 2;

  // 1. own rows of Q (unpacked from the strict upper triangle, entry (i, j),
  //    i < j, at i*sz - i(i+1)/2 + (j-i-1)) and of A = I - Q; eight rows'
  //    loads in flight at a time
  for (int t0 = 0; t0 < RPT; t0 += 8) {
    float q[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const int gi = r0 + i0 + t0 + t;
      q[t] = 0.f;
      if (gi < sz && j < sz && gi != j)
        q[t] = gi < j ? g[gi * sz - gi * (gi + 1) / 2 + (j - gi - 1)]
                      : -g[j * sz - j * (j + 1) / 2 + (gi - j - 1)];
    }
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const int gi = r0 + i0 + t0 + t;
      cs.Q[base + static_cast<int64_t>(gi) * BS + j] = q[t];
      A[(i0 + t0 + t) * BS + j] = (gi == j ? 1.f : 0.f) - q[t];
    }
  }

  // 2. Gauss-Jordan, one panel of W pivots at a time
  for (int k0 = 0; k0 < BS; k0 += W) {
    const int owner = k0 / RB;
    const int ok0 = k0 - RB * owner;  // first pivot row within the owner's rows
    const bool own_pivots = static_cast<int>(rank) == owner;
    // every CTA's previous update is complete; the panel buffers may be rewritten
    cluster_sync();
    const uint32_t oA = dsmem_addr(A, static_cast<uint32_t>(owner));
    // pivot block (warp w holds rows w + NW*u, lane = column) and this CTA's
    // slice of the pivot rows, both from the owner; own pivot columns
    float d[U], ak[E_AK], cp[E_CP];
#pragma unroll
    for (int u = 0; u < U; ++u)
      d[u] = dsmem_ld_f(oA + 4u * static_cast<uint32_t>((ok0 + warp + NW * u) * BS + k0 + lane));
#pragma unroll
    for (int u = 0; u < E_AK; ++u) {
      const int e = tid + NT * u, p = e / CS, jj = e % CS;
      ak[u] = dsmem_ld_f(oA + 4u * static_cast<uint32_t>((ok0 + p) * BS + c0 + jj));
    }
#pragma unroll
    for (int u = 0; u < E_CP; ++u) {
      const int e = tid + NT * u, i = e / W, p = e % W;
      cp[u] = A[i * BS + k0 + p];
    }
#pragma unroll
    for (int u = 0; u < E_AK; ++u) {
      const int e = tid + NT * u, p = e / CS, jj = e % CS;
      AK[p * CS + jj] = ak[u];
    }
#pragma unroll
    for (int u = 0; u < E_CP; ++u) {
      const int e = tid + NT * u, i = e / W, p = e % W;
      Cp[i * W + p] = cp[u];
    }
    if (warp == 0) rowbuf[lane] = d[0];  // pivot row 0 (warp 0, u = 0)
    // D = A_KK^-1 in registers: unpivoted Gauss-Jordan, one pivot per step;
    // the pivot row goes through shared memory (ping-pong), the pivot column
    // through warp shuffles
#pragma unroll 1
    for (int p = 0; p < W; ++p) {
      __syncthreads();
      const float* rb = rowbuf + (p & 1) * W;
      const float inv = __frcp_rn(rb[p]);
      const float rq = rb[lane] * inv;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const float f = __shfl_sync(0xffffffffu, d[u], p);
        if (warp + NW * u == p) d[u] = (lane == p) ? inv : rq;
        else d[u] = (lane == p) ? -f * inv : fmaf(-f, rq, d[u]);
      }
      const int pn = p + 1;
      if (pn < W && pn % NW == warp) {
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (u == pn / NW) rowbuf[(pn & 1) * W + lane] = d[u];
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) Dinv[(warp + NW * u) * DLD + lane] = d[u];
    __syncthreads();
    // this CTA's columns of R = D A_K* (columns inside K are never read);
    // thread t forms E_AK entries of one column jj
    {
      const int jj = tid % CS, p0 = tid / CS;
      constexpr int PS = NT / CS;  // row stride between a thread's entries
      if (!(c0 + jj >= k0 && c0 + jj < k0 + W)) {
        float acc[E_AK];
#pragma unroll
        for (int u = 0; u < E_AK; ++u) acc[u] = 0.f;
#pragma unroll 8
        for (int q = 0; q < W; ++q) {
          const float a = AK[q * CS + jj];
#pragma unroll
          for (int u = 0; u < E_AK; ++u) acc[u] = fmaf(Dinv[(p0 + PS * u) * DLD + q], a, acc[u]);
        }
#pragma unroll
        for (int u = 0; u < E_AK; ++u) RS[jj * RLD + p0 + PS * u] = acc[u];
      }
    }
    cluster_sync();  // every CTA's columns of R are complete
    // the panel column of thread t's column j
    const bool inK = j >= k0 && j < k0 + W;
    float r[W];
    if (inK) {
#pragma unroll
      for (int q = 0; q < W; ++q) r[q] = Dinv[q * DLD + (j - k0)];
    } else {
      const uint32_t src = dsmem_addr(RS + (j % CS) * RLD, static_cast<uint32_t>(j / CS));
#pragma unroll
      for (int q4 = 0; q4 < W / 4; ++q4) {
        const float4 v = dsmem_ld_f4(src + 16u * static_cast<uint32_t>(q4));
        r[4 * q4] = v.x;
        r[4 * q4 + 1] = v.y;
        r[4 * q4 + 2] = v.z;
        r[4 * q4 + 3] = v.w;
      }
    }
    // rank-W update of the thread's rows outside K, four at a time; the
    // pivot rows get R outside K and D inside
    const bool has_pivots = own_pivots && ok0 >= i0 && ok0 < i0 + RPT;
    {
#pragma unroll 1
      for (int t0 = 0; t0 < RPT; t0 += 4) {
        const int i = i0 + t0;
        if (has_pivots && i >= ok0 && i < ok0 + W) continue;
        float acc[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) acc[t] = inK ? 0.f : A[(i + t) * BS + j];
#pragma unroll
        for (int q4 = 0; q4 < W / 4; ++q4) {
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const float4 c = reinterpret_cast<const float4*>(Cp + (i + t) * W)[q4];
            acc[t] = fmaf(-c.x, r[4 * q4], acc[t]);
            acc[t] = fmaf(-c.y, r[4 * q4 + 1], acc[t]);
            acc[t] = fmaf(-c.z, r[4 * q4 + 2], acc[t]);
            acc[t] = fmaf(-c.w, r[4 * q4 + 3], acc[t]);
          }
        }
#pragma unroll
        for (int t = 0; t < 4; ++t) A[(i + t) * BS + j] = acc[t];
      }
    }
    if (has_pivots) {
#pragma unroll
      for (int p = 0; p < W; ++p) A[(ok0 + p) * BS + j] = r[p];
    }
  }
  // no CTA leaves while another may still read its shared memory
  cluster_sync();

  // 3. outputs of the thread's rows: M, B = 2M - I, and for bf16 layers the
  //    super-block arrays (super-block = block here): Bsb rows are rows of B,
  //    BsbT rows are columns of B
  for (int t = 0; t < RPT; ++t) {
    const int i = i0 + t, gi = r0 + i;
    const float mv = A[i * BS + j];
    const float bv = 2.f * mv - (gi == j ? 1.f : 0.f);
    cs.M[base + static_cast<int64_t>(gi) * BS + j] = mv;
    cs.B[base + static_cast<int64_t>(gi) * BS + j] = bv;
    if (cs.Bsb) cs.Bsb[(static_cast<int64_t>(k) * BS + gi) * cs.sb + j] = __float2bfloat16_rn(bv);
    A[i * BS + j] = bv;
  }
  if (cs.BsbT) {
    // row k*BS + j of BsbT, columns [r0 + i0, r0 + i0 + RPT), from this
    // thread's own entries of A (no other thread wrote them)
    __nv_bfloat16* dst = cs.BsbT + (static_cast<int64_t>(k) * BS + j) * cs.sb + r0 + i0;
#pragma unroll 1
    for (int i8 = 0; i8 < RPT; i8 += 8) {
      const float* a = A + (i0 + i8) * BS + j;
      uint4 v;
      v.x = pack_bf16x2(a[0], a[BS]);
      v.y = pack_bf16x2(a[2 * BS], a[3 * BS]);
      v.z = pack_bf16x2(a[4 * BS], a[5 * BS]);
      v.w = pack_bf16x2(a[6 * BS], a[7 * BS]);
      *reinterpret_cast<uint4*>(dst + i8) = v;
    }
  }
}

}  // namespace poetx
