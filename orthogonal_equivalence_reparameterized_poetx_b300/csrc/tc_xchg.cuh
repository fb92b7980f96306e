// Permutation passes fused with the 128-wide block transforms (tcgen05),
// exchanging token bands through a small ring in global memory that stays
// in L2.
//
// "POET-X: Memory-efficient LLM Training by Scaling Orthogonal
// Transformation" (gist.science summary), Methodologie §2 keeps the outer
// permutations as index maps and §3 treats the block-diagonal factors as
// independent small matrices.  A permutation of features needs whole rows on
// chip (a 2-byte column gather has no TMA form), while a block transform
// wants its block matrix resident across many tokens.  This kernel gives
// each CTA both jobs:
//   tile side  the CTA owns g super-blocks of 128 features (their matrices
//              resident in TMEM as the A operand) and transforms 64-token
//              tiles of them: D (128 features x 64 tokens) = S_j x tile^T;
//              with RED it also accumulates G_j += tile^T C over its tokens
//              (the generator-gradient token reduction) in TMEM;
//   band side  up to eight warps permute whole rows staged in shared memory,
//              each warp its own rows, with its own bulk copies and barriers.
// CTAs form slots of Q (the Q CTAs of a slot own all super-blocks); slot s
// takes the 64-token bands k = s, s + S, ...  Band k lives in ring entry
// k % E (E a multiple of S, at least two rounds per slot).
//   GATHER (forward P: X -> u -> v; backward R: dY -> dz -> dh, with RED):
//     band side: ring rows = input rows gathered by idx = pi, produced[k]
//     counts the rows written; tile side: waits until all 64 rows of band k
//     are there, loads its tiles from the ring, consumed[k] += 1 per CTA,
//     transforms, stores the output tile.  With ring_full the band side
//     writes a T-row buffer (the saved u) instead, which is never reused.
//   SCATTER (forward R: h -> z -> Y; backward P: dv -> du -> dX, with RED):
//     tile side: loads activation tiles, transforms, writes them into the
//     ring, produced[k] += 1 per CTA; band side: waits until all Q CTAs
//     wrote band k, loads its ring rows, consumed[k] counts the rows loaded,
//     writes the output rows permuted by idx = pi^-1.
// Local row r of a band belongs to CTA r % Q of the slot and, among that
// CTA's rows, to band warp (r / Q) % aw, so every row is counted once.  A
// ring entry is rewritten only after its previous band was fully consumed.
// The roles publish their progress inside the CTA through monotonic
// counters in shared memory (release / acquire at CTA scope); one
// signaling warp turns them into the grid-visible per-band counters
// (release at GPU scope), so no data-path warp waits for a GPU-scope
// release.  Every CTA of the grid must be resident at once (cooperative
// launch, one CTA per SM).  Every wait, on an mbarrier or on a counter, is
// bounded: after the deadline the CTA records a timeout, raises the
// grid-wide abort word (so the other CTAs stop waiting too), drains its
// copies in flight, frees TMEM and returns.
//
// Warps: 0 TMA producer, 1 TMEM allocator + MMA issuer, 2..5 and 6..9 the
// two epilogue groups (group e takes the tiles of TMEM accumulator e, i.e.
// every other tile; warp w reads TMEM lanes 32 (w % 4) ..), 10..17 band
// side (the first aw active, bpw row buffers each), 18..20 signaling (lane 0
// of each: produced, consumed, ring gate of the SCATTER tile side; one warp
// per role, so that one role's waits never hold up another's).
#pragma once

#include "ptx.cuh"

namespace poetx {

struct XchgArgs {
  int T;          // tokens
  int d;          // features of this side
  int nsb;        // 128-wide super-blocks
  int Q;          // CTAs per slot
  int S;          // slots
  int nbands;     // 64-token bands
  int E;          // ring entries (multiple of S)
  int ring_full;  // GATHER: the band side writes a T-row buffer (no ring reuse)
  int aw;         // active band-side warps (1..8)
  int bpw;        // row buffers per band-side warp (1..2)
  const int32_t* idx;        // band-side gather index (length d, values < d <= 12288)
  const uint16_t* band_src;  // rows of d bf16
  uint16_t* band_dst;        // rows of d bf16
  uint16_t* ring;            // SCATTER: the ring the tile side writes (E * 64 rows of d)
  const __nv_bfloat16* Bmat; // nsb * 128 rows of 128: row f = output feature f (A operand)
  float* partial;            // RED: [S][nsb][128][128] fp32
  uint32_t* produced;        // [nbands]
  uint32_t* consumed;        // [nbands]
  uint32_t* abort_word;      // grid-wide abort
  uint64_t timeout_ns;
};

struct XchgCfg {
  static constexpr int BOX = 64 * 64 * 2;   // 64 tokens x 64 features: 8 KB
  static constexpr int TILE = 2 * BOX;      // 64 tokens x 128 features: 16 KB
  static constexpr int BAND_BYTES = 72 * 1024;  // band-side row buffers
  static constexpr int MAX_D = 12288;           // features (16-bit indices, one row per buffer)
  static constexpr int IDX_BYTES = 2 * MAX_D;   // gather index as 16-bit values
  static constexpr int BAND_WARPS = 8;
  static constexpr int MAX_BPW = 2;
  static constexpr int THREADS = 672;
  template <bool RED>
  __host__ __device__ static constexpr int stages() { return RED ? 3 : 6; }
  template <bool RED>
  __host__ __device__ static constexpr int stage_bytes() { return RED ? 2 * TILE : TILE; }
  template <bool RED>
  __host__ __device__ static constexpr int smem() {
    return 1024 + stages<RED>() * stage_bytes<RED>() + 2 * TILE + BAND_BYTES + IDX_BYTES + 512;
  }
  __host__ __device__ static constexpr int max_g(bool red) { return red ? 2 : 6; }
};
static_assert(XchgCfg::smem<true>() <= 232448 && XchgCfg::smem<false>() <= 232448, "shared memory");

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// CTA-scope release store / acquire load of a shared-memory counter.
__device__ __forceinline__ void st_release_cta(uint32_t* p, uint32_t v) {
  asm volatile("st.release.cta.shared.u32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_cta(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.cta.shared.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}

// Orders generic-proxy global accesses with async-proxy (TMA, bulk copy)
// accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait_le() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait_read_le() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Gives up a wait: after an abort (this CTA's or the grid's), or after the
// deadline, when it records the timeout and raises both aborts.
__device__ __forceinline__ bool give_up(uint64_t t0, uint64_t timeout_ns, volatile int* abort_cta,
                                        uint32_t* abort_grid) {
  if (*abort_cta) return true;
  if (ld_relaxed_u32(abort_grid) != 0u) {
    *abort_cta = 1;
    return true;
  }
  if (global_timer_ns() - t0 > timeout_ns) {
    record_status(kStatusTimeout);
    atomicExch(abort_grid, 1u);
    *abort_cta = 1;
    return true;
  }
  return false;
}

// Waits until the global counter *p >= target (acquire, GPU scope).
__device__ __noinline__ bool poll_geq(const uint32_t* p, uint32_t target, uint64_t timeout_ns,
                                      volatile int* abort_cta, uint32_t* abort_grid) {
  if (ld_acquire_u32(p) >= target) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (ld_acquire_u32(p) >= target) return true;
    if ((i & 15u) == 0u && give_up(t0, timeout_ns, abort_cta, abort_grid)) return false;
  }
}

// Waits until the shared counter *p >= target (acquire, CTA scope).
__device__ __noinline__ bool poll_cta_geq(const uint32_t* p, uint32_t target, uint64_t timeout_ns,
                                          volatile int* abort_cta, uint32_t* abort_grid) {
  if (ld_acquire_cta(p) >= target) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    __nanosleep(20);
    if (ld_acquire_cta(p) >= target) return true;
    if ((i & 63u) == 0u && give_up(t0, timeout_ns, abort_cta, abort_grid)) return false;
  }
}

// mbarrier wait that also gives up when the grid-wide abort word is raised.
__device__ __forceinline__ bool xwait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns,
                                      volatile int* abort_cta, uint32_t* abort_grid) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 31u) == 0u && give_up(t0, timeout_ns, abort_cta, abort_grid)) return false;
  }
}

// 16 bytes of a row staged in shared memory at `row` (shared address):
// elements i0.x, i0.y, ..., i1.w, packed in that order.
__device__ __forceinline__ uint4 gather8(uint32_t row, int4 i0, int4 i1) {
  uint16_t e[8];
  const int id[8] = {i0.x, i0.y, i0.z, i0.w, i1.x, i1.y, i1.z, i1.w};
#pragma unroll
  for (int q = 0; q < 8; ++q)
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(e[q]) : "r"(row + 2u * static_cast<uint32_t>(id[q])));
  return make_uint4(e[0] | (static_cast<uint32_t>(e[1]) << 16), e[2] | (static_cast<uint32_t>(e[3]) << 16),
                    e[4] | (static_cast<uint32_t>(e[5]) << 16), e[6] | (static_cast<uint32_t>(e[7]) << 16));
}

template <bool GATHER, bool RED>
__global__ void __launch_bounds__(XchgCfg::THREADS, 1)
    tc_xchg_kernel(const __grid_constant__ CUtensorMap tmIn, const __grid_constant__ CUtensorMap tmC,
                   const __grid_constant__ CUtensorMap tmOut, const XchgArgs a) {
  using Cfg = XchgCfg;
  constexpr int NST = Cfg::stages<RED>();
  constexpr int STB = Cfg::stage_bytes<RED>();
  constexpr int NWB = Cfg::BAND_WARPS * Cfg::MAX_BPW;  // band-side mbarriers
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned by pointer arithmetic on the shared array, so that the
  // compiler keeps shared-memory instructions for every access through it
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* stages = smem;
  uint8_t* out_stage = stages + NST * STB;              // one 16 KB output tile per epilogue group
  uint8_t* bstage = out_stage + 2 * Cfg::TILE;          // band-side row buffers
  uint16_t* idx16 = reinterpret_cast<uint16_t*>(bstage + Cfg::BAND_BYTES);
  uint64_t* full = reinterpret_cast<uint64_t*>(bstage + Cfg::BAND_BYTES + Cfg::IDX_BYTES);
  uint64_t* empty = full + NST;
  uint64_t* tfull = empty + NST;
  uint64_t* tempty = tfull + 2;
  uint64_t* bload = tempty + 2;
  uint64_t* gdone = bload + 1;
  uint64_t* bfull = gdone + 1;
  // progress counters (monotonic, in bands): band warps, epilogue groups,
  // MMA issuer (tiles of a band in shared memory), ring gate
  uint32_t* warp_done = reinterpret_cast<uint32_t*>(bfull + NWB);
  uint32_t* group_done = warp_done + Cfg::BAND_WARPS;
  uint32_t* mma_loaded = group_done + 2;
  uint32_t* ring_ok = mma_loaded + 1;
  uint32_t* tmem_slot = ring_ok + 1;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint64_t tmo = a.timeout_ns;
  const int s = blockIdx.x / a.Q;  // slot
  const int q = blockIdx.x % a.Q;  // member of the slot
  const int lo = q * a.nsb / a.Q;  // first owned super-block
  const int g = (q + 1) * a.nsb / a.Q - lo;
  const int nb = (a.nbands > s) ? (a.nbands - s + a.S - 1) / a.S : 0;  // bands of this slot
  const int nr = (q < 64) ? (63 - q) / a.Q + 1 : 0;                      // rows of this CTA in a band
  // TMEM columns: RED: G_j at 128 j, transform accumulators at 256, block
  // matrices at 384 + 64 j; otherwise accumulators at 0, matrices at 128 + 64 j
  constexpr uint32_t kD = RED ? 256u : 0u;
  constexpr uint32_t kB = RED ? 384u : 128u;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 128);
    }
    mbar_init(bload, 256);
    mbar_init(gdone, 1);
    for (int i = 0; i < NWB; ++i) mbar_init(&bfull[i], 1);
    for (int i = 0; i < Cfg::BAND_WARPS; ++i) warp_done[i] = 0;
    group_done[0] = group_done[1] = 0;
    *mma_loaded = 0;
    *ring_ok = 0;
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmIn);
    if constexpr (RED) tma_prefetch_desc(&tmC);
    if constexpr (GATHER) tma_prefetch_desc(&tmOut);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  for (int j = threadIdx.x; j < a.d; j += blockDim.x) idx16[j] = static_cast<uint16_t>(__ldg(a.idx + j));
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_phase[NST];
      bool issued[NST];
      for (int i = 0; i < NST; ++i) issued[i] = false, issued_phase[i] = 0;
      bool ok = true;
      for (int i = 0; i < nb && ok; ++i) {
        const int k = s + i * a.S;
        const int y_in = GATHER ? (a.ring_full ? k * 64 : (k % a.E) * 64) : k * 64;
        for (int j = 0; j < g; ++j) {
          if (!xwait(&empty[stage], phase ^ 1u, tmo, abort_flag, a.abort_word)) { ok = false; break; }
          if (GATHER && j == 0) {
            if (!poll_geq(a.produced + k, 64u, tmo, abort_flag, a.abort_word)) {  // all 64 rows
              ok = false;
              break;
            }
            fence_proxy_async_global();
          }
          uint8_t* st = stages + stage * STB;
          const int x = (lo + j) * 128;
          mbar_arrive_expect_tx(&full[stage], STB);
          tma_load_2d(st, &tmIn, &full[stage], x, y_in);
          tma_load_2d(st + Cfg::BOX, &tmIn, &full[stage], x + 64, y_in);
          if constexpr (RED) {
            tma_load_2d(st + Cfg::TILE, &tmC, &full[stage], x, k * 64);
            tma_load_2d(st + Cfg::TILE + Cfg::BOX, &tmC, &full[stage], x + 64, k * 64);
          }
          issued[stage] = true;
          issued_phase[stage] = phase;
          if (++stage == NST) stage = 0, phase ^= 1u;
        }
      }
      // copies in flight must land before the CTA may exit
      volatile int never = 0;
      for (int i = 0; i < NST; ++i)
        if (issued[i]) mbar_wait(&full[i], issued_phase[i], tmo, &never);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      // transform: D (128 features x 64 tokens) = S_j (TMEM) x tile^T (K-major)
      constexpr uint32_t idesc_t = idesc_bf16_f32(128, 64, false, false);
      // reduction: G_j (128 x 128) += tile^T (MN-major) x C (MN-major), K = tokens
      constexpr uint32_t idesc_g = idesc_bf16_f32(128, 128, true, true);
      bool ok = (nb == 0) || xwait(bload, 0, tmo, abort_flag, a.abort_word);
      if (ok) tc_fence_after();
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      for (int i = 0; i < nb && ok; ++i) {
        for (int j = 0; j < g; ++j, ++it) {
          const int acc = it & 1;
          const uint32_t acc_phase = (it >> 1) & 1;
          if (!xwait(&tempty[acc], acc_phase ^ 1u, tmo, abort_flag, a.abort_word)) { ok = false; break; }
          if (!xwait(&full[stage], phase, tmo, abort_flag, a.abort_word)) { ok = false; break; }
          tc_fence_after();
          // all of band i's ring tiles are in shared memory: the entry may be reused
          if (GATHER && j == g - 1) st_release_cta(mma_loaded, static_cast<uint32_t>(i + 1));
          const uint32_t st = smem_u32(stages + stage * STB);
          const uint32_t d_t = tmem_base + kD + acc * 64;
          const uint32_t b_t = tmem_base + kB + 64 * j;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * Cfg::BOX + (kk & 3) * 32;
            mma_bf16_f32_ta(d_t, b_t + 8 * kk, smem_desc_sw128(st + off, 16, 1024), idesc_t,
                            kk != 0 ? 1u : 0u);
          }
          if constexpr (RED) {
            const uint32_t d_g = tmem_base + 128 * j;
#pragma unroll
            for (int kt = 0; kt < 4; ++kt) {
              const uint32_t off = kt * 16 * 128;
              mma_bf16_f32(d_g, smem_desc_sw128(st + off, Cfg::BOX, 1024),
                           smem_desc_sw128(st + Cfg::TILE + off, Cfg::BOX, 1024), idesc_g,
                           (i | kt) != 0 ? 1u : 0u);
            }
          }
          mma_commit(&empty[stage]);
          mma_commit(&tfull[acc]);
          if (++stage == NST) stage = 0, phase ^= 1u;
        }
      }
      // every MMA issued must finish before TMEM is read for G or released
      mma_commit(gdone);
      volatile int never = 0;
      mbar_wait(gdone, 0, tmo, &never);
    }
  } else if (warp < 10) {
    // -------------------------------------------------------------- epilogue
    const int e = (warp - 2) >> 2;     // group: tiles of TMEM accumulator e
    const int lg = warp & 3;           // TMEM lane group: features 32 lg ..
    const int f = lg * 32 + lane;      // feature within the super-block
    const int gt = (warp - 2 - 4 * e) * 32 + lane;  // thread within the group, 0 .. 127
    const bool leader = (gt == 0);
    const int bar_id = 1 + e;
    const uint32_t lane_off = static_cast<uint32_t>(lg * 32) << 16;
    uint8_t* ob = out_stage + e * Cfg::TILE;
    bool ok = true;
    if (nb > 0) {
      // block matrices into TMEM: row f of super-block lo + j, input features
      // [64 e, 64 e + 64) as 32 columns of two bf16
      for (int j = 0; j < g; ++j) {
        const uint4* src = reinterpret_cast<const uint4*>(
            a.Bmat + (static_cast<int64_t>(lo + j) * 128 + f) * 128 + 64 * e);
        uint32_t w[32];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 x = __ldg(src + u);
          w[4 * u] = x.x;
          w[4 * u + 1] = x.y;
          w[4 * u + 2] = x.z;
          w[4 * u + 3] = x.w;
        }
        tmem_st_32x32b_x32(tmem_base + kB + 64 * j + 32 * e + lane_off, w);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bload);
    }
    const int ntiles = nb * g;
    // nothing of this group before the band of its first tile
    if (!GATHER && leader)
      st_release_cta(&group_done[e], static_cast<uint32_t>(e < ntiles ? e / g : nb));
    for (int it = e; it < ntiles && ok; it += 2) {
      const int i = it / g, j = it % g;
      const int k = s + i * a.S;
      const uint32_t acc_phase = (it >> 1) & 1;
      const bool w = xwait(&tfull[e], acc_phase, tmo, abort_flag, a.abort_word);
      if (named_barrier_any(bar_id, 128, !w)) {  // leave together: a named barrier has no deadline
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t v[2][32];
      tmem_ld_32x32b_x32(tmem_base + kD + e * 64 + lane_off, v[0]);
      tmem_ld_32x32b_x32(tmem_base + kD + e * 64 + 32 + lane_off, v[1]);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&tempty[e]);
      if (GATHER && leader) bulk_wait_read_le<0>();  // the group's previous store has read ob
      named_barrier(bar_id, 128);
      // tile [64 tokens][128 features] as two 64-feature boxes with 128-byte
      // swizzle: feature f of token t at box f / 64, row t, 16-byte chunk
      // ((f % 64) / 8) ^ (t % 8), element f % 8
      {
        uint8_t* box = ob + (f / 64) * Cfg::BOX;
        const int fc = (f % 64) / 8, fe = f % 8;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const __nv_bfloat16 bv = __float2bfloat16_rn(__uint_as_float(v[c >> 5][c & 31]));
          *reinterpret_cast<__nv_bfloat16*>(box + c * 128 + ((fc ^ (c & 7)) << 4) + 2 * fe) = bv;
        }
      }
      const int x = (lo + j) * 128;
      if constexpr (GATHER) {
        fence_proxy_async_smem();
        named_barrier(bar_id, 128);
        if (leader) {
          if (x < a.d) tma_store_2d(&tmOut, ob, x, k * 64);
          if (x + 64 < a.d) tma_store_2d(&tmOut, ob + Cfg::BOX, x + 64, k * 64);
          bulk_commit();
        }
      } else {
        named_barrier(bar_id, 128);
        // the ring entry may be written once its previous band was read
        bool wok = true;
        if (it - 2 < i * g)
          wok = poll_cta_geq(ring_ok, static_cast<uint32_t>(i + 1), tmo, abort_flag, a.abort_word);
        if (named_barrier_any(bar_id, 128, !wok)) {
          ok = false;
          break;
        }
        // 64 rows x 16 chunks of 16 bytes: thread gt copies chunks gt, gt + 128, ...
        uint16_t* rrow = a.ring + static_cast<int64_t>(k % a.E) * 64 * a.d;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int cid = gt + 128 * u;
          const int t = cid >> 4, cc = cid & 15;
          if (x + 8 * cc < a.d) {
            uint4 val;
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(val.x), "=r"(val.y), "=r"(val.z), "=r"(val.w)
                         : "r"(smem_u32(ob + (cc >> 3) * Cfg::BOX + t * 128 + (((cc & 7) ^ (t & 7)) << 4))));
            *reinterpret_cast<uint4*>(rrow + static_cast<int64_t>(t) * a.d + x + 8 * cc) = val;
          }
        }
        const bool last = (it + 2 >= (i + 1) * g);
        if (last) fence_proxy_async_global();  // before the band is published (bulk-copy readers)
        named_barrier(bar_id, 128);
        // done with every band before the next one holding a tile of this group
        if (last && leader) {
          const int next = (it + 2 < ntiles) ? (it + 2) / g : nb;
          st_release_cta(&group_done[e], static_cast<uint32_t>(next));
        }
      }
    }
    if (GATHER && leader) bulk_wait_le<0>();
    if constexpr (RED) {
      // reduction rows f of super-block lo + j, columns [64 e, 64 e + 64)
      const bool have = (nb > 0) && xwait(gdone, 0, tmo, abort_flag, a.abort_word);
      if (have) tc_fence_after();
      for (int j = 0; j < g; ++j) {
        float* out = a.partial + (static_cast<int64_t>(s) * a.nsb + lo + j) * 128 * 128 +
                     static_cast<int64_t>(f) * 128 + 64 * e;
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          uint32_t r[32];
          if (nb > 0) {
            tmem_ld_32x32b_x32(tmem_base + 128 * j + 64 * e + 32 * c + lane_off, r);
            tmem_ld_wait();
          }
          if (!have) {
#pragma unroll
            for (int u = 0; u < 32; ++u) r[u] = 0u;
          }
#pragma unroll
          for (int u = 0; u < 8; ++u)
            reinterpret_cast<uint4*>(out + 32 * c)[u] =
                make_uint4(r[4 * u], r[4 * u + 1], r[4 * u + 2], r[4 * u + 3]);
        }
      }
    }
  } else if (warp < 18) {
    // ------------------------------------------------------------ band side
    // The CTA's rows form one sequence over its bands: item n is row
    // j = n % nr of band n / nr (local row r = q + Q j).  Band warp w takes
    // items w, w + aw, ...: one bulk copy per row into one of its bpw
    // buffers, then the row permuted with the 16-bit indices in shared
    // memory (16-byte chunks, one per lane at a time).  warp_done[w] counts
    // its finished items (GATHER: rows written; SCATTER: ring rows loaded).
    const int w = warp - 10;
    const int d = a.d;
    const int vpr = d / 8;                                  // 16-byte chunks per row
    const uint32_t rowb = static_cast<uint32_t>(d) * 2;
    const int N = nb * nr;                                  // items of this CTA
    const int mine = (w < a.aw && w < N) ? (N - 1 - w) / a.aw + 1 : 0;  // items of this warp
    const int bpw = a.bpw;
    uint8_t* wbuf = bstage + static_cast<size_t>(w) * bpw * rowb;
    uint64_t* wbar = bfull + w * Cfg::MAX_BPW;
    const uint32_t idx_s = smem_u32(idx16);
    auto item = [&](int m) { return w + a.aw * m; };       // the warp's m-th item
    int polled = -1;  // SCATTER: last band known to be produced (lane 0)
    // Issues the warp's m-th row copy (lane 0).  In SCATTER the row exists
    // only once all Q CTAs produced its band: with `block` false the call
    // returns false without issuing when they have not, so issue-ahead never
    // waits.
    auto issue = [&](int m, bool block) -> bool {
      const int n = item(m), i = n / nr;
      const int k = s + i * a.S, r = q + a.Q * (n % nr);
      if (!GATHER && i > polled) {
        if (block) {
          if (!poll_geq(a.produced + k, static_cast<uint32_t>(a.Q), tmo, abort_flag, a.abort_word))
            return false;
        } else if (ld_acquire_u32(a.produced + k) < static_cast<uint32_t>(a.Q)) {
          return false;
        }
        fence_proxy_async_global();
        polled = i;
      }
      const int64_t t = static_cast<int64_t>(k) * 64 + r;
      const int b = m % bpw;
      mbar_arrive_expect_tx(&wbar[b], t < a.T ? rowb : 0u);
      if (t < a.T) {
        const int64_t src = GATHER ? t : static_cast<int64_t>(k % a.E) * 64 + r;
        bulk_load(wbuf + static_cast<size_t>(b) * rowb, a.band_src + src * d, rowb, &wbar[b]);
      }
      return true;
    };
    int next_issue = 0;  // the warp's items below it are issued (lane 0 keeps the count)
    int gated = -1;      // GATHER: last band whose ring entry is known to be free (lane 0)
    bool ok = true;
    if (lane == 0)
      while (next_issue < bpw && next_issue < mine && issue(next_issue, false)) ++next_issue;
    int mfail = -1;
    for (int m = 0; m < mine; ++m) {
      const int n = item(m), i = n / nr;
      const int k = s + i * a.S, r = q + a.Q * (n % nr);
      if (lane == 0 && ok && next_issue == m) {  // not issued ahead: wait for its band, then issue
        ok = issue(m, true);
        if (ok) ++next_issue;
      }
      if (lane == 0 && ok && GATHER && !a.ring_full && i > gated) {
        // the ring entry's previous band must have been loaded by all Q CTAs
        if (k >= a.E &&
            !poll_geq(a.consumed + (k - a.E), static_cast<uint32_t>(a.Q), tmo, abort_flag, a.abort_word))
          ok = false;
        gated = i;
      }
      if (ok) ok = xwait(&wbar[m % bpw], static_cast<uint32_t>((m / bpw) & 1), tmo, abort_flag, a.abort_word);
      if (__any_sync(0xffffffffu, !ok)) {  // one decision for the warp
        ok = false;
        mfail = m;
        break;
      }
      // SCATTER: this ring row is in shared memory
      if (!GATHER && lane == 0) st_release_cta(&warp_done[w], static_cast<uint32_t>(m + 1));
      const int64_t t = static_cast<int64_t>(k) * 64 + r;
      const int64_t drow = (GATHER && !a.ring_full) ? static_cast<int64_t>(k % a.E) * 64 + r : t;
      uint4* orow = reinterpret_cast<uint4*>(a.band_dst + drow * d);
      if (t < a.T) {
        const uint32_t row = smem_u32(wbuf + static_cast<size_t>(m % bpw) * rowb);
#pragma unroll 4
        for (int c = lane; c < vpr; c += 32) {
          uint4 iv;
          asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(iv.x), "=r"(iv.y), "=r"(iv.z), "=r"(iv.w)
                       : "r"(idx_s + 16u * static_cast<uint32_t>(c)));
          const int4 i0 = make_int4(iv.x & 0xffff, iv.x >> 16, iv.y & 0xffff, iv.y >> 16);
          const int4 i1 = make_int4(iv.z & 0xffff, iv.z >> 16, iv.w & 0xffff, iv.w >> 16);
          orow[c] = gather8(row, i0, i1);
        }
      } else if (GATHER && !a.ring_full) {
        // ring rows past the last token are zero (they meet zero rows of the
        // reduction's second operand; stale data could hold non-finite values)
        for (int c = lane; c < vpr; c += 32) orow[c] = make_uint4(0u, 0u, 0u, 0u);
      }
      if (GATHER) fence_proxy_async_global();  // before the row is published (TMA readers)
      __syncwarp();  // the buffer is read and this item's row is written by every lane
      if (lane == 0) {
        if (GATHER) st_release_cta(&warp_done[w], static_cast<uint32_t>(m + 1));
        // issue ahead into the buffer now free, as far as the bands are ready
        while (next_issue <= m + bpw && next_issue < mine && issue(next_issue, false)) ++next_issue;
      }
    }
    // copies still landing must complete before the shared memory is released
    if (lane == 0 && mfail >= 0) {
      volatile int never = 0;
      for (int m = mfail; m < next_issue; ++m)
        mbar_wait(&wbar[m % bpw], static_cast<uint32_t>((m / bpw) & 1), tmo, &never);
    }
  } else {
    // ------------------------------------------------------------ signaling
    // warp 18: produced[k] (GATHER: every band warp of the CTA wrote its rows
    // of band k, adding this CTA's row count; SCATTER: both epilogue groups
    // wrote their tiles, adding 1).  warp 19: consumed[k] (GATHER: the MMA
    // issuer has the band's tiles in shared memory, adding 1; SCATTER: every
    // band warp has its ring rows, adding this CTA's row count).  Each role
    // publishes every band completed so far behind one GPU-scope release
    // fence, so its cost is shared by all the bands that completed meanwhile.
    // warp 20 (SCATTER): ring gate, band i's entry free once consumed[k - E]
    // is full.
    // Bands whose rows every band warp has finished (at least `need`): warp w
    // has finished its items below w + aw * warp_done[w], so every item below
    // the minimum of those is finished, and with it every band below
    // minimum / nr.
    const int N = nb * nr;
    const int nwarps = min(a.aw, N);
    auto warps_progress = [&](uint32_t need, uint32_t* got) -> bool {
      const uint32_t need_items = min(need * static_cast<uint32_t>(nr), static_cast<uint32_t>(N));
      uint32_t lo_item = 0xffffffffu;
      for (int w = 0; w < nwarps; ++w) {
        // items of warp w below need_items: the count it must have finished
        const uint32_t cnt = need_items > static_cast<uint32_t>(w)
                                 ? (need_items - 1 - w) / a.aw + 1 : 0u;
        if (!poll_cta_geq(&warp_done[w], cnt, tmo, abort_flag, a.abort_word)) return false;
        const uint32_t mine_w = (N - 1 - w) / a.aw + 1;
        const uint32_t done = ld_acquire_cta(&warp_done[w]);
        const uint32_t next = done >= mine_w ? static_cast<uint32_t>(N) : w + a.aw * done;
        lo_item = min(lo_item, next);
      }
      *got = lo_item / static_cast<uint32_t>(nr);
      return true;
    };
    auto groups_progress = [&](uint32_t need, uint32_t* got) -> bool {
      if (!poll_cta_geq(&group_done[0], need, tmo, abort_flag, a.abort_word) ||
          !poll_cta_geq(&group_done[1], need, tmo, abort_flag, a.abort_word))
        return false;
      *got = min(ld_acquire_cta(&group_done[0]), ld_acquire_cta(&group_done[1]));
      return true;
    };
    auto mma_progress = [&](uint32_t need, uint32_t* got) -> bool {
      if (!poll_cta_geq(mma_loaded, need, tmo, abort_flag, a.abort_word)) return false;
      *got = ld_acquire_cta(mma_loaded);
      return true;
    };
    // publishes bands [i, got) into cnt[], adding `add` to each: one release
    // fence, then relaxed adds (each forms a release pattern with the fence)
    auto publish = [&](uint32_t* cnt, int i, uint32_t got, uint32_t add) {
      const int end = min(static_cast<int>(got), nb);
      asm volatile("fence.acq_rel.gpu;" ::: "memory");
      for (int b = i; b < end; ++b)
        asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(cnt + (s + b * a.S)), "r"(add)
                     : "memory");
      return end;
    };
    const int role = warp - 18;
    if (lane != 0) {
      // idle lanes
    } else if (role == 0 && !(GATHER && nr == 0)) {
      for (int i = 0; i < nb;) {
        uint32_t got = 0;
        const bool ok = GATHER ? warps_progress(static_cast<uint32_t>(i + 1), &got)
                               : groups_progress(static_cast<uint32_t>(i + 1), &got);
        if (!ok) break;
        i = publish(a.produced, i, got, GATHER ? static_cast<uint32_t>(nr) : 1u);
      }
    } else if (role == 1 && !(GATHER && a.ring_full) && !(!GATHER && nr == 0)) {
      for (int i = 0; i < nb;) {
        uint32_t got = 0;
        const bool ok = GATHER ? mma_progress(static_cast<uint32_t>(i + 1), &got)
                               : warps_progress(static_cast<uint32_t>(i + 1), &got);
        if (!ok) break;
        i = publish(a.consumed, i, got, GATHER ? 1u : static_cast<uint32_t>(nr));
      }
    } else if (role == 2 && !GATHER) {
      for (int i = 0; i < nb; ++i) {
        const int k = s + i * a.S;
        if (k >= a.E && !poll_geq(a.consumed + (k - a.E), 64u, tmo, abort_flag, a.abort_word)) break;
        st_release_cta(ring_ok, static_cast<uint32_t>(i + 1));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

}  // namespace poetx
