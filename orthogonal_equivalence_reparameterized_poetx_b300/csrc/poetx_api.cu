// C ABI of the POET-X layer (declared in include/poetx.h): argument checks,
// buffer layouts, host-side permutation generation, and the launch sequence
// of the forward, backward, build and merge passes.
//
// Passages followed ("POET-X: Memory-efficient LLM Training by Scaling
// Orthogonal Transformation", gist.science summary, Methodologie):
//   §1 input-centric evaluation: Y = R(W0(P x)) as maps on the input;
//   §2 permutations as index maps, two of four merged into the weight;
//   §3 block-diagonal factors as independent small matrices;
//   §4 Cayley-Neumann parameterisation from packed upper triangles;
//   §5 gradient checkpointing (recompute v and h in the backward).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "poetx.h"
#include "ptx.cuh"
#include "simt.cuh"
#include "tc_gemm.cuh"
#include "tc_bdgr.cuh"
#include "tc_bdgr256.cuh"
#include "tc_gbd.cuh"
#include "tc_merge.cuh"
#include "tc_f32gemm.cuh"
#include "tc_gemm2.cuh"
#include "tc_gemm_r.cuh"
#include "tc_gemm_p.cuh"
#include "tc_gemm2r.cuh"
#include "cayley_cluster.cuh"
#include "tc_neumann.cuh"
#include "tc_neumann_bwd.cuh"

using namespace poetx;

namespace {

constexpr size_t kAlign = 256;
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;
uint64_t g_timeout_ns = kDefaultTimeoutNs;

inline size_t align_up(size_t x, size_t a = kAlign) { return (x + a - 1) / a * a; }

// ------------------------------------------------------------------ profiling
std::atomic<int64_t> g_launches{0};

struct ProfRecord {
  int kind;
  cudaEvent_t start, stop;
};

struct Profiler {
  std::mutex mu;
  bool on = false;
  std::vector<ProfRecord> recs;
  std::vector<cudaEvent_t> pool;
  cudaEvent_t get() {
    if (!pool.empty()) {
      cudaEvent_t e = pool.back();
      pool.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
  }
};
Profiler g_prof;

// Records a timing event on `st`.  Inside a stream capture the record becomes
// an event-record node of the graph (an external record), so each replay of
// the graph times the captured launches.
void prof_record(cudaEvent_t e, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(e, st, cudaEventRecordExternal);
  else
    cudaEventRecord(e, st);
}

// Brackets the launches made during its lifetime with events on `st`.
struct ProfScope {
  int kind;
  cudaStream_t st;
  cudaEvent_t start = nullptr;
  ProfScope(int k, cudaStream_t s) : kind(k), st(s) {
    if (!g_prof.on) return;
    std::lock_guard<std::mutex> lock(g_prof.mu);
    start = g_prof.get();
    prof_record(start, st);
  }
  ~ProfScope() {
    if (!start) return;
    std::lock_guard<std::mutex> lock(g_prof.mu);
    cudaEvent_t stop = g_prof.get();
    prof_record(stop, st);
    g_prof.recs.push_back(ProfRecord{kind, start, stop});
  }
};

// ------------------------------------------------------------------ permutations
// splitmix64 (Steele, Lea & Flood, OOPSLA 2014) drives a Fisher-Yates shuffle;
// a draw in [0, bound) rejects values at or above the largest multiple of
// bound representable in 2^64 and reduces the rest modulo bound.
struct SplitMix64 {
  uint64_t state;
  uint64_t next() {
    state += 0x9E3779B97F4A7C15ull;
    uint64_t z = state;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
  }
};

uint64_t draw_below(SplitMix64& g, uint64_t bound) {
  // 2^64 mod bound, computed without 128-bit arithmetic
  const uint64_t rem = (0 - bound) % bound;           // (2^64 - bound) mod bound
  const uint64_t limit = 0 - rem;                      // 2^64 - rem (wraps to 0 if rem == 0)
  for (;;) {
    const uint64_t r = g.next();
    if (rem == 0 || r < limit) return r % bound;
  }
}

void make_permutation(uint64_t seed, int d, int32_t* out) {
  for (int i = 0; i < d; ++i) out[i] = i;
  SplitMix64 g{seed};
  for (int i = d - 1; i >= 1; --i) {
    const int j = static_cast<int>(draw_below(g, static_cast<uint64_t>(i) + 1));
    std::swap(out[i], out[j]);
  }
}

// ------------------------------------------------------------------ layouts

struct SideLayout {
  SideGeom g;
  int sb, nsb;          // tensor-core super-block size and count
  size_t off_B, off_M, off_Q;
  size_t off_Bsb, off_BsbT;
  size_t off_s1, off_s2, off_s3;  // build scratch
  size_t bb() const { return static_cast<size_t>(g.b) * g.b; }
};

struct ParamsLayout {
  size_t off_piR, off_piRinv, off_piP, off_piPinv;
  SideLayout R, P;
  size_t total;
};

SideGeom side_geom(int d, int b) {
  SideGeom s;
  s.d = d;
  s.b = b;
  s.nblk = (d + b - 1) / b;
  s.last = d - (s.nblk - 1) * b;
  return s;
}

void layout_side(SideLayout& L, int d, int b, const poetx_layer_desc& desc, size_t& off) {
  L.g = side_geom(d, b);
  L.sb = std::max(b, 128);
  L.nsb = (d + L.sb - 1) / L.sb;
  const size_t mat = static_cast<size_t>(L.g.nblk) * b * b * sizeof(float);
  L.off_B = off; off = align_up(off + mat);
  L.off_M = off; off = align_up(off + mat);
  L.off_Q = off; off = align_up(off + mat);
  if (desc.dtype == POETX_DTYPE_BF16) {
    const size_t sbm = static_cast<size_t>(L.nsb) * L.sb * L.sb * sizeof(__nv_bfloat16);
    L.off_Bsb = off; off = align_up(off + sbm);
    L.off_BsbT = off; off = align_up(off + sbm);
  } else {
    L.off_Bsb = L.off_BsbT = 0;
  }
  // scratch: exact b > 128 needs column panel (b x 128), pivot inverse
  // (128 x 128) and row panel (128 x b) per block; Neumann needs two b x b.
  size_t s1 = 0, s2 = 0, s3 = 0;
  if (desc.mode == POETX_MODE_NEUMANN) {
    s1 = s2 = mat;
  } else if (b > 128) {
    s1 = static_cast<size_t>(L.g.nblk) * b * 128 * sizeof(float);
    s2 = static_cast<size_t>(L.g.nblk) * 128 * 128 * sizeof(float);
    s3 = s1;
  }
  L.off_s1 = off; off = align_up(off + s1);
  L.off_s2 = off; off = align_up(off + s2);
  L.off_s3 = off; off = align_up(off + s3);
}

ParamsLayout params_layout(const poetx_layer_desc& d) {
  ParamsLayout L{};
  size_t off = 0;
  L.off_piR = off; off = align_up(off + sizeof(int32_t) * d.m);
  L.off_piRinv = off; off = align_up(off + sizeof(int32_t) * d.m);
  L.off_piP = off; off = align_up(off + sizeof(int32_t) * d.n);
  L.off_piPinv = off; off = align_up(off + sizeof(int32_t) * d.n);
  layout_side(L.R, d.m, d.b_R, d, off);
  layout_side(L.P, d.n, d.b_P, d, off);
  L.total = off;
  return L;
}

// GradRed token splits: the smallest split count whose tiles keep at least 95%
// of one wave's SMs busy (few partials to reduce), each split a multiple of 64
// tokens; the count is recomputed from the rounded chunk so that every split
// holds at least one token.
struct Splits {
  int splits, chunk;
};

// Token splits of the separate reduction: `units` CTAs (or CTA pairs) each
// taking tile x tile output tiles of the sb x sb products.
Splits gradred_splits(const SideLayout& S, int64_t T, int nsm, int tile = 128) {
  const int tps = S.sb / tile;
  const int per_split = S.nsb * tps * tps;
  const int64_t Tc = std::max<int64_t>(T, 1);
  const int64_t smax = std::max<int64_t>(1, std::min<int64_t>((4 * nsm + per_split - 1) / per_split,
                                                              (Tc + 63) / 64));
  int64_t target = smax;
  for (int64_t sp = 1; sp <= smax; ++sp) {
    const int64_t tiles = sp * per_split;
    const int64_t rounds = (tiles + nsm - 1) / nsm;
    if (tiles * 100 >= 95 * rounds * nsm) {
      target = sp;
      break;
    }
  }
  const int64_t per = (Tc + target - 1) / target;
  const int64_t chunk = (per + 63) / 64 * 64;
  const int64_t splits = (Tc + chunk - 1) / chunk;
  return Splits{static_cast<int>(splits), static_cast<int>(chunk)};
}

struct WorkLayout {
  size_t off_n1, off_n2, off_m1, off_m2, off_m3;
  size_t off_partR, off_partP, off_GR, off_GP, off_t1, off_t2, off_nsc, off_wdq;
  int splitsR, splitsP;
  size_t total;
};

// SM count of the device current at the first call (148 when no device can be
// queried, e.g. for the size functions on a host without a GPU).
int device_sm_count() {
  static const int nsm = [] {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      return 148;
    return n;
  }();
  return nsm;
}

// SMs the library's persistent launches size their grids for.
int launch_sms() { return device_sm_count(); }

// Upper bound on the reduction partial slots written for T tokens: GradRed
// token splits or the fused transform + reduction's token slots.
int64_t partial_slots_bound(const SideLayout& S, int64_t T) {
  auto bound = [&](int tile, int units) {
    const int tps = S.sb / tile;
    const int64_t per_split = static_cast<int64_t>(S.nsb) * tps * tps;
    return std::max<int64_t>(
        1, std::min<int64_t>((4 * static_cast<int64_t>(units) + per_split - 1) / per_split, (T + 63) / 64));
  };
  int64_t smax = bound(128, device_sm_count());
  if (S.sb >= 256) smax = std::max(smax, bound(256, std::max(1, device_sm_count() / 2)));
  const int64_t fused = std::max<int64_t>(1, device_sm_count() / S.nsb);
  return std::max(smax, fused);
}

// Pre-merged weight buffer: m x n of the dtype, or (POET-XQ) m x n int8
// codes followed, at the next 256-byte boundary, by m float32 row scales.
bool weight_int8(const poetx_layer_desc& d) { return d.weight_format == POETX_WEIGHT_INT8; }
size_t weight_codes_bytes(const poetx_layer_desc& d) {
  return align_up(static_cast<size_t>(d.m) * d.n);
}
size_t weight_bytes(const poetx_layer_desc& d) {
  if (weight_int8(d)) return weight_codes_bytes(d) + align_up(static_cast<size_t>(d.m) * 4);
  return static_cast<size_t>(d.m) * d.n * (d.dtype == POETX_DTYPE_BF16 ? 2 : 4);
}

WorkLayout work_layout(const poetx_layer_desc& d, const ParamsLayout& P, int64_t T, int nsm) {
  WorkLayout W{};
  const size_t e = d.dtype == POETX_DTYPE_BF16 ? 2 : 4;
  const size_t tn = static_cast<size_t>(T) * d.n * e, tm = static_cast<size_t>(T) * d.m * e;
  size_t off = 0;
  W.off_n1 = off; off = align_up(off + tn);
  W.off_n2 = off; off = align_up(off + tn);
  W.off_m1 = off; off = align_up(off + tm);
  W.off_m2 = off; off = align_up(off + tm);
  W.off_m3 = off; off = align_up(off + tm);
  W.splitsR = W.splitsP = 0;
  if (d.dtype == POETX_DTYPE_BF16) {
    W.splitsR = static_cast<int>(partial_slots_bound(P.R, T));
    W.splitsP = static_cast<int>(partial_slots_bound(P.P, T));
    W.off_partR = off;
    off = align_up(off + static_cast<size_t>(W.splitsR) * P.R.nsb * P.R.sb * P.R.sb * 4);
    W.off_partP = off;
    off = align_up(off + static_cast<size_t>(W.splitsP) * P.P.nsb * P.P.sb * P.P.sb * 4);
  } else {
    W.off_partR = W.off_partP = off;
  }
  const size_t gR = static_cast<size_t>(P.R.g.nblk) * P.R.bb() * 4;
  const size_t gP = static_cast<size_t>(P.P.g.nblk) * P.P.bb() * 4;
  const size_t gmax = std::max(gR, gP);
  W.off_GR = off; off = align_up(off + gR);
  W.off_GP = off; off = align_up(off + gP);
  W.off_t1 = off; off = align_up(off + gmax);
  W.off_t2 = off; off = align_up(off + gmax);
  W.off_nsc = off;
  // Neumann scratch: the batched chain rule keeps k + 3 matrices per side;
  // the fused tensor-core backward keeps five per side for both sides
  if (d.mode == POETX_MODE_NEUMANN) off = align_up(off + gmax * std::max(d.neumann_k + 3, 10));
  W.off_wdq = off;  // dequantized int8 weight (bf16 m x n)
  if (weight_int8(d)) off = align_up(off + static_cast<size_t>(d.m) * d.n * 2);
  W.total = off;
  return W;
}

// ------------------------------------------------------------------ checks

poetx_status check_desc(const poetx_layer_desc* d) {
  if (!d) return POETX_ERR_INVALID_ARG;
  if (d->m < 1 || d->n < 1 || d->b_R < 1 || d->b_P < 1 || d->b_R > d->m || d->b_P > d->n)
    return POETX_ERR_INVALID_ARG;
  if (d->mode != POETX_MODE_CAYLEY && d->mode != POETX_MODE_NEUMANN) return POETX_ERR_INVALID_ARG;
  if (d->mode == POETX_MODE_NEUMANN && (d->neumann_k < 1 || d->neumann_k > 6))
    return POETX_ERR_INVALID_ARG;
  if (d->dtype != POETX_DTYPE_FP32 && d->dtype != POETX_DTYPE_BF16) return POETX_ERR_INVALID_ARG;
  if (d->weight_format != POETX_WEIGHT_DENSE && d->weight_format != POETX_WEIGHT_INT8)
    return POETX_ERR_INVALID_ARG;
  if (d->weight_format == POETX_WEIGHT_INT8 && d->dtype != POETX_DTYPE_BF16) return POETX_ERR_UNSUPPORTED;
  auto b_ok_fp32 = [](int b) { return b <= 128 || (b % 128 == 0 && b <= 1024); };
  auto b_ok_bf16 = [](int b) { return b == 32 || b == 64 || b == 128 || b == 256 || b == 512; };
  if (d->dtype == POETX_DTYPE_FP32) {
    if (!b_ok_fp32(d->b_R) || !b_ok_fp32(d->b_P)) return POETX_ERR_UNSUPPORTED;
  } else {
    if (d->m % 8 || d->n % 8) return POETX_ERR_UNSUPPORTED;
    if (!b_ok_bf16(d->b_R) || !b_ok_bf16(d->b_P)) return POETX_ERR_UNSUPPORTED;
  }
  return POETX_OK;
}

inline bool aligned(const void* p, size_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

#define POETX_CUDA(...)                          \
  do {                                           \
    if ((__VA_ARGS__) != cudaSuccess) {          \
      (void)cudaGetLastError();                  \
      return POETX_ERR_CUDA;                     \
    }                                            \
  } while (0)

#define POETX_LAUNCHED()                         \
  do {                                           \
    g_launches.fetch_add(1, std::memory_order_relaxed); \
    if (cudaGetLastError() != cudaSuccess) return POETX_ERR_CUDA; \
  } while (0)

#define POETX_TRY(...)                           \
  do {                                           \
    poetx_status _s = (__VA_ARGS__);             \
    if (_s != POETX_OK) return _s;               \
  } while (0)

// ------------------------------------------------------------------ launch helpers

// Programmatic dependent launch of the layer's pass kernels (on by default).
// A kernel launched this way may be scheduled while the previous kernel of
// the stream drains: its CTAs initialise their barriers and tensor memory,
// then wait in griddep_enter for that kernel's completion before their first
// global-memory access.  This hides the launch gap and the set-up of each
// kernel behind the tail of the one before it.
//
// Only passes over at most kDependentLaunchMaxBytes of activation (and the
// small fixed-size generator and optimizer kernels) are launched this way.
// Measured on B300 (20-step means, two runs each): the LLaMA-60M-shaped block
// (passes of 8-23 MB, about 5 us each) goes from 0.714 to 0.666 ms per step,
// while with every pass launched this way the d = 4096 FFN pair went from
// 35.6-35.8 to 36.5-36.6 ms and the d = 2048 block from 17.27-17.33 to
// 17.40-17.44 ms; with dependents released only as CTAs exit instead of at
// entry, neither gained nor lost.
std::atomic<bool> g_dependent_launch{true};
constexpr int64_t kDependentLaunchMaxBytes = int64_t(32) << 20;

// Launches `kern` (a kernel that calls griddep_enter on every path) on `st`
// and counts the launch.  `pass_bytes`: size of the activation the pass
// reads or writes (0 for fixed-size work), which decides the launch form.
template <typename... KArgs, typename... Args>
poetx_status launch_dep(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                        int64_t pass_bytes, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed =
      (g_dependent_launch.load(std::memory_order_relaxed) && pass_bytes <= kDependentLaunchMaxBytes)
          ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...) != cudaSuccess) {
    (void)cudaGetLastError();
    return POETX_ERR_CUDA;
  }
  return POETX_OK;
}

int grid_for(int64_t work, int per_block = 256, int max_blocks = 148 * 16) {
  const int64_t g = (work + per_block - 1) / per_block;
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(g, max_blocks)));
}

template <typename TA, typename TB, typename TC>
poetx_status simt_gemm(cudaStream_t st, int M, int N, int K, int batch, const TA* A, int64_t sAm,
                       int64_t sAk, int64_t bsA, const TB* B, int64_t sBk, int64_t sBn, int64_t bsB,
                       TC* C, int64_t sCm, int64_t sCn, int64_t bsC, float alpha, float beta) {
  if (M <= 0 || N <= 0 || batch <= 0) return POETX_OK;
  SimtGemmArgs g{M, N, K, batch, A, sAm, sAk, bsA, B, sBk, sBn, bsB, C, sCm, sCn, bsC, alpha, beta};
  if (M >= 128 && N >= 128) {
    dim3 grid((N + 127) / 128, (M + 127) / 128, batch);
    return launch_dep(simt_gemm128_kernel<TA, TB, TC>, grid, 256, 0, st,
                      int64_t(M) * N * batch * int64_t(sizeof(TC)), g);
  }
  dim3 grid((N + 63) / 64, (M + 63) / 64, batch);
  return launch_dep(simt_gemm_kernel<TA, TB, TC>, grid, 256, 0, st, int64_t(M) * N * batch * int64_t(sizeof(TC)),
                    g);
}

// Narrowest bf16 rows (bytes) for which the pipelined gather takes several
// rows per pass instead of the pair-interleaved kernel.  Measured on B300:
// 2 KB rows (d1024 block) 1.33 -> 1.23 ms of gathers per step; at 1 KB rows
// (LLaMA-60M, 8192 tokens) the pair-interleaved kernel stays faster (0.280
// vs 0.299 ms per step).
constexpr size_t kNarrowGatherMinBytes = 2048;

template <typename T>
poetx_status gather_cols(cudaStream_t st, const T* in, T* out, const int32_t* idx, int64_t rows,
                         int d) {
  if (rows <= 0) return POETX_OK;
  ProfScope prof(POETX_KIND_GATHER, st);
  if ((static_cast<size_t>(d) * sizeof(T)) % 16 != 0) {
    const int grid = static_cast<int>(std::min<int64_t>(rows, launch_sms() * 8));
    return launch_dep(gather_cols_scalar_kernel<T>, grid, 256, 0, st, rows * d * int64_t(sizeof(T)), in, out, idx, rows, d);
  }
  const size_t row_bytes = static_cast<size_t>(d) * sizeof(T);
  if constexpr (sizeof(T) == 2) {
    // rows of at least 4 KB: persistent CTAs (three per SM) with two blocks
    // of rows (about 32 KB each) in flight per CTA.  Narrower rows keep the
    // pair-interleaved kernel below, whose short per-CTA iterations suit the
    // smaller passes (measured on B300: the pipelined kernel is 18% faster at
    // d = 2048 and 5% slower at d = 1024; three CTAs of 32 KB blocks beat two
    // of 48 KB by 2% at d = 2048 and 5% at d = 4096).
    const int rb = static_cast<int>(std::max<size_t>(1, std::min<size_t>(32, (32 * 1024) / row_bytes)));
    const size_t psmem = 2 * rb * row_bytes + 64;
    const int vpr = d / 8;
    const bool narrow = row_bytes >= kNarrowGatherMinBytes && vpr < 256 && 256 % vpr == 0;
    if ((row_bytes >= 4096 || narrow) && psmem <= 200 * 1024) {
      // the chunk indices of rows of up to 1024 (6 * 256 for wider rows)
      // 16-byte chunks stay in registers
      const bool wide = vpr > 4 * 256;
      auto kern = narrow ? gather_rows_pipelined_kernel<1, true>
                         : (wide ? gather_rows_pipelined_kernel<6, false> : gather_rows_pipelined_kernel<4, false>);
      static cudaError_t attr1 = cudaFuncSetAttribute(
          gather_rows_pipelined_kernel<1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
      static cudaError_t attr4 = cudaFuncSetAttribute(
          gather_rows_pipelined_kernel<4, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
      static cudaError_t attr6 = cudaFuncSetAttribute(
          gather_rows_pipelined_kernel<6, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
      if (attr1 != cudaSuccess || attr4 != cudaSuccess || attr6 != cudaSuccess) return POETX_ERR_CUDA;
      const int64_t nblocks = (rows + rb - 1) / rb;
      const int grid = static_cast<int>(std::min<int64_t>(nblocks, launch_sms() * 3));
      return launch_dep(kern, grid, 256, psmem, st, rows * d * 2, reinterpret_cast<const uint16_t*>(in),
                        reinterpret_cast<uint4*>(out), idx, rows, d, rb, g_timeout_ns);
    }
    // interleaved row pairs, about 32 KB staged per iteration (at least one pair)
    const int ppi = static_cast<int>(std::max<size_t>(1, std::min<size_t>(8, (16 * 1024) / row_bytes)));
    const size_t smem = 2 * row_bytes * ppi;
    if (smem > 48 * 1024) {
      static std::once_flag once2;
      std::call_once(once2, [] {
        cudaFuncSetAttribute(gather_cols_bf16x2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             200 * 1024);
      });
      if (smem > 200 * 1024) return POETX_ERR_UNSUPPORTED;
    }
    const int64_t iters = (rows + 2 * ppi - 1) / (2 * ppi);
    const int grid = static_cast<int>(std::min<int64_t>(iters, launch_sms() * 6));
    return launch_dep(gather_cols_bf16x2_kernel, grid, 256, smem, st, rows * d * 2,
                      reinterpret_cast<const uint4*>(in), reinterpret_cast<uint4*>(out), idx, rows,
                      d, ppi);
  }
  // stage about 32 KB of rows per iteration (at least one row)
  const int rpi = static_cast<int>(std::max<size_t>(1, std::min<size_t>(16, (32 * 1024) / row_bytes)));
  const size_t smem = row_bytes * rpi;
  if (smem > 48 * 1024) {
    static std::once_flag once;
    std::call_once(once, [] {
      cudaFuncSetAttribute(gather_cols_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           200 * 1024);
    });
    if (smem > 200 * 1024) return POETX_ERR_UNSUPPORTED;
  }
  const int64_t iters = (rows + rpi - 1) / rpi;
  const int grid = static_cast<int>(std::min<int64_t>(iters, launch_sms() * 8));
  return launch_dep(gather_cols_kernel<T>, grid, 256, smem, st, rows * d * int64_t(sizeof(T)), in, out, idx, rows, d, rpi);
}

// ------------------------------------------------------------------ tensor maps

typedef CUresult (*PFN_encodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                    const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                    const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                    CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

PFN_encodeTiled get_encode_fn() {
  static PFN_encodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_encodeTiled>(p);
  });
  return fn;
}

// Row-major bf16 matrix [rows][cols] with leading dimension ld (elements);
// box = box_rows x 64 columns, 128-byte swizzle, zero fill out of bounds.
poetx_status tmap_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                       uint64_t ld, uint32_t box_rows) {
  PFN_encodeTiled enc = get_encode_fn();
  if (!enc) return POETX_ERR_CUDA;
  if (!aligned(base, 16) || (ld * 2) % 16 != 0) return POETX_ERR_MISALIGNED;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? POETX_OK : POETX_ERR_CUDA;
}

// Row-major bf16 matrix [rows][cols] staged as unswizzled boxes of 256
// columns x box_rows rows (zero fill out of bounds).
poetx_status tmap_bf16_rows(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                            uint32_t box_rows) {
  PFN_encodeTiled enc = get_encode_fn();
  if (!enc) return POETX_ERR_CUDA;
  if (!aligned(base, 16) || (cols * 2) % 16 != 0) return POETX_ERR_MISALIGNED;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {256, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? POETX_OK : POETX_ERR_CUDA;
}

template <int BN, bool A_MN, bool B_MN, TileMode MODE, typename OutT>
poetx_status launch_tc(cudaStream_t st, const CUtensorMap& ta, const CUtensorMap& tb,
                       const CUtensorMap& tc, TcGemmArgs args) {
  if (args.num_tiles <= 0) return POETX_OK;
  auto kern = tc_gemm_kernel<BN, A_MN, B_MN, MODE, OutT>;
  constexpr int smem = TcGemmCfg<BN, MODE != TileMode::GradRed>::SMEM_BYTES;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  });
  if (attr_err != cudaSuccess) return POETX_ERR_CUDA;
  args.timeout_ns = g_timeout_ns;
  const int grid = std::min(args.num_tiles, launch_sms());
  const int64_t pass_bytes = MODE == TileMode::GradRed
                                 ? int64_t(args.tokens) * args.nsb * args.sb * 2
                                 : int64_t(args.M) * args.N * 2;
  return launch_dep(kern, grid, 320, smem, st, pass_bytes, ta, tb, tc, args);
}

// CTA-pair kernel (tc_gemm2.cuh) with 256 x 256 tiles, in any tile mode.
template <bool B_MN, PairMode MODE>
poetx_status launch_pair_mode(cudaStream_t st, const CUtensorMap& ta, const CUtensorMap& tb,
                              const CUtensorMap& tc, TcPairArgs a, int64_t pass_bytes) {
  if (a.num_tiles <= 0) return POETX_OK;
  a.timeout_ns = g_timeout_ns;
  auto kern = tc_gemm_pair_kernel<B_MN, MODE>;
  static cudaError_t attr_err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, TcPairCfg::SMEM_BYTES);
  if (attr_err != cudaSuccess) return POETX_ERR_CUDA;
  const int pairs = std::max(1, std::min(a.num_tiles, launch_sms() / 2));
  return launch_dep(kern, 2 * pairs, 320, TcPairCfg::SMEM_BYTES, st, pass_bytes, ta, tb, tc, a);
}

// Dense GEMM on CTA pairs.
template <bool B_MN>
poetx_status launch_pair(cudaStream_t st, const CUtensorMap& ta, const CUtensorMap& tb,
                         const CUtensorMap& tc, int64_t T, int N, int K) {
  TcPairArgs a{};
  a.M = static_cast<int>(T);
  a.N = N;
  a.K = K;
  a.num_tiles = static_cast<int>((T + 255) / 256) * ((N + 255) / 256);
  return launch_pair_mode<B_MN, PairMode::Dense>(st, ta, tb, tc, a, T * N * 2);
}

// Wide outputs (N >= 1024) run on CTA pairs, narrower ones on single CTAs.
bool use_pair(int64_t T, int N) { return N >= 1024 && T >= 256 && launch_sms() >= 2; }

// h (T x N) = A (T x K) * W^T, W row-major N x K (both K-major).
poetx_status tc_dense_nt(cudaStream_t st, const void* A, const void* W, void* C, int64_t T, int N,
                         int K) {
  if (T <= 0) return POETX_OK;
  ProfScope prof(POETX_KIND_GEMM_FWD, st);
  if (use_pair(T, N)) {
    CUtensorMap ta, tb, tc;
    POETX_TRY(tmap_bf16(&ta, A, T, K, K, 128));
    POETX_TRY(tmap_bf16(&tb, W, N, K, K, 128));
    POETX_TRY(tmap_bf16(&tc, C, T, N, N, 128));
    return launch_pair<false>(st, ta, tb, tc, T, N, K);
  }
  const bool wide = N >= 1024;
  const int BN = wide ? 256 : 128;
  CUtensorMap ta, tb, tc;
  POETX_TRY(tmap_bf16(&ta, A, T, K, K, 128));
  POETX_TRY(tmap_bf16(&tb, W, N, K, K, BN));
  POETX_TRY(tmap_bf16(&tc, C, T, N, N, 128));
  TcGemmArgs a{};
  a.M = static_cast<int>(T);
  a.N = N;
  a.K = K;
  a.C = C;
  a.ldc = N;
  a.num_tiles = static_cast<int>((T + 127) / 128) * ((N + BN - 1) / BN);
  if (wide) return launch_tc<256, false, false, TileMode::Dense, __nv_bfloat16>(st, ta, tb, tc, a);
  return launch_tc<128, false, false, TileMode::Dense, __nv_bfloat16>(st, ta, tb, tc, a);
}

// h = v W0'^T and z[:, s] = h[:, s] S_s^T in one launch (tc_gemm_r.cuh),
// for R sides with 128-wide super-blocks; h is written only when H is given.
poetx_status tc_dense_nt_r(cudaStream_t st, const void* V, const void* W, const void* Ssb, void* H,
                           void* Z, int64_t T, int N, int K, int nsb) {
  if (T <= 0) return POETX_OK;
  ProfScope prof(POETX_KIND_GEMM_FWD, st);
  CUtensorMap ta, tb, ts, th, tz;
  POETX_TRY(tmap_bf16(&ta, V, T, K, K, 128));
  POETX_TRY(tmap_bf16(&tb, W, N, K, K, 128));
  POETX_TRY(tmap_bf16(&ts, Ssb, static_cast<uint64_t>(nsb) * 128, 128, 128, 128));
  POETX_TRY(tmap_bf16(&th, H ? H : Z, T, N, N, 128));
  POETX_TRY(tmap_bf16(&tz, Z, T, N, N, 128));
  TcGemmRArgs a{};
  a.M = static_cast<int>(T);
  a.N = N;
  a.K = K;
  a.num_tiles = static_cast<int>((T + 127) / 128) * ((N + 127) / 128);
  a.store_h = H != nullptr;
  a.timeout_ns = g_timeout_ns;
  static cudaError_t attr_err = cudaFuncSetAttribute(
      tc_gemm_r_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, TcGemmRCfg::SMEM);
  if (attr_err != cudaSuccess) return POETX_ERR_CUDA;
  return launch_dep(tc_gemm_r_kernel, std::min(a.num_tiles, launch_sms()), 320, TcGemmRCfg::SMEM, st,
                    T * N * 2, ta, tb, ts, th, tz, a);
}

// The same on CTA pairs with 256 x 256 tiles (tc_gemm2r.cuh), for wide outputs.
poetx_status tc_dense_nt_pair_r(cudaStream_t st, const void* V, const void* W, const void* Ssb, void* H,
                                void* Z, int64_t T, int N, int K, int nsb) {
  if (T <= 0) return POETX_OK;
  ProfScope prof(POETX_KIND_GEMM_FWD, st);
  CUtensorMap ta, tb, ts, th, tz;
  POETX_TRY(tmap_bf16(&ta, V, T, K, K, 128));
  POETX_TRY(tmap_bf16(&tb, W, N, K, K, 128));
  POETX_TRY(tmap_bf16(&ts, Ssb, static_cast<uint64_t>(nsb) * 128, 128, 128, 64));
  POETX_TRY(tmap_bf16(&th, H ? H : Z, T, N, N, 128));
  POETX_TRY(tmap_bf16(&tz, Z, T, N, N, 128));
  TcPairRArgs a{};
  a.M = static_cast<int>(T);
  a.N = N;
  a.K = K;
  a.num_tiles = static_cast<int>((T + 255) / 256) * ((N + 255) / 256);
  a.store_h = H != nullptr;
  a.timeout_ns = g_timeout_ns;
  static cudaError_t attr_err = cudaFuncSetAttribute(
      tc_gemm_pair_r_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, TcPairRCfg::SMEM_BYTES);
  if (attr_err != cudaSuccess) return POETX_ERR_CUDA;
  const int pairs = std::max(1, std::min(a.num_tiles, launch_sms() / 2));
  return launch_dep(tc_gemm_pair_r_kernel, 2 * pairs, 320, TcPairRCfg::SMEM_BYTES, st, T * N * 2, ta, tb,
                    ts, th, tz, a);
}

// Whether the forward runs the R transform in the GEMM epilogue
// (tc_gemm_r.cuh) instead of as a separate pass over h: where the plain
// forward GEMM is the single-CTA 128 x 128 engine as well (outputs narrower
// than 1024), and for outputs of at most kREpilogueMaxBytes.  Measured on
// B300 (20-step means, two runs each), LLaMA-60M-shaped block: 0.587 ms per
// step with no fused epilogue, 0.573 with it on the 512-wide outputs only,
// 0.560 with it also on the 1376-wide ones (22.5 MB).  With the fused kernel
// on every output width: d1024 block 4.24 -> 4.33 ms, d2048 block 17.14 ->
// 18.89 ms and d4096 FFN pair 35.47 -> 39.66 ms, because wide outputs
// otherwise run on CTA pairs with 256 x 256 tiles, which this kernel does not
// have (1.9 ms slower forward GEMMs per d2048 step against 0.95 ms saved in
// the R pass).
constexpr int64_t kREpilogueMaxBytes = int64_t(32) << 20;
bool r_epilogue(const SideLayout& R, int64_t T, int N) {
  return R.sb == 128 && (!use_pair(T, N) || T * N * 2 <= kREpilogueMaxBytes);
}

// Wide outputs: the R transform in the epilogue of the CTA-pair GEMM.
// Measured on B300 against the pair GEMM plus the separate R pass (20-step
// means, two runs each): d1024 block 4.23 -> 4.08 ms per step, d2048 block
// 17.00 -> 16.84 ms, d4096 FFN pair 34.70 -> 34.39 ms.  The forward GEMM
// class itself gets slower (4.06 -> 5.05 ms per d2048 step: four pipeline
// stages instead of six, the transform MMAs, and the extra shared-memory
// traffic of staging h and z) but the R pass (0.95 ms) disappears.
bool pair_r_epilogue(const SideLayout& R, int64_t T, int N) { return R.sb == 128 && use_pair(T, N); }

// dv (T x N) = A (T x K) * W, W row-major K x N (B operand MN-major).
poetx_status tc_dense_nn(cudaStream_t st, const void* A, const void* W, void* C, int64_t T, int N,
                         int K) {
  if (T <= 0) return POETX_OK;
  ProfScope prof(POETX_KIND_GEMM_DGRAD, st);
  if (use_pair(T, N)) {
    CUtensorMap ta, tb, tc;
    POETX_TRY(tmap_bf16(&ta, A, T, K, K, 128));
    POETX_TRY(tmap_bf16(&tb, W, K, N, N, 64));
    POETX_TRY(tmap_bf16(&tc, C, T, N, N, 128));
    return launch_pair<true>(st, ta, tb, tc, T, N, K);
  }
  const bool wide = N >= 1024;
  const int BN = wide ? 256 : 128;
  CUtensorMap ta, tb, tc;
  POETX_TRY(tmap_bf16(&ta, A, T, K, K, 128));
  POETX_TRY(tmap_bf16(&tb, W, K, N, N, 64));
  POETX_TRY(tmap_bf16(&tc, C, T, N, N, 128));
  TcGemmArgs a{};
  a.M = static_cast<int>(T);
  a.N = N;
  a.K = K;
  a.C = C;
  a.ldc = N;
  a.num_tiles = static_cast<int>((T + 127) / 128) * ((N + BN - 1) / BN);
  if (wide) return launch_tc<256, false, true, TileMode::Dense, __nv_bfloat16>(st, ta, tb, tc, a);
  return launch_tc<128, false, true, TileMode::Dense, __nv_bfloat16>(st, ta, tb, tc, a);
}

// dv = dh W0' with du = dv B_P and the dv^T u partials in the epilogue
// (tc_gemm_p.cuh), for P sides with 128-wide super-blocks; dv is not written.
// Adds the partial slots it writes to *slots.
poetx_status tc_dense_nn_p(cudaStream_t st, const SideLayout& P, const void* dh, const void* W,
                           const void* SsbT, const void* u, void* du, float* partial, int64_t T, int N,
                           int K, int* slots) {
  if (T <= 0) return POETX_OK;
  ProfScope prof(POETX_KIND_GEMM_DGRAD, st);
  CUtensorMap ta, tb, ts, tu, tdu;
  POETX_TRY(tmap_bf16(&ta, dh, T, K, K, 128));
  POETX_TRY(tmap_bf16(&tb, W, K, N, N, 64));
  POETX_TRY(tmap_bf16(&ts, SsbT, static_cast<uint64_t>(P.nsb) * 128, 128, 128, 128));
  POETX_TRY(tmap_bf16(&tu, u, T, N, N, 128));
  POETX_TRY(tmap_bf16(&tdu, du, T, N, N, 128));
  TcGemmPArgs a{};
  a.M = static_cast<int>(T);
  a.N = N;
  a.K = K;
  a.nsb = P.nsb;
  a.nslots = std::max(1, launch_sms() / P.nsb);
  a.b = P.g.b;
  a.partial = partial;
  a.timeout_ns = g_timeout_ns;
  static cudaError_t attr_err = cudaFuncSetAttribute(
      tc_gemm_p_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, TcGemmPCfg::SMEM);
  if (attr_err != cudaSuccess) return POETX_ERR_CUDA;
  POETX_TRY(launch_dep(tc_gemm_p_kernel, a.nslots * P.nsb, 320, TcGemmPCfg::SMEM, st, T * N * 2, ta, tb, ts,
                       tu, tdu, a));
  *slots += a.nslots;
  return POETX_OK;
}

// Whether the backward runs the P side's transform and token reduction in
// the dgrad GEMM epilogue (tc_gemm_p.cuh): under the same rule as the
// forward's R epilogue.  Measured on B300 (20-step means): LLaMA-60M-shaped
// block 0.560 -> 0.532 ms per step; with the fused dgrad on every output
// width, d1024 block 4.21 -> 4.39 ms, d2048 block 16.97 -> 18.60 ms and d4096
// FFN pair 34.94 -> 41.17 ms (wide dgrads otherwise run on CTA pairs).
bool p_epilogue(const SideLayout& P, int64_t T, int N) {
  return P.sb == 128 && P.nsb <= launch_sms() && (!use_pair(T, N) || T * N * 2 <= kREpilogueMaxBytes);
}

// out[:, s] = in[:, s] * S_s^T over super-blocks: in/out T x d, Ssb (nsb*sb) x sb.
poetx_status tc_blockdiag(cudaStream_t st, const void* in, const void* Ssb, void* out, int64_t T,
                          int d, int sb, int nsb) {
  if (T <= 0) return POETX_OK;
  ProfScope prof(POETX_KIND_BLOCKDIAG, st);
  // (256 x 256 tiles on CTA pairs with K = sb were measured slower for sb >=
  // 256 than these single-CTA 128 x 256 tiles: d4096 b = 256 block
  // transforms 5.0 vs 3.9 ms per step)
  const int BN = sb >= 256 ? 256 : 128;
  CUtensorMap ta, tb, tc;
  POETX_TRY(tmap_bf16(&ta, in, T, d, d, 128));
  POETX_TRY(tmap_bf16(&tb, Ssb, static_cast<uint64_t>(nsb) * sb, sb, sb, BN));
  POETX_TRY(tmap_bf16(&tc, out, T, d, d, 128));
  TcGemmArgs a{};
  a.M = static_cast<int>(T);
  a.N = d;
  a.sb = sb;
  a.C = out;
  a.ldc = d;
  a.num_tiles = static_cast<int>((T + 127) / 128) * ((d + BN - 1) / BN);
  if (BN == 256) return launch_tc<256, false, false, TileMode::BlockDiag, __nv_bfloat16>(st, ta, tb, tc, a);
  return launch_tc<128, false, false, TileMode::BlockDiag, __nv_bfloat16>(st, ta, tb, tc, a);
}

// partial[p][s] = sum_{t in split p} A[t, s]^T B[t, s] (fp32, sb x sb per super-block).
// Writes sp.splits partial slots starting at `partial` and adds that count to
// *slots (the caller appends the next call's slots after them).
poetx_status tc_gradred(cudaStream_t st, const SideLayout& S, const void* A, const void* B,
                        float* partial, int64_t T, int* slots) {
  const int d = S.g.d, sb = S.sb, nsb = S.nsb;
  if (sb >= 256 && use_pair(T, d)) {  // 256 x 256 tiles of each product on CTA pairs
    const Splits sp = gradred_splits(S, T, std::max(1, launch_sms() / 2), 256);
    *slots += sp.splits;
    ProfScope prof(POETX_KIND_GRADRED, st);
    CUtensorMap ta, tb;
    POETX_TRY(tmap_bf16(&ta, A, T, d, d, 64));
    POETX_TRY(tmap_bf16(&tb, B, T, d, d, 64));
    TcPairArgs a{};
    a.sb = sb;
    a.nsb = nsb;
    a.tokens = static_cast<int>(T);
    a.chunk = sp.chunk;
    a.C = partial;
    a.split_stride = static_cast<int64_t>(nsb) * sb * sb;
    a.num_tiles = sp.splits * nsb * (sb / 256) * (sb / 256);
    return launch_pair_mode<true, PairMode::GradRed>(st, ta, tb, ta, a, T * static_cast<int64_t>(nsb) * sb * 2);
  }
  const Splits sp = gradred_splits(S, T, launch_sms());
  *slots += sp.splits;
  ProfScope prof(POETX_KIND_GRADRED, st);
  CUtensorMap ta, tb;
  POETX_TRY(tmap_bf16(&ta, A, T, d, d, 64));
  POETX_TRY(tmap_bf16(&tb, B, T, d, d, 64));
  TcGemmArgs a{};
  a.sb = sb;
  a.nsb = nsb;
  a.tokens = static_cast<int>(T);
  a.chunk = sp.chunk;
  a.C = partial;
  a.split_stride = static_cast<int64_t>(nsb) * sb * sb;
  const int tps = sb / 128;
  a.num_tiles = sp.splits * nsb * tps * tps;
  return launch_tc<128, true, true, TileMode::GradRed, float>(st, ta, tb, ta, a);
}

// Fused block transform + token reduction for 128-wide super-blocks:
// out = in S^T per super-block and partial slots of in^T C (see tc_bdgr.cuh).
// A fused transform + reduction grid is a whole number of token slots times
// the CTAs of one slot; true when that covers at least 80% of the SMs.
bool fused_grid_fills(int ctas_per_slot) {
  const int sms = launch_sms();
  return ctas_per_slot <= sms && 5 * (sms / ctas_per_slot) * ctas_per_slot >= 4 * sms;
}

// 128-wide super-blocks: fused whenever one slot fits (measured on B300 at
// d = 11008, where one slot covers 86 of 148 SMs, it still beats the separate
// transform and reduction: 4.19 vs 4.37 ms per step at d = 4096, b = 128).
bool bdgr_ok(const SideLayout& S) { return S.sb == 128 && S.nsb <= launch_sms(); }

poetx_status tc_bdgr(cudaStream_t st, const SideLayout& S, const void* in, const void* Ssb,
                     void* out, const void* Cm, float* partial, int64_t T, int* slots) {
  if (T <= 0) return POETX_OK;
  ProfScope prof(POETX_KIND_BLOCKDIAG, st);
  const int d = S.g.d;
  CUtensorMap ta, tsb, tc, to;
  POETX_TRY(tmap_bf16(&ta, in, T, d, d, 128));
  POETX_TRY(tmap_bf16(&tsb, Ssb, static_cast<uint64_t>(S.nsb) * 128, 128, 128, 128));
  POETX_TRY(tmap_bf16(&tc, Cm, T, d, d, 128));
  POETX_TRY(tmap_bf16(&to, out, T, d, d, 128));
  BdgrArgs a{};
  a.M = static_cast<int>(T);
  a.N = d;
  a.nsb = S.nsb;
  a.nslots = std::max(1, launch_sms() / S.nsb);
  a.b = S.g.b;
  a.partial = partial;
  a.timeout_ns = g_timeout_ns;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(tc_bdgr_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    BdgrCfg::SMEM);
  });
  if (attr_err != cudaSuccess) return POETX_ERR_CUDA;
  POETX_TRY(launch_dep(tc_bdgr_kernel, a.nslots * S.nsb, 320, BdgrCfg::SMEM, st, int64_t(a.M) * a.N * 2, ta, tsb, tc, to, a));
  *slots += a.nslots;
  return POETX_OK;
}

// Column permutation fused into the block transform (tc_gbd.cuh): sides of
// 256 to g_gbd_max_cols features, 128-wide super-blocks; off by default.
// Every CTA of a token tile stages its whole rows to use 128 of their
// columns, so the staged bytes grow with d while the launch it saves is a
// fixed cost.  Measured on B300 (20-step means, two runs each, same box):
// LLaMA-60M-shaped block 0.538 ms per step with the 512-wide sides fused and
// 0.576 with every side up to 1536 fused, against 0.534 with the separate
// passes; d1024 block 4.35 against 3.96 ms.  The fused kernels' own time is
// below that of the two kernels they replace (LLaMA-60M: about 50 us per
// step less in the library's per-class events), but in the graph-replayed,
// dependent-launched step the light gather kernels overlap their neighbours
// and nothing is gained.
constexpr int kGbdDefaultMaxCols = 0;
std::atomic<int> g_gbd_max_cols{kGbdDefaultMaxCols};

bool gbd_ok(const SideLayout& S) {
  return S.sb == 128 && S.nsb <= launch_sms() && S.g.d >= 256 &&
         S.g.d <= g_gbd_max_cols.load(std::memory_order_relaxed);
}

// A = src[:, perm]; out = A S^T per super-block; with REDUCE also the partial
// slots of A^T C (appended at *slots); a_out (may be null) receives A.
template <bool REDUCE>
poetx_status tc_gather_bd(cudaStream_t st, const SideLayout& S, const __nv_bfloat16* src,
                          const int32_t* perm, const void* Ssb, void* out, void* a_out, const void* Cm,
                          float* partial, int64_t T, int* slots) {
  if (T <= 0) return POETX_OK;
  ProfScope prof(POETX_KIND_BLOCKDIAG, st);
  using Cfg = GbdCfg<REDUCE>;
  const int d = S.g.d;
  GbdArgs a{};
  a.M = static_cast<int>(T);
  a.N = d;
  a.nsb = S.nsb;
  a.nslots = std::max(1, launch_sms() / S.nsb);
  a.b = S.g.b;
  // staged chunks: a power of two of rows (so a chunk never straddles two
  // token tiles), as large as lets two chunks be in flight, and up to four
  a.nbox = (d + 255) / 256;
  const int row_bytes = a.nbox * 512;
  a.chunk_rows = 128;
  while (a.chunk_rows > 1 && 2 * a.chunk_rows * row_bytes > Cfg::STG_BYTES) a.chunk_rows /= 2;
  if (2 * a.chunk_rows * row_bytes > Cfg::STG_BYTES || d % 8 != 0) return POETX_ERR_UNSUPPORTED;
  a.nstg = std::min(Cfg::MAX_SLOTS, Cfg::STG_BYTES / (a.chunk_rows * row_bytes));
  a.store_a = a_out != nullptr;
  a.perm = perm;
  a.partial = partial;
  a.timeout_ns = g_timeout_ns;
  CUtensorMap tx, ts, tc, to, ta;
  POETX_TRY(tmap_bf16_rows(&tx, src, T, d, a.chunk_rows));
  POETX_TRY(tmap_bf16(&ts, Ssb, static_cast<uint64_t>(S.nsb) * 128, 128, 128, 128));
  POETX_TRY(tmap_bf16(&tc, REDUCE ? Cm : out, T, d, d, 128));
  POETX_TRY(tmap_bf16(&to, out, T, d, d, 128));
  POETX_TRY(tmap_bf16(&ta, a_out ? a_out : out, T, d, d, 128));
  auto kern = tc_gbd_kernel<REDUCE>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
  });
  if (attr_err != cudaSuccess) return POETX_ERR_CUDA;
  POETX_TRY(launch_dep(kern, a.nslots * S.nsb, Cfg::THREADS, Cfg::SMEM, st, T * d * 2, tx, ts, tc, to, ta, a));
  if (REDUCE) *slots += a.nslots;
  return POETX_OK;
}

// 256-wide super-blocks: two CTAs per super-block and token slot (one per
// half of its output features), tiles of 64 tokens (tc_bdgr256.cuh).  Used
// only when its grid fills the GPU (measured on B300 at d = 11008, 86 of 148
// SMs: 5.94 ms per step against 5.16 for the separate passes at d = 4096,
// b = 256; at d = 2048 it saves 0.3 ms per step).
bool bdgr256_ok(const SideLayout& S) { return S.sb == 256 && fused_grid_fills(2 * S.nsb); }

poetx_status tc_bdgr256(cudaStream_t st, const SideLayout& S, const void* in, const void* Ssb, void* out,
                        const void* Cm, float* partial, int64_t T, int* slots) {
  if (T <= 0) return POETX_OK;
  ProfScope prof(POETX_KIND_BLOCKDIAG, st);
  const int d = S.g.d;
  CUtensorMap ta, tc, to;
  POETX_TRY(tmap_bf16(&ta, in, T, d, d, 64));
  POETX_TRY(tmap_bf16(&tc, Cm, T, d, d, 64));
  POETX_TRY(tmap_bf16(&to, out, T, d, d, 64));
  if (!aligned(Ssb, 16)) return POETX_ERR_MISALIGNED;
  Bdgr256Args a{};
  a.S = reinterpret_cast<const __nv_bfloat16*>(Ssb);
  a.M = static_cast<int>(T);
  a.N = d;
  a.nsb = S.nsb;
  a.nslots = std::max(1, launch_sms() / (2 * S.nsb));
  a.partial = partial;
  a.timeout_ns = g_timeout_ns;
  static cudaError_t attr_err = cudaFuncSetAttribute(
      tc_bdgr256_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Bdgr256Cfg::SMEM);
  if (attr_err != cudaSuccess) return POETX_ERR_CUDA;
  POETX_TRY(launch_dep(tc_bdgr256_kernel, a.nslots * S.nsb * 2, 320, Bdgr256Cfg::SMEM, st,
                       int64_t(a.M) * a.N * 2, ta, tc, to, a));
  *slots += a.nslots;
  return POETX_OK;
}

// One tensor-core merge pass (tc_merge.cuh): with A = Ahi (+ Alo), M x N
// row-major, and the super-blocks D = Dhi + Dlo of B - I over the N columns,
// writes (A B^T)^T = (A + A D^T)^T as out_hi (+ out_lo), N x M row-major.
template <bool A_SPLIT>
poetx_status tc_merge_pass(cudaStream_t st, const __nv_bfloat16* Ahi, const __nv_bfloat16* Alo, int M,
                           int N, int sb, int nsb, const __nv_bfloat16* Dhi, const __nv_bfloat16* Dlo,
                           __nv_bfloat16* out_hi, __nv_bfloat16* out_lo) {
  CUtensorMap tah, tal, tdh, tdl;
  POETX_TRY(tmap_bf16(&tah, Ahi, M, N, N, 128));
  POETX_TRY(tmap_bf16(&tal, A_SPLIT ? Alo : Ahi, M, N, N, 128));
  POETX_TRY(tmap_bf16(&tdh, Dhi, static_cast<uint64_t>(nsb) * sb, sb, sb, 128));
  POETX_TRY(tmap_bf16(&tdl, Dlo, static_cast<uint64_t>(nsb) * sb, sb, sb, 128));
  MergeArgs a{};
  a.M = M;
  a.N = N;
  a.sb = sb;
  a.num_tiles = ((M + 127) / 128) * ((N + 127) / 128);
  a.res_hi = Ahi;
  a.res_lo = A_SPLIT ? Alo : nullptr;
  a.out_hi = out_hi;
  a.out_lo = out_lo;
  a.timeout_ns = g_timeout_ns;
  auto kern = tc_merge_kernel<A_SPLIT>;
  constexpr int smem = MergeCfg<A_SPLIT>::SMEM;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  });
  if (attr_err != cudaSuccess) return POETX_ERR_CUDA;
  kern<<<std::min(a.num_tiles, launch_sms()), 320, smem, st>>>(tah, tal, tdh, tdl, a);
  POETX_LAUNCHED();
  return POETX_OK;
}

// An fp32 operand of tc_f32_gemm: element (r, k) of batch z at
// p[z * bs + r * rs + k * cs]; rs == 1 or cs == 1.
struct F32Operand {
  const float* p;
  int64_t rs, cs, bs;
};

// 3-D fp32 tensor map (contiguous index, other index, batch), no swizzle.
poetx_status tmap_f32_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                         uint64_t s1_bytes, uint64_t s2_bytes, uint32_t box0, uint32_t box1) {
  PFN_encodeTiled enc = get_encode_fn();
  if (!enc) return POETX_ERR_CUDA;
  if (!aligned(base, 16) || s1_bytes % 16 != 0 || s2_bytes % 16 != 0) return POETX_ERR_MISALIGNED;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {s1_bytes, s2_bytes};
  cuuint32_t box[3] = {box0, box1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? POETX_OK : POETX_ERR_CUDA;
}

// Tensor map of an operand with `rows` rows and K columns per batch; sets
// *kcontig.  UNSUPPORTED when neither stride is 1 or the strides are not
// multiples of 16 bytes.
poetx_status f32_operand_map(CUtensorMap* map, const F32Operand& o, int rows, int K, int batch,
                             bool* kcontig) {
  const uint64_t s2 = static_cast<uint64_t>(std::max<int64_t>(o.bs, 1)) * 4;
  if (o.cs == 1 && (o.rs * 4) % 16 == 0 && s2 % 16 == 0) {
    *kcontig = true;
    return tmap_f32_3d(map, o.p, K, rows, batch, o.rs * 4, s2, 64, 128);
  }
  if (o.rs == 1 && (o.cs * 4) % 16 == 0 && s2 % 16 == 0) {
    *kcontig = false;
    return tmap_f32_3d(map, o.p, rows, K, batch, o.cs * 4, s2, 128, 64);
  }
  return POETX_ERR_UNSUPPORTED;
}

template <bool AK, bool BK>
poetx_status launch_f32gemm(cudaStream_t st, const CUtensorMap& ta, const CUtensorMap& tb,
                            const F32GemmArgs& a, int tiles, int batch) {
  auto kern = tc_f32gemm_kernel<AK, BK>;
  static cudaError_t attr_err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, F32GemmCfg::SMEM);
  if (attr_err != cudaSuccess) return POETX_ERR_CUDA;
  return launch_dep(kern, dim3(tiles, batch), 320, F32GemmCfg::SMEM, st, 0, ta, tb, a);
}

// Batched C = alpha A B^T + beta C on the tensor cores with fp32-grade
// products (tc_f32gemm.cuh); A is M x K, B is N x K, C row-major (unit
// column stride) with row stride c_rs and batch stride c_bs.
poetx_status tc_f32_gemm(cudaStream_t st, int M, int N, int K, int batch, const F32Operand& A,
                         const F32Operand& B, float* C, int64_t c_rs, int64_t c_bs, float alpha,
                         float beta) {
  if (M <= 0 || N <= 0 || batch <= 0) return POETX_OK;
  if (K <= 0) return POETX_ERR_INVALID_ARG;
  CUtensorMap ta, tb;
  bool ak = false, bk = false;
  POETX_TRY(f32_operand_map(&ta, A, M, K, batch, &ak));
  POETX_TRY(f32_operand_map(&tb, B, N, K, batch, &bk));
  F32GemmArgs a{};
  a.M = M;
  a.N = N;
  a.K = K;
  a.c = C;
  a.c_rs = c_rs;
  a.c_bs = c_bs;
  a.alpha = alpha;
  a.beta = beta;
  a.timeout_ns = g_timeout_ns;
  const int tiles = ((M + 127) / 128) * ((N + 127) / 128);
  if (ak && bk) return launch_f32gemm<true, true>(st, ta, tb, a, tiles, batch);
  if (ak) return launch_f32gemm<true, false>(st, ta, tb, a, tiles, batch);
  if (bk) return launch_f32gemm<false, true>(st, ta, tb, a, tiles, batch);
  return launch_f32gemm<false, false>(st, ta, tb, a, tiles, batch);
}

// C = alpha A B + beta C with the strides of simt_gemm (A(i,k) = A[i sAm +
// k sAk], B(k,j) = B[k sBk + j sBn]): on the tensor cores when `tc` (bf16
// layers, fp32-grade products) and on the CUDA cores otherwise.
poetx_status dense_f32_gemm(bool tc, cudaStream_t st, int M, int N, int K, int batch, const float* A,
                            int64_t sAm, int64_t sAk, int64_t bsA, const float* B, int64_t sBk,
                            int64_t sBn, int64_t bsB, float* C, int64_t sCm, int64_t sCn, int64_t bsC,
                            float alpha, float beta) {
  if (tc && M >= 64 && N >= 64 && K >= 64 && sCn == 1) {
    const F32Operand a{A, sAm, sAk, bsA}, b{B, sBn, sBk, bsB};
    const poetx_status r = tc_f32_gemm(st, M, N, K, batch, a, b, C, sCm, bsC, alpha, beta);
    if (r != POETX_ERR_UNSUPPORTED && r != POETX_ERR_MISALIGNED) return r;
  }
  return simt_gemm<float, float, float>(st, M, N, K, batch, A, sAm, sAk, bsA, B, sBk, sBn, bsB, C, sCm,
                                        sCn, bsC, alpha, beta);
}

// ------------------------------------------------------------------ builder

bool fused_cayley_ok(const poetx_layer_desc& d, int b) {
  return d.mode == POETX_MODE_CAYLEY && (b <= 128 || b == 256 || b == 512);
}

CayleySide cayley_side(const poetx_layer_desc& d, const SideLayout& S, const float* gen,
                       uint8_t* params) {
  const bool bf = d.dtype == POETX_DTYPE_BF16;
  CayleySide c;
  c.gen = gen;
  c.s = S.g;
  c.B = reinterpret_cast<float*>(params + S.off_B);
  c.M = reinterpret_cast<float*>(params + S.off_M);
  c.Q = reinterpret_cast<float*>(params + S.off_Q);
  c.sb = S.sb;
  c.nsb = S.nsb;
  c.Bsb = bf ? reinterpret_cast<__nv_bfloat16*>(params + S.off_Bsb) : nullptr;
  c.BsbT = bf ? reinterpret_cast<__nv_bfloat16*>(params + S.off_BsbT) : nullptr;
  return c;
}

// Exact Cayley blocks of one side, or of both sides at once when `second`
// is given (same block size), in a single launch.
poetx_status launch_cayley_blocks(cudaStream_t st, const poetx_layer_desc& d, const CayleySide& a,
                                  const CayleySide* second) {
  const int b = a.s.b;
  const int grid_blocks = a.s.nblk + (second ? second->s.nblk : 0);
  if (b == 256 || b == 512) {
    // one cluster per block
    static std::once_flag once_cluster;
    std::call_once(once_cluster, [] {
      cudaFuncSetAttribute(cayley_cluster_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(CcCfg<256>::SMEM));
      cudaFuncSetAttribute(cayley_cluster_kernel<512>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(CcCfg<512>::SMEM));
    });
    if (b == 256)
      cayley_cluster_kernel<256><<<CcCfg<256>::C * grid_blocks, CcCfg<256>::NT, CcCfg<256>::SMEM, st>>>(
          a, second ? *second : a);
    else
      cayley_cluster_kernel<512><<<CcCfg<512>::C * grid_blocks, CcCfg<512>::NT, CcCfg<512>::SMEM, st>>>(
          a, second ? *second : a);
    POETX_LAUNCHED();
    return POETX_OK;
  }
  static std::once_flag once;
  std::call_once(once, [] {
    const int lim = 128 * 129 * 4;
    cudaFuncSetAttribute(cayley_block_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
    cudaFuncSetAttribute(cayley_block_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
    cudaFuncSetAttribute(cayley_block_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
    cudaFuncSetAttribute(cayley_block_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
  });
  const size_t smem = d.dtype == POETX_DTYPE_BF16 ? static_cast<size_t>(b) * (b + 1) * 4 : 0;
  const int R = std::min(b, 1024 / b);
  const int grid = grid_blocks;
  auto kern = b == 128 ? cayley_block_kernel<128>
            : b == 64  ? cayley_block_kernel<64>
            : b == 32  ? cayley_block_kernel<32>
                       : cayley_block_kernel<0>;
  kern<<<grid, b * R, smem, st>>>(a, second ? *second : a);
  POETX_LAUNCHED();
  return POETX_OK;
}

// bf16 layers build 128-, 256- and 512-wide Neumann blocks in one launch
// with fp32-grade tensor-core products; fp32 layers keep CUDA-core products
// (the split-bf16 products are not fp32 round-off).
bool fused_neumann_ok(const poetx_layer_desc& d, int b) {
  return d.mode == POETX_MODE_NEUMANN && d.dtype == POETX_DTYPE_BF16 &&
         (b == 128 || b == 256 || b == 512);
}

NeumannSide neumann_side(const SideLayout& S, const float* gen, uint8_t* params) {
  NeumannSide n;
  n.gen = gen;
  n.s = S.g;
  n.B = reinterpret_cast<float*>(params + S.off_B);
  n.Q = reinterpret_cast<float*>(params + S.off_Q);
  n.S0 = reinterpret_cast<float*>(params + S.off_s1);
  n.S1 = reinterpret_cast<float*>(params + S.off_s2);
  n.sb = S.sb;
  n.Bsb = reinterpret_cast<__nv_bfloat16*>(params + S.off_Bsb);
  n.BsbT = reinterpret_cast<__nv_bfloat16*>(params + S.off_BsbT);
  return n;
}

template <int BS>
void launch_neumann_kernel(cudaStream_t st, const NeumannSide& a, const NeumannSide& b2, int blocks,
                           int k) {
  using Cfg = NeuCfg<BS>;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(tc_neumann_kernel<BS>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
  });
  tc_neumann_kernel<BS><<<Cfg::C * blocks, Cfg::THREADS, Cfg::SMEM, st>>>(a, b2, k, g_timeout_ns);
}

// Neumann blocks of one side, or of both sides at once when `second` is
// given (same block size), in a single launch.
poetx_status launch_neumann_blocks(cudaStream_t st, const poetx_layer_desc& d, const NeumannSide& a,
                                   const NeumannSide* second) {
  const int blocks = a.s.nblk + (second ? second->s.nblk : 0);
  const NeumannSide& b2 = second ? *second : a;
  switch (a.s.b) {
    case 128: launch_neumann_kernel<128>(st, a, b2, blocks, d.neumann_k); break;
    case 256: launch_neumann_kernel<256>(st, a, b2, blocks, d.neumann_k); break;
    case 512: launch_neumann_kernel<512>(st, a, b2, blocks, d.neumann_k); break;
    default: return POETX_ERR_UNSUPPORTED;
  }
  POETX_LAUNCHED();
  return POETX_OK;
}

poetx_status build_side(cudaStream_t st, const poetx_layer_desc& d, const SideLayout& S,
                        const float* gen, uint8_t* params) {
  ProfScope prof(POETX_KIND_BUILD, st);
  float* B = reinterpret_cast<float*>(params + S.off_B);
  float* M = reinterpret_cast<float*>(params + S.off_M);
  float* Q = reinterpret_cast<float*>(params + S.off_Q);
  const int b = S.g.b, nb = S.g.nblk;
  const int64_t bb = static_cast<int64_t>(b) * b;
  if (fused_cayley_ok(d, b)) {
    POETX_TRY(launch_cayley_blocks(st, d, cayley_side(d, S, gen, params), nullptr));
    return POETX_OK;
  }
  if (fused_neumann_ok(d, b)) return launch_neumann_blocks(st, d, neumann_side(S, gen, params), nullptr);
  // bf16 layers run the dense products of the build on the tensor cores
  // with fp32-grade (split bf16) operands; fp32 layers keep fp32 CUDA cores
  const bool tcg = d.dtype == POETX_DTYPE_BF16;
  unpack_kernel<<<dim3(nb, (b + 7) / 8), 256, 0, st>>>(gen, S.g, Q, M);
  POETX_LAUNCHED();
  if (d.mode == POETX_MODE_CAYLEY) {
    {
      // b > 128: block Gauss-Jordan with 128-wide panels: for panel k,
      // C = A[:, k], D = A_kk^-1, R = D A[k, :], A -= C R, A[k, :] = R,
      // A[:, k] = -C D, A_kk = D.
      float* Cc = reinterpret_cast<float*>(params + S.off_s1);
      float* D = reinterpret_cast<float*>(params + S.off_s2);
      float* Rr = reinterpret_cast<float*>(params + S.off_s3);
      const int P = 128;
      for (int k = 0; k < b / P; ++k) {
        const int o = k * P;
        copy2d_kernel<<<dim3(grid_for(static_cast<int64_t>(b) * P), nb), 256, 0, st>>>(
            M + o, bb, b, Cc, static_cast<int64_t>(b) * P, P, b, P, 1.f, 0.f);
        POETX_LAUNCHED();
        gj_invert128_kernel<<<nb, 1024, 0, st>>>(M + static_cast<int64_t>(o) * b + o, bb, b, D,
                                                 static_cast<int64_t>(P) * P, P);
        POETX_LAUNCHED();
        POETX_TRY(dense_f32_gemm(tcg, st, P, b, P, nb, D, P, 1, static_cast<int64_t>(P) * P,
                                                 M + static_cast<int64_t>(o) * b, b, 1, bb, Rr, b, 1,
                                                 static_cast<int64_t>(P) * b, 1.f, 0.f));
        POETX_TRY(dense_f32_gemm(tcg, st, b, b, P, nb, Cc, P, 1, static_cast<int64_t>(b) * P,
                                                 Rr, b, 1, static_cast<int64_t>(P) * b, M, b, 1, bb,
                                                 -1.f, 1.f));
        copy2d_kernel<<<dim3(grid_for(static_cast<int64_t>(b) * P), nb), 256, 0, st>>>(
            Rr, static_cast<int64_t>(P) * b, b, M + static_cast<int64_t>(o) * b, bb, b, P, b, 1.f, 0.f);
        POETX_LAUNCHED();
        POETX_TRY(dense_f32_gemm(tcg, st, b, P, P, nb, Cc, P, 1, static_cast<int64_t>(b) * P,
                                                 D, P, 1, static_cast<int64_t>(P) * P, M + o, b, 1, bb,
                                                 -1.f, 0.f));
        copy2d_kernel<<<dim3(grid_for(static_cast<int64_t>(P) * P), nb), 256, 0, st>>>(
            D, static_cast<int64_t>(P) * P, P, M + static_cast<int64_t>(o) * b + o, bb, b, P, P, 1.f,
            0.f);
        POETX_LAUNCHED();
      }
    }
    // B = 2M - I
    copy2d_kernel<<<dim3(grid_for(bb), nb), 256, 0, st>>>(M, bb, b, B, bb, b, b, b, 2.f, -1.f);
    POETX_LAUNCHED();
  } else {
    // Neumann: S_0 = I, S_i = I + Q S_{i-1} (i = 1..k), B = S_k + Q S_k.
    float* Sa = reinterpret_cast<float*>(params + S.off_s1);
    float* Sb = reinterpret_cast<float*>(params + S.off_s2);
    copy2d_kernel<<<dim3(grid_for(bb), nb), 256, 0, st>>>(Q, bb, b, Sa, bb, b, b, b, 0.f, 1.f);
    POETX_LAUNCHED();
    for (int i = 1; i <= d.neumann_k; ++i) {
      copy2d_kernel<<<dim3(grid_for(bb), nb), 256, 0, st>>>(Q, bb, b, Sb, bb, b, b, b, 0.f, 1.f);
      POETX_LAUNCHED();
      POETX_TRY(dense_f32_gemm(tcg, st, b, b, b, nb, Q, b, 1, bb, Sa, b, 1, bb, Sb, b, 1,
                                               bb, 1.f, 1.f));
      std::swap(Sa, Sb);
    }
    copy2d_kernel<<<dim3(grid_for(bb), nb), 256, 0, st>>>(Sa, bb, b, B, bb, b, b, b, 1.f, 0.f);
    POETX_LAUNCHED();
    POETX_TRY(dense_f32_gemm(tcg, st, b, b, b, nb, Q, b, 1, bb, Sa, b, 1, bb, B, b, 1, bb,
                                             1.f, 1.f));
  }
  if (d.dtype == POETX_DTYPE_BF16) {
    auto* Bsb = reinterpret_cast<__nv_bfloat16*>(params + S.off_Bsb);
    auto* BsbT = reinterpret_cast<__nv_bfloat16*>(params + S.off_BsbT);
    superblock_kernel<<<grid_for(static_cast<int64_t>(S.nsb) * S.sb * S.sb), 256, 0, st>>>(
        B, S.g, S.sb, S.nsb, Bsb, BsbT);
    POETX_LAUNCHED();
  }
  return POETX_OK;
}

// dL/dQ from dL/dB per block (fp32), then packed into dGen.
poetx_status generator_backward(cudaStream_t st, const poetx_layer_desc& d, const SideLayout& S,
                                const uint8_t* params, const float* G, float* t1, float* t2,
                                float* nsc, float* dGen, int accumulate) {
  ProfScope prof(POETX_KIND_GENBWD, st);
  const int b = S.g.b, nb = S.g.nblk;
  const int64_t bb = static_cast<int64_t>(b) * b;
  const float* M = reinterpret_cast<const float*>(params + S.off_M);
  const float* Q = reinterpret_cast<const float*>(params + S.off_Q);
  float* GQ = t2;
  const bool tcg = d.dtype == POETX_DTYPE_BF16;  // tensor-core products for bf16 layers
  if (d.mode == POETX_MODE_CAYLEY) {
    // dL/dQ = 2 M^T G M^T
    POETX_TRY(dense_f32_gemm(tcg, st, b, b, b, nb, M, 1, b, bb, G, b, 1, bb, t1, b, 1, bb,
                                             1.f, 0.f));
    POETX_TRY(dense_f32_gemm(tcg, st, b, b, b, nb, t1, b, 1, bb, M, 1, b, bb, GQ, b, 1,
                                             bb, 2.f, 0.f));
  } else {
    // B = sum_p c_p Q^p (c_0 = 1, c_1..c_k = 2, c_{k+1} = 1), so
    // dL/dQ = sum_{a+c <= k} c_{a+c+1} Qt^a G Qt^c with Qt = Q^T.
    // R_c = G Qt^c; T_a = sum_c c_{a+c+1} R_c; dL/dQ = T_0 + Qt(T_1 + Qt(... T_k)).
    const int k = d.neumann_k;
    const int64_t tstride = static_cast<int64_t>(nb) * bb;
    float* R = nsc;                          // R_0 .. R_k
    float* cur = nsc + (k + 1) * tstride;    // Horner accumulator
    float* nxt = t1;
    POETX_TRY(launch_dep(copy2d_kernel, dim3(grid_for(bb), nb), 256, 0, st, 0, G, bb, b, R, bb, b, b, b,
                         1.f, 0.f));
    for (int c = 1; c <= k; ++c)  // R_c = R_{c-1} Qt
      POETX_TRY(dense_f32_gemm(tcg, st, b, b, b, nb, R + (c - 1) * tstride, b, 1, bb, Q,
                                               1, b, bb, R + c * tstride, b, 1, bb, 1.f, 0.f));
    auto coef = [&](int p) { return (p == 0 || p == k + 1) ? 1.f : 2.f; };
    for (int a = k; a >= 0; --a) {
      float* dst = (a == k) ? cur : nxt;  // T_a
      POETX_TRY(launch_dep(copy2d_kernel, dim3(grid_for(bb), nb), 256, 0, st, 0, R, bb, b, dst, bb, b, b, b,
                           coef(a + 1), 0.f));
      for (int c = 1; c <= k - a; ++c)
        POETX_TRY(launch_dep(axpy_kernel, grid_for(tstride), 256, 0, st, 0, dst, R + c * tstride,
                             coef(a + c + 1), tstride));
      if (a != k) {  // nxt = T_a + Qt cur
        POETX_TRY(dense_f32_gemm(tcg, st, b, b, b, nb, Q, 1, b, bb, cur, b, 1, bb, nxt, b,
                                                 1, bb, 1.f, 1.f));
        std::swap(cur, nxt);
      }
    }
    GQ = cur;
  }
  return launch_dep(pack_grad_kernel, dim3(nb, (b + 7) / 8), 256, 0, st, 0, GQ, S.g, dGen, accumulate);
}

}  // namespace

namespace {

// ------------------------------------------------------------------ pinned staging
// Host-generated permutations reach the device through a small ring of
// pinned host slots, so the copies stay asynchronous.  A slot is reused only
// after the copy that last read it has executed (an event wait that only
// blocks if the ring wraps before the stream reaches that copy).
struct PinnedRing {
  std::mutex mu;
  uint8_t* buf = nullptr;
  size_t slot_bytes = 0;
  static constexpr int kSlots = 32;
  cudaEvent_t ev[kSlots] = {};
  bool pending[kSlots] = {};
  int next = 0;
};
PinnedRing g_ring;

poetx_status ring_upload(cudaStream_t st, const std::vector<std::pair<const int32_t*, size_t>>& parts,
                         const std::vector<void*>& dsts) {
  std::lock_guard<std::mutex> lock(g_ring.mu);
  size_t need = 0;
  for (auto& p : parts) need += align_up(p.second * sizeof(int32_t), 16);
  if (need > g_ring.slot_bytes) {
    for (int s = 0; s < PinnedRing::kSlots; ++s)
      if (g_ring.pending[s]) POETX_CUDA(cudaEventSynchronize(g_ring.ev[s]));
    if (g_ring.buf) POETX_CUDA(cudaFreeHost(g_ring.buf));
    g_ring.buf = nullptr;
    const size_t slot = align_up(std::max<size_t>(need, 1 << 16), 4096);
    POETX_CUDA(cudaHostAlloc(reinterpret_cast<void**>(&g_ring.buf), slot * PinnedRing::kSlots,
                             cudaHostAllocDefault));
    g_ring.slot_bytes = slot;
    for (int s = 0; s < PinnedRing::kSlots; ++s) {
      if (!g_ring.ev[s]) POETX_CUDA(cudaEventCreateWithFlags(&g_ring.ev[s], cudaEventDisableTiming));
      g_ring.pending[s] = false;
    }
  }
  const int s = g_ring.next;
  g_ring.next = (s + 1) % PinnedRing::kSlots;
  if (g_ring.pending[s]) POETX_CUDA(cudaEventSynchronize(g_ring.ev[s]));
  uint8_t* base = g_ring.buf + static_cast<size_t>(s) * g_ring.slot_bytes;
  size_t off = 0;
  for (size_t i = 0; i < parts.size(); ++i) {
    const size_t bytes = parts[i].second * sizeof(int32_t);
    std::memcpy(base + off, parts[i].first, bytes);
    POETX_CUDA(cudaMemcpyAsync(dsts[i], base + off, bytes, cudaMemcpyHostToDevice, st));
    off += align_up(bytes, 16);
  }
  POETX_CUDA(cudaEventRecord(g_ring.ev[s], st));
  g_ring.pending[s] = true;
  return POETX_OK;
}

void perm_and_inverse(uint64_t seed, int d, std::vector<int32_t>& p, std::vector<int32_t>& inv) {
  p.resize(d);
  inv.resize(d);
  make_permutation(seed, d, p.data());
  for (int i = 0; i < d; ++i) inv[p[i]] = i;
}

// ------------------------------------------------------------------ fp32 path helpers

// out[:, blk] = in[:, blk] * B_blk^T (transpose) or * B_blk, per block, T rows,
// leading dimension ld; the ragged last block uses its top-left corner.
template <typename TI, typename TO>
poetx_status simt_blocks(cudaStream_t st, const SideLayout& S, const uint8_t* params, const TI* in,
                         TO* out, int64_t T, int64_t ld, bool transpose) {
  const float* B = reinterpret_cast<const float*>(params + S.off_B);
  const int b = S.g.b;
  const int64_t bb = static_cast<int64_t>(b) * b;
  const int full = S.g.nblk - (S.g.last < b ? 1 : 0);
  const int64_t sBk = transpose ? 1 : b, sBn = transpose ? b : 1;
  POETX_TRY(simt_gemm<TI, float, TO>(st, static_cast<int>(T), b, b, full, in, ld, 1, b, B, sBk, sBn,
                                     bb, out, ld, 1, b, 1.f, 0.f));
  if (S.g.last < b) {
    const int64_t o = static_cast<int64_t>(full) * b;
    POETX_TRY(simt_gemm<TI, float, TO>(st, static_cast<int>(T), S.g.last, S.g.last, 1, in + o, ld, 1,
                                       0, B + full * bb, sBk, sBn, 0, out + o, ld, 1, 0, 1.f, 0.f));
  }
  return POETX_OK;
}

// G[k] = A[:, blk]^T Bm[:, blk] (b x b per block, fp32), contraction over T.
poetx_status simt_gradblocks(cudaStream_t st, const SideLayout& S, const float* A, const float* Bm,
                             float* G, int64_t T, int64_t ld) {
  const int b = S.g.b;
  const int64_t bb = static_cast<int64_t>(b) * b;
  POETX_CUDA(cudaMemsetAsync(G, 0, static_cast<size_t>(S.g.nblk) * bb * 4, st));
  const int full = S.g.nblk - (S.g.last < b ? 1 : 0);
  POETX_TRY(simt_gemm<float, float, float>(st, b, b, static_cast<int>(T), full, A, 1, ld, b, Bm, ld, 1,
                                           b, G, b, 1, bb, 1.f, 0.f));
  if (S.g.last < b) {
    const int64_t o = static_cast<int64_t>(full) * b;
    POETX_TRY(simt_gemm<float, float, float>(st, S.g.last, S.g.last, static_cast<int>(T), 1, A + o, 1,
                                             ld, 0, Bm + o, ld, 1, 0, G + full * bb, b, 1, 0, 1.f,
                                             0.f));
  }
  return POETX_OK;
}

struct Ctx {
  const poetx_layer_desc& d;
  ParamsLayout L;
  WorkLayout W;
  const uint8_t* params;
  uint8_t* ws;
  cudaStream_t st;
  const int32_t* piR() const { return reinterpret_cast<const int32_t*>(params + L.off_piR); }
  const int32_t* piRinv() const { return reinterpret_cast<const int32_t*>(params + L.off_piRinv); }
  const int32_t* piP() const { return reinterpret_cast<const int32_t*>(params + L.off_piP); }
  const int32_t* piPinv() const { return reinterpret_cast<const int32_t*>(params + L.off_piPinv); }
  template <typename T> T* w(size_t off) const { return reinterpret_cast<T*>(ws + off); }
  template <typename T> const T* p(size_t off) const { return reinterpret_cast<const T*>(params + off); }
  // reduction partial slots written by the backward (bf16 path)
  mutable int slotsR = 0, slotsP = 0;
};

// An event recorded on one stream for later waits on others.
struct Ev {
  cudaEvent_t e = nullptr;
  ~Ev() {
    if (e) cudaEventDestroy(e);
  }
  poetx_status record(cudaStream_t st) {
    if (!e) POETX_CUDA(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
    POETX_CUDA(cudaEventRecord(e, st));
    return POETX_OK;
  }
  poetx_status wait_on(cudaStream_t st) const {
    POETX_CUDA(cudaStreamWaitEvent(st, e, 0));
    return POETX_OK;
  }
};

poetx_status fwd_fp32(const Ctx& c, const float* W0p, const float* X, int64_t T, float* Y, float* hs,
                      float* us) {
  const int m = c.d.m, n = c.d.n;
  float* u = us ? us : c.w<float>(c.W.off_n1);
  float* v = c.w<float>(c.W.off_n2);
  float* h = hs ? hs : c.w<float>(c.W.off_m1);
  float* z = c.w<float>(c.W.off_m2);
  POETX_TRY(gather_cols<float>(c.st, X, u, c.piP(), T, n));
  {
    ProfScope prof(POETX_KIND_SIMT, c.st);
    POETX_TRY(simt_blocks<float, float>(c.st, c.L.P, c.params, u, v, T, n, true));
    POETX_TRY(simt_gemm<float, float, float>(c.st, static_cast<int>(T), m, n, 1, v, n, 1, 0, W0p, 1, n,
                                             0, h, m, 1, 0, 1.f, 0.f));
    POETX_TRY(simt_blocks<float, float>(c.st, c.L.R, c.params, h, z, T, m, true));
  }
  POETX_TRY(gather_cols<float>(c.st, z, Y, c.piRinv(), T, m));
  return POETX_OK;
}

// Forward, bf16 ("POET-X ...", Methodologie §1: Y = R(W0(P x)) evaluated on
// the input):  X -> u = X[:, pi_P] (gather) -> v = u B_P^T (blocks) ->
// h = v W0'^T -> z = h B_R^T (blocks) -> Y[:, pi_R] = z (scatter).
poetx_status fwd_bf16(const Ctx& c, const __nv_bfloat16* W0p, const __nv_bfloat16* X, int64_t T,
                      __nv_bfloat16* Y, __nv_bfloat16* hs, __nv_bfloat16* us) {
  const int m = c.d.m, n = c.d.n;
  auto* u = us ? us : c.w<__nv_bfloat16>(c.W.off_n1);
  auto* v = c.w<__nv_bfloat16>(c.W.off_n2);
  auto* h = hs ? hs : c.w<__nv_bfloat16>(c.W.off_m1);
  auto* z = c.w<__nv_bfloat16>(c.W.off_m2);
  const SideLayout &R = c.L.R, &P = c.L.P;
  if (gbd_ok(P)) {  // u and v from one kernel (u is kept for the backward)
    POETX_TRY(tc_gather_bd<false>(c.st, P, X, c.piP(), c.p<__nv_bfloat16>(P.off_Bsb), v, u, nullptr,
                                  nullptr, T, nullptr));
  } else {
    POETX_TRY(gather_cols<__nv_bfloat16>(c.st, X, u, c.piP(), T, n));
    POETX_TRY(tc_blockdiag(c.st, u, c.p<__nv_bfloat16>(P.off_Bsb), v, T, n, P.sb, P.nsb));
  }
  if (r_epilogue(R, T, m)) {
    POETX_TRY(tc_dense_nt_r(c.st, v, W0p, c.p<__nv_bfloat16>(R.off_Bsb), hs, z, T, m, n, R.nsb));
  } else if (pair_r_epilogue(R, T, m)) {
    POETX_TRY(tc_dense_nt_pair_r(c.st, v, W0p, c.p<__nv_bfloat16>(R.off_Bsb), hs, z, T, m, n, R.nsb));
  } else {
    POETX_TRY(tc_dense_nt(c.st, v, W0p, h, T, m, n));
    POETX_TRY(tc_blockdiag(c.st, h, c.p<__nv_bfloat16>(R.off_Bsb), z, T, m, R.sb, R.nsb));
  }
  return gather_cols<__nv_bfloat16>(c.st, z, Y, c.piRinv(), T, m);
}

bool fused_cayley_bwd_ok(const poetx_layer_desc& d, int b) {
  return d.dtype == POETX_DTYPE_BF16 && d.mode == POETX_MODE_CAYLEY &&
         (b == 32 || b == 64 || b == 128 || b == 256 || b == 512);
}

// 128-wide blocks of one or two sides on four-CTA clusters (side b may be empty).
poetx_status launch_cayley_bwd_clusters(cudaStream_t st, const CbwdSide& a, const CbwdSide& b,
                                        int accumulate) {
  static cudaError_t attr_err = cudaFuncSetAttribute(
      cayley_bwd_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kCbwdSmem);
  if (attr_err != cudaSuccess) return POETX_ERR_CUDA;
  const int blocks = a.s.nblk + b.s.nblk;
  if (blocks == 0) return POETX_OK;
  return launch_dep(cayley_bwd_cluster_kernel, blocks * 4, 256, kCbwdSmem, st, 0, a, b, accumulate);
}

// 32- or 64-wide blocks of one or two sides (side b may be empty), one CTA
// per block (see cayley_bwd_kernel).
poetx_status launch_cayley_bwd_small(cudaStream_t st, int P, const CbwdSide& a, const CbwdSide& b,
                                     int accumulate) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(cayley_bwd_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(cbwd_smem<64>()));
  });
  if (attr_err != cudaSuccess) return POETX_ERR_CUDA;
  const int blocks = a.s.nblk + b.s.nblk;
  if (blocks == 0) return POETX_OK;
  if (P == 64)
    return launch_dep(cayley_bwd_kernel<64>, blocks, kCbwdThreads, cbwd_smem<64>(), st, 0, a, b, accumulate);
  if (P == 32)
    return launch_dep(cayley_bwd_kernel<32>, blocks, kCbwdThreads, cbwd_smem<32>(), st, 0, a, b, accumulate);
  return POETX_ERR_UNSUPPORTED;
}

// Fused reduction + Cayley backward + packing for one side (see cayley_bwd_kernel).
poetx_status fused_cayley_bwd(cudaStream_t st, const SideLayout& S, const uint8_t* params,
                              const float* partial, int splits, float* t1, float* t2, float* dGen,
                              int accumulate) {
  ProfScope prof(POETX_KIND_GENBWD, st);
  const int b = S.g.b;
  const float* M = reinterpret_cast<const float*>(params + S.off_M);
  const int64_t stride = static_cast<int64_t>(S.nsb) * S.sb * S.sb;
  if (b >= 256) {
    // G = sum of the split partials (super-block k is block k), then on the
    // tensor cores with fp32-grade products T = M^T G and GQ = 2 T M^T,
    // then the pack
    const int nb = S.g.nblk;
    const int64_t bb = static_cast<int64_t>(b) * b;
    POETX_TRY(launch_dep(gradred_reduce_kernel, grid_for(nb * bb), 256, 0, st, 0, partial, stride, splits,
                         S.g, S.sb, t2));
    const F32Operand mt{M, 1, b, bb};   // A(i, q) = M[q][i]
    const F32Operand g{t2, 1, b, bb};   // B(j, q) = G[q][j]
    POETX_TRY(tc_f32_gemm(st, b, b, b, nb, mt, g, t1, b, bb, 1.f, 0.f));
    const F32Operand t{t1, b, 1, bb};   // A(i, q) = T[i][q]
    const F32Operand m{M, b, 1, bb};    // B(j, q) = M[j][q]
    POETX_TRY(tc_f32_gemm(st, b, b, b, nb, t, m, t2, b, bb, 2.f, 0.f));
    return launch_dep(pack_grad_kernel, dim3(nb, (b + 7) / 8), 256, 0, st, 0, t2, S.g, dGen, accumulate);
  }
  CbwdSide a{partial, stride, splits, S.g, M, dGen}, none{};
  none.s.nblk = 0;
  if (b == 128) return launch_cayley_bwd_clusters(st, a, none, accumulate);  // four CTAs per block
  return launch_cayley_bwd_small(st, b, a, none, accumulate);
}

// bf16 Neumann layers with 128-wide blocks: the chain rule of the
// polynomial for every block of one side, or of both sides when `second` is
// given, in one tensor-core launch.  Measured on d2048 (k = 3): at b = 128
// it cuts the generator backward from 2.05 to 1.36 ms per step; at b = 256
// and 512 its 2k dependent products per CTA are slower than the batched
// products over 128 x 128 tiles (3.2 vs 2.5-2.8 ms at b = 256), so those keep
// the batched chain rule.
bool fused_neumann_bwd_ok(const poetx_layer_desc& d, int b) { return fused_neumann_ok(d, b) && b == 128; }

template <int BS>
poetx_status launch_neumann_bwd_kernel(cudaStream_t st, const NeumannBwdSide& a,
                                       const NeumannBwdSide& b2, int blocks, int k, int accumulate) {
  using Cfg = NeuCfg<BS>;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(tc_neumann_bwd_kernel<BS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         Cfg::SMEM);
  });
  return launch_dep(tc_neumann_bwd_kernel<BS>, Cfg::C * blocks, Cfg::THREADS, Cfg::SMEM, st, 0, a, b2, k,
                    accumulate, g_timeout_ns);
}

poetx_status launch_neumann_bwd(cudaStream_t st, const poetx_layer_desc& d, const NeumannBwdSide& a,
                                const NeumannBwdSide* second, int accumulate) {
  ProfScope prof(POETX_KIND_GENBWD, st);
  const int blocks = a.s.nblk + (second ? second->s.nblk : 0);
  const NeumannBwdSide& b2 = second ? *second : a;
  if (a.s.b != 128) return POETX_ERR_UNSUPPORTED;
  return launch_neumann_bwd_kernel<128>(st, a, b2, blocks, d.neumann_k, accumulate);
}

poetx_status bwd_common_tail(const Ctx& c, float* dGenR, float* dGenP, int accumulate) {
  float* GR = c.w<float>(c.W.off_GR);
  float* GP = c.w<float>(c.W.off_GP);
  float* t1 = c.w<float>(c.W.off_t1);
  float* t2 = c.w<float>(c.W.off_t2);
  float* nsc = c.w<float>(c.W.off_nsc);
  const bool doR = dGenR && poetx_gen_length(c.d.m, c.d.b_R) > 0;
  const bool doP = dGenP && poetx_gen_length(c.d.n, c.d.b_P) > 0;
  if (doR && doP && c.d.b_R == c.d.b_P && c.d.b_R <= 128 && fused_cayley_bwd_ok(c.d, c.d.b_R)) {
    // both sides' blocks in one launch
    ProfScope prof(POETX_KIND_GENBWD, c.st);
    const CbwdSide r{c.w<float>(c.W.off_partR), static_cast<int64_t>(c.L.R.nsb) * c.L.R.sb * c.L.R.sb,
                     c.slotsR, c.L.R.g, c.p<float>(c.L.R.off_M), dGenR};
    const CbwdSide p{c.w<float>(c.W.off_partP), static_cast<int64_t>(c.L.P.nsb) * c.L.P.sb * c.L.P.sb,
                     c.slotsP, c.L.P.g, c.p<float>(c.L.P.off_M), dGenP};
    if (c.d.b_R == 128) return launch_cayley_bwd_clusters(c.st, r, p, accumulate);
    return launch_cayley_bwd_small(c.st, c.d.b_R, r, p, accumulate);
  }
  if (fused_neumann_bwd_ok(c.d, c.d.b_R) || fused_neumann_bwd_ok(c.d, c.d.b_P)) {
    // five scratch matrices per side: side R at nsc, side P after them
    const int64_t gstride = static_cast<int64_t>(std::max(c.L.R.g.nblk * c.L.R.bb(),
                                                          c.L.P.g.nblk * c.L.P.bb()));
    const float* Qr = c.p<float>(c.L.R.off_Q);
    const float* Qp = c.p<float>(c.L.P.off_Q);
    const NeumannBwdSide r{GR, Qr, nsc, gstride, c.L.R.g, dGenR};
    const NeumannBwdSide p{GP, Qp, nsc + 5 * gstride, gstride, c.L.P.g, dGenP};
    const bool fr = doR && fused_neumann_bwd_ok(c.d, c.d.b_R);
    const bool fp = doP && fused_neumann_bwd_ok(c.d, c.d.b_P);
    if (fr && fp && c.d.b_R == c.d.b_P) return launch_neumann_bwd(c.st, c.d, r, &p, accumulate);
    if (fr) POETX_TRY(launch_neumann_bwd(c.st, c.d, r, nullptr, accumulate));
    else if (doR) POETX_TRY(generator_backward(c.st, c.d, c.L.R, c.params, GR, t1, t2, nsc, dGenR, accumulate));
    if (fp) POETX_TRY(launch_neumann_bwd(c.st, c.d, p, nullptr, accumulate));
    else if (doP) POETX_TRY(generator_backward(c.st, c.d, c.L.P, c.params, GP, t1, t2, nsc, dGenP, accumulate));
    return POETX_OK;
  }
  if (doR) {
    if (fused_cayley_bwd_ok(c.d, c.d.b_R))
      POETX_TRY(fused_cayley_bwd(c.st, c.L.R, c.params, c.w<float>(c.W.off_partR), c.slotsR, t1, t2,
                                 dGenR, accumulate));
    else
      POETX_TRY(generator_backward(c.st, c.d, c.L.R, c.params, GR, t1, t2, nsc, dGenR, accumulate));
  }
  if (doP) {
    if (fused_cayley_bwd_ok(c.d, c.d.b_P))
      POETX_TRY(fused_cayley_bwd(c.st, c.L.P, c.params, c.w<float>(c.W.off_partP), c.slotsP, t1, t2,
                                 dGenP, accumulate));
    else
      POETX_TRY(generator_backward(c.st, c.d, c.L.P, c.params, GP, t1, t2, nsc, dGenP, accumulate));
  }
  return POETX_OK;
}

poetx_status bwd_fp32(const Ctx& c, const float* W0p, const float* X, const float* dY,
                      const float* hs, const float* us, int64_t T, float* dX) {
  const int m = c.d.m, n = c.d.n;
  float* ubuf = c.w<float>(c.W.off_n1);
  float* v = c.w<float>(c.W.off_n2);
  float* hbuf = c.w<float>(c.W.off_m1);
  float* dz = c.w<float>(c.W.off_m2);
  float* dh = c.w<float>(c.W.off_m3);
  if (!us) POETX_TRY(gather_cols<float>(c.st, X, ubuf, c.piP(), T, n));
  const float* u = us ? us : ubuf;
  const float* h = hs;
  {
    ProfScope prof(POETX_KIND_SIMT, c.st);
    if (!hs) {
      POETX_TRY(simt_blocks<float, float>(c.st, c.L.P, c.params, u, v, T, n, true));
      POETX_TRY(simt_gemm<float, float, float>(c.st, static_cast<int>(T), m, n, 1, v, n, 1, 0, W0p, 1,
                                               n, 0, hbuf, m, 1, 0, 1.f, 0.f));
      h = hbuf;
    }
  }
  POETX_TRY(gather_cols<float>(c.st, dY, dz, c.piR(), T, m));
  float* dv = v;
  float* du = ubuf;  // u is dead once the dv^T u reduction has read it (a saved u is not written)
  {
    ProfScope prof(POETX_KIND_SIMT, c.st);
    POETX_TRY(simt_gradblocks(c.st, c.L.R, dz, h, c.w<float>(c.W.off_GR), T, m));
    POETX_TRY(simt_blocks<float, float>(c.st, c.L.R, c.params, dz, dh, T, m, false));
    POETX_TRY(simt_gemm<float, float, float>(c.st, static_cast<int>(T), n, m, 1, dh, m, 1, 0, W0p, n, 1,
                                             0, dv, n, 1, 0, 1.f, 0.f));
    POETX_TRY(simt_gradblocks(c.st, c.L.P, dv, u, c.w<float>(c.W.off_GP), T, n));
    POETX_TRY(simt_blocks<float, float>(c.st, c.L.P, c.params, dv, du, T, n, false));
  }
  if (dX) POETX_TRY(gather_cols<float>(c.st, du, dX, c.piPinv(), T, n));
  return POETX_OK;
}

// Backward, bf16 (the chain rule of the forward's steps):
//   u    = X[:, pi_P] when not kept; in recompute mode also v = u B_P^T and
//          h = v W0'^T (gradient checkpointing, Methodologie §5)
//   dz   = dY[:, pi_R];  dh = dz B_R;  partials of G_R = dz^T h
//   dv   = dh W0'
//   du   = dv B_P;  partials of G_P = dv^T u;  dX[:, pi_P] = du
// The per-block reductions of the partials follow in bwd_common_tail.
poetx_status bwd_bf16(const Ctx& c, const __nv_bfloat16* W0p, const __nv_bfloat16* X,
                      const __nv_bfloat16* dY, const __nv_bfloat16* hs, const __nv_bfloat16* us,
                      int64_t T, __nv_bfloat16* dX) {
  const int m = c.d.m, n = c.d.n;
  const SideLayout &R = c.L.R, &P = c.L.P;
  auto* ubuf = c.w<__nv_bfloat16>(c.W.off_n1);
  const __nv_bfloat16* u = us ? us : ubuf;
  auto* v = c.w<__nv_bfloat16>(c.W.off_n2);
  auto* hbuf = c.w<__nv_bfloat16>(c.W.off_m1);
  auto* dz = c.w<__nv_bfloat16>(c.W.off_m2);
  auto* dh = c.w<__nv_bfloat16>(c.W.off_m3);
  float* partR = c.w<float>(c.W.off_partR);
  float* partP = c.w<float>(c.W.off_partP);
  const auto* BsbP = c.p<__nv_bfloat16>(P.off_Bsb);
  const auto* BsbRT = c.p<__nv_bfloat16>(R.off_BsbT);
  const auto* BsbPT = c.p<__nv_bfloat16>(P.off_BsbT);
  const bool recompute = (hs == nullptr);
  const __nv_bfloat16* h = recompute ? hbuf : hs;
  auto* dv = v;     // v is dead once h is formed
  auto* du = ubuf;  // u is dead once the dv^T u partials are formed (a saved u is not written)
  const int64_t strideR = static_cast<int64_t>(R.nsb) * R.sb * R.sb;
  const int64_t strideP = static_cast<int64_t>(P.nsb) * P.sb * P.sb;
  c.slotsR = c.slotsP = 0;

  // u (when not kept), and in recompute mode v and h
  if (!us && recompute && gbd_ok(P)) {  // u and v from one kernel
    POETX_TRY(tc_gather_bd<false>(c.st, P, X, c.piP(), BsbP, v, ubuf, nullptr, nullptr, T, nullptr));
  } else {
    if (!us) POETX_TRY(gather_cols<__nv_bfloat16>(c.st, X, ubuf, c.piP(), T, n));
    if (recompute) POETX_TRY(tc_blockdiag(c.st, u, BsbP, v, T, n, P.sb, P.nsb));
  }
  if (recompute) POETX_TRY(tc_dense_nt(c.st, v, W0p, hbuf, T, m, n));

  // R side: dz, dh and the dz^T h partials
  if (gbd_ok(R)) {  // dz = dY[:, pi_R] gathered inside the fused transform + reduction
    POETX_TRY(tc_gather_bd<true>(c.st, R, dY, c.piR(), BsbRT, dh, nullptr, h, partR, T, &c.slotsR));
  } else if (bdgr_ok(R)) {  // dh = dz B_R and the dz^T h partials from one read of dz
    POETX_TRY(gather_cols<__nv_bfloat16>(c.st, dY, dz, c.piR(), T, m));
    POETX_TRY(tc_bdgr(c.st, R, dz, BsbRT, dh, h, partR, T, &c.slotsR));
  } else if (bdgr256_ok(R)) {
    POETX_TRY(gather_cols<__nv_bfloat16>(c.st, dY, dz, c.piR(), T, m));
    POETX_TRY(tc_bdgr256(c.st, R, dz, BsbRT, dh, h, partR, T, &c.slotsR));
  } else {
    POETX_TRY(gather_cols<__nv_bfloat16>(c.st, dY, dz, c.piR(), T, m));
    POETX_TRY(tc_blockdiag(c.st, dz, BsbRT, dh, T, m, R.sb, R.nsb));
    POETX_TRY(tc_gradred(c.st, R, dz, h, partR, T, &c.slotsR));
  }

  // P side: dv, du, the dv^T u partials and dX
  if (dX && p_epilogue(P, T, n)) {  // du and the partials in the dgrad epilogue
    POETX_TRY(tc_dense_nn_p(c.st, P, dh, W0p, BsbPT, u, du, partP, T, n, m, &c.slotsP));
    POETX_TRY(gather_cols<__nv_bfloat16>(c.st, du, dX, c.piPinv(), T, n));
  } else if (dX && bdgr_ok(P)) {  // du = dv B_P (over u) and the dv^T u partials from one read of dv
    POETX_TRY(tc_dense_nn(c.st, dh, W0p, dv, T, n, m));
    POETX_TRY(tc_bdgr(c.st, P, dv, BsbPT, du, u, partP, T, &c.slotsP));
    POETX_TRY(gather_cols<__nv_bfloat16>(c.st, du, dX, c.piPinv(), T, n));
  } else if (dX && bdgr256_ok(P)) {
    POETX_TRY(tc_dense_nn(c.st, dh, W0p, dv, T, n, m));
    POETX_TRY(tc_bdgr256(c.st, P, dv, BsbPT, du, u, partP, T, &c.slotsP));
    POETX_TRY(gather_cols<__nv_bfloat16>(c.st, du, dX, c.piPinv(), T, n));
  } else {
    POETX_TRY(tc_dense_nn(c.st, dh, W0p, dv, T, n, m));
    POETX_TRY(tc_gradred(c.st, P, dv, u, partP, T, &c.slotsP));
    if (dX) {
      POETX_TRY(tc_blockdiag(c.st, dv, BsbPT, du, T, n, P.sb, P.nsb));
      POETX_TRY(gather_cols<__nv_bfloat16>(c.st, du, dX, c.piPinv(), T, n));
    }
  }

  ProfScope prof(POETX_KIND_GENBWD, c.st);
  // exact Cayley blocks of b <= 128: the generator backward runs fused per block
  // in bwd_common_tail; otherwise reduce the partials into G here.
  if (!fused_cayley_bwd_ok(c.d, R.g.b)) {
    POETX_TRY(launch_dep(gradred_reduce_kernel, grid_for(static_cast<int64_t>(R.g.nblk) * R.bb()), 256, 0,
                         c.st, 0, partR, strideR, c.slotsR, R.g, R.sb, c.w<float>(c.W.off_GR)));
  }
  if (!fused_cayley_bwd_ok(c.d, P.g.b)) {
    POETX_TRY(launch_dep(gradred_reduce_kernel, grid_for(static_cast<int64_t>(P.g.nblk) * P.bb()), 256, 0,
                         c.st, 0, partP, strideP, c.slotsP, P.g, P.sb, c.w<float>(c.W.off_GP)));
  }
  return POETX_OK;
}

poetx_status check_tensor(const void* p) {
  if (!p) return POETX_ERR_INVALID_ARG;
  if (!aligned(p, 16)) return POETX_ERR_MISALIGNED;
  return POETX_OK;
}

// POET-XQ: an int8 weight buffer (codes, then row scales) to bf16 m x n,
// with `lo` also the bf16 remainder (out + lo = scale * code to 2^-17).
poetx_status dequant_weight(cudaStream_t st, const poetx_layer_desc& d, const void* W0p,
                            __nv_bfloat16* out, __nv_bfloat16* lo = nullptr) {
  ProfScope prof(POETX_KIND_DEQUANT, st);
  const auto* codes = reinterpret_cast<const int8_t*>(W0p);
  const auto* scales =
      reinterpret_cast<const float*>(reinterpret_cast<const uint8_t*>(W0p) + weight_codes_bytes(d));
  dequant_int8_kernel<<<grid_for(static_cast<int64_t>(d.m) * d.n / 8), 256, 0, st>>>(codes, scales, out,
                                                                                     lo, d.m, d.n);
  POETX_LAUNCHED();
  return POETX_OK;
}

// POET-XQ: quantizes row i from S[row_map[i]][col_map[j]], S = hi (+ lo), into
// the int8 weight buffer (quantize_rows_kernel).
poetx_status quantize_weight(cudaStream_t st, const poetx_layer_desc& d, const __nv_bfloat16* hi,
                             const __nv_bfloat16* lo, const int32_t* row_map, const int32_t* col_map,
                             void* W0p) {
  const size_t smem = static_cast<size_t>(d.n) * 4;
  if (smem > 200 * 1024) return POETX_ERR_UNSUPPORTED;
  static cudaError_t attr_err =
      cudaFuncSetAttribute(quantize_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
  if (attr_err != cudaSuccess) return POETX_ERR_CUDA;
  auto* codes = reinterpret_cast<int8_t*>(W0p);
  auto* scales = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(W0p) + weight_codes_bytes(d));
  quantize_rows_kernel<<<d.m, 256, smem, st>>>(hi, lo, row_map, col_map, d.n, codes, scales);
  POETX_LAUNCHED();
  return POETX_OK;
}

// Merge scratch.  fp32 layers: T1 = W0' B_P and K = B_R T1 (fp32, m x n).
// bf16 layers (tensor-core passes): W1 = (W0' B_P)^T as a bf16 hi/lo pair
// (n x m each), K = B_R W0' B_P in bf16 (m x n), and the hi/lo super-block
// arrays of B_P^T - I and B_R - I.  Both: the re-basing index maps rho.
struct MergeLayout {
  size_t off_T1, off_K;              // fp32
  size_t off_W1hi, off_W1lo, off_Kb;  // bf16
  size_t off_Wdq, off_Wdqlo, off_Klo;  // int8 weights: dequantized input (hi, lo), low half of K
  size_t off_DPhi, off_DPlo, off_DRhi, off_DRlo;
  size_t off_rhoR, off_rhoP;
  size_t total;
};

MergeLayout merge_layout(const poetx_layer_desc& d, const ParamsLayout& L) {
  MergeLayout M{};
  const size_t mn = static_cast<size_t>(d.m) * d.n;
  size_t off = 0;
  if (d.dtype == POETX_DTYPE_FP32) {
    M.off_T1 = off; off = align_up(off + mn * 4);
    M.off_K = off;  off = align_up(off + mn * 4);
  } else {
    const size_t dp = static_cast<size_t>(L.P.nsb) * L.P.sb * L.P.sb * 2;
    const size_t dr = static_cast<size_t>(L.R.nsb) * L.R.sb * L.R.sb * 2;
    M.off_W1hi = off; off = align_up(off + mn * 2);
    M.off_W1lo = off; off = align_up(off + mn * 2);
    M.off_Kb = off;   off = align_up(off + mn * 2);
    M.off_DPhi = off; off = align_up(off + dp);
    M.off_DPlo = off; off = align_up(off + dp);
    M.off_DRhi = off; off = align_up(off + dr);
    M.off_DRlo = off; off = align_up(off + dr);
    if (weight_int8(d)) {
      M.off_Wdq = off; off = align_up(off + mn * 2);
      M.off_Wdqlo = off; off = align_up(off + mn * 2);
      M.off_Klo = off; off = align_up(off + mn * 2);
    }
  }
  M.off_rhoR = off; off = align_up(off + static_cast<size_t>(d.m) * 4);
  M.off_rhoP = off; off = align_up(off + static_cast<size_t>(d.n) * 4);
  M.total = off;
  return M;
}

}  // namespace

// ====================================================================== C ABI

extern "C" {

const char* poetx_status_string(int32_t s) {
  switch (s) {
    case POETX_OK: return "POETX_OK";
    case POETX_ERR_INVALID_ARG: return "POETX_ERR_INVALID_ARG";
    case POETX_ERR_UNSUPPORTED: return "POETX_ERR_UNSUPPORTED";
    case POETX_ERR_MISALIGNED: return "POETX_ERR_MISALIGNED";
    case POETX_ERR_CUDA: return "POETX_ERR_CUDA";
    case POETX_ERR_TIMEOUT: return "POETX_ERR_TIMEOUT";
    default: return "POETX_ERR_UNKNOWN";
  }
}

int32_t poetx_version(void) { return 1000; }

poetx_status poetx_perm_generate(uint64_t seed, int32_t d, int32_t* host_out) {
  if (d < 1 || !host_out) return POETX_ERR_INVALID_ARG;
  make_permutation(seed, d, host_out);
  return POETX_OK;
}

int64_t poetx_gen_length(int32_t d, int32_t b) {
  if (d < 1 || b < 1 || b > d) return -1;
  const SideGeom g = side_geom(d, b);
  return static_cast<int64_t>(g.nblk - 1) * b * (b - 1) / 2 +
         static_cast<int64_t>(g.last) * (g.last - 1) / 2;
}

size_t poetx_params_size(const poetx_layer_desc* d) {
  if (check_desc(d) != POETX_OK) return 0;
  return params_layout(*d).total;
}

poetx_status poetx_blocks_build(const poetx_layer_desc* desc, const float* genR, const float* genP,
                                void* params, void* stream) {
  POETX_TRY(check_desc(desc));
  if (!params) return POETX_ERR_INVALID_ARG;
  if ((poetx_gen_length(desc->m, desc->b_R) > 0 && !genR) ||
      (poetx_gen_length(desc->n, desc->b_P) > 0 && !genP))
    return POETX_ERR_INVALID_ARG;
  if (!aligned(params, kAlign)) return POETX_ERR_MISALIGNED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const ParamsLayout L = params_layout(*desc);
  uint8_t* pb = reinterpret_cast<uint8_t*>(params);
  if (desc->b_R == desc->b_P && fused_cayley_ok(*desc, desc->b_R)) {
    ProfScope prof(POETX_KIND_BUILD, st);
    const CayleySide r = cayley_side(*desc, L.R, genR, pb), p = cayley_side(*desc, L.P, genP, pb);
    return launch_cayley_blocks(st, *desc, r, &p);
  }
  if (desc->b_R == desc->b_P && fused_neumann_ok(*desc, desc->b_R)) {
    ProfScope prof(POETX_KIND_BUILD, st);
    const NeumannSide r = neumann_side(L.R, genR, pb), p = neumann_side(L.P, genP, pb);
    return launch_neumann_blocks(st, *desc, r, &p);
  }
  POETX_TRY(build_side(st, *desc, L.R, genR, pb));
  POETX_TRY(build_side(st, *desc, L.P, genP, pb));
  return POETX_OK;
}

poetx_status poetx_params_build(const poetx_layer_desc* desc, const float* genR, const float* genP,
                                void* params, void* stream) {
  POETX_TRY(check_desc(desc));
  if (!params) return POETX_ERR_INVALID_ARG;
  if ((poetx_gen_length(desc->m, desc->b_R) > 0 && !genR) ||
      (poetx_gen_length(desc->n, desc->b_P) > 0 && !genP))
    return POETX_ERR_INVALID_ARG;
  if (!aligned(params, kAlign)) return POETX_ERR_MISALIGNED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const ParamsLayout L = params_layout(*desc);
  uint8_t* pb = reinterpret_cast<uint8_t*>(params);
  std::vector<int32_t> piR, piRinv, piP, piPinv;
  perm_and_inverse(desc->seed_R, desc->m, piR, piRinv);
  perm_and_inverse(desc->seed_P, desc->n, piP, piPinv);
  POETX_TRY(ring_upload(st,
                        {{piR.data(), piR.size()}, {piRinv.data(), piRinv.size()},
                         {piP.data(), piP.size()}, {piPinv.data(), piPinv.size()}},
                        {pb + L.off_piR, pb + L.off_piRinv, pb + L.off_piP, pb + L.off_piPinv}));
  return poetx_blocks_build(desc, genR, genP, params, stream);
}

poetx_status poetx_weight_premerge(const poetx_layer_desc* desc, const void* params, const void* W0,
                                   void* W0p, void* stream) {
  POETX_TRY(check_desc(desc));
  if (!params || !W0 || !W0p || W0 == W0p) return POETX_ERR_INVALID_ARG;
  if (!aligned(params, kAlign)) return POETX_ERR_MISALIGNED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const ParamsLayout L = params_layout(*desc);
  const uint8_t* pb = reinterpret_cast<const uint8_t*>(params);
  const int32_t* piR = reinterpret_cast<const int32_t*>(pb + L.off_piR);
  const int32_t* piP = reinterpret_cast<const int32_t*>(pb + L.off_piP);
  const int grid = std::min(desc->m, device_sm_count() * 8);
  ProfScope prof(POETX_KIND_MERGE, st);
  if (weight_int8(*desc))
    return quantize_weight(st, *desc, reinterpret_cast<const __nv_bfloat16*>(W0), nullptr, piR, piP, W0p);
  if (desc->dtype == POETX_DTYPE_BF16)
    gather2d_kernel<__nv_bfloat16, __nv_bfloat16><<<grid, 256, 0, st>>>(
        reinterpret_cast<const __nv_bfloat16*>(W0), reinterpret_cast<__nv_bfloat16*>(W0p), piR, piP,
        desc->m, desc->n);
  else
    gather2d_kernel<float, float><<<grid, 256, 0, st>>>(reinterpret_cast<const float*>(W0),
                                                        reinterpret_cast<float*>(W0p), piR, piP,
                                                        desc->m, desc->n);
  POETX_LAUNCHED();
  return POETX_OK;
}

size_t poetx_weight_size(const poetx_layer_desc* desc) {
  if (check_desc(desc) != POETX_OK) return 0;
  return weight_bytes(*desc);
}

size_t poetx_workspace_size(const poetx_layer_desc* desc, int64_t T) {
  if (check_desc(desc) != POETX_OK || T < 0) return 0;
  return work_layout(*desc, params_layout(*desc), T, device_sm_count()).total;
}

poetx_status poetx_linear_fwd(const poetx_layer_desc* desc, const void* params, const void* W0p,
                              const void* X, int64_t T, void* Y, void* saved_h, void* saved_u,
                              void* workspace, void* stream) {
  POETX_TRY(check_desc(desc));
  if (T < 0) return POETX_ERR_INVALID_ARG;
  if (T == 0) return POETX_OK;
  if (!params || !workspace) return POETX_ERR_INVALID_ARG;
  POETX_TRY(check_tensor(W0p));
  POETX_TRY(check_tensor(X));
  POETX_TRY(check_tensor(Y));
  if (saved_h) POETX_TRY(check_tensor(saved_h));
  if (saved_u) POETX_TRY(check_tensor(saved_u));
  if (saved_u && (saved_u == X || saved_u == Y || saved_u == saved_h)) return POETX_ERR_INVALID_ARG;
  if (!aligned(params, kAlign) || !aligned(workspace, kAlign)) return POETX_ERR_MISALIGNED;
  if (T > (int64_t(1) << 31) - 256) return POETX_ERR_UNSUPPORTED;
  const ParamsLayout L = params_layout(*desc);
  Ctx c{*desc, L, work_layout(*desc, L, T, device_sm_count()),
        reinterpret_cast<const uint8_t*>(params), reinterpret_cast<uint8_t*>(workspace),
        reinterpret_cast<cudaStream_t>(stream)};
  if (weight_int8(*desc)) {
    auto* wdq = c.w<__nv_bfloat16>(c.W.off_wdq);
    POETX_TRY(dequant_weight(c.st, *desc, W0p, wdq));
    W0p = wdq;
  }
  if (desc->dtype == POETX_DTYPE_FP32)
    return fwd_fp32(c, reinterpret_cast<const float*>(W0p), reinterpret_cast<const float*>(X), T,
                    reinterpret_cast<float*>(Y), reinterpret_cast<float*>(saved_h),
                    reinterpret_cast<float*>(saved_u));
  return fwd_bf16(c, reinterpret_cast<const __nv_bfloat16*>(W0p),
                  reinterpret_cast<const __nv_bfloat16*>(X), T, reinterpret_cast<__nv_bfloat16*>(Y),
                  reinterpret_cast<__nv_bfloat16*>(saved_h), reinterpret_cast<__nv_bfloat16*>(saved_u));
}

poetx_status poetx_linear_bwd(const poetx_layer_desc* desc, const void* params, const void* W0p,
                              const void* X, const void* dY, const void* saved_h,
                              const void* saved_u, int64_t T, void* dX, float* dGenR, float* dGenP,
                              int32_t accumulate, void* workspace, void* stream) {
  POETX_TRY(check_desc(desc));
  if (T < 0) return POETX_ERR_INVALID_ARG;
  if (!params || !workspace) return POETX_ERR_INVALID_ARG;
  if ((poetx_gen_length(desc->m, desc->b_R) > 0 && !dGenR) ||
      (poetx_gen_length(desc->n, desc->b_P) > 0 && !dGenP))
    return POETX_ERR_INVALID_ARG;
  if (T == 0) {
    // No tokens: the generator gradients are zero (with accumulate: unchanged).
    cudaStream_t st0 = reinterpret_cast<cudaStream_t>(stream);
    if (!accumulate) {
      const int64_t lr = poetx_gen_length(desc->m, desc->b_R);
      const int64_t lp = poetx_gen_length(desc->n, desc->b_P);
      if (lr > 0) POETX_CUDA(cudaMemsetAsync(dGenR, 0, lr * 4, st0));
      if (lp > 0) POETX_CUDA(cudaMemsetAsync(dGenP, 0, lp * 4, st0));
    }
    return POETX_OK;
  }
  POETX_TRY(check_tensor(W0p));
  if (saved_u) POETX_TRY(check_tensor(saved_u));
  else POETX_TRY(check_tensor(X));  // X is read only to form u
  POETX_TRY(check_tensor(dY));
  if (saved_h) POETX_TRY(check_tensor(saved_h));
  if (dX) POETX_TRY(check_tensor(dX));
  if (!aligned(params, kAlign) || !aligned(workspace, kAlign)) return POETX_ERR_MISALIGNED;
  if (T > (int64_t(1) << 31) - 256) return POETX_ERR_UNSUPPORTED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const ParamsLayout L = params_layout(*desc);
  Ctx c{*desc, L, work_layout(*desc, L, T, device_sm_count()),
        reinterpret_cast<const uint8_t*>(params), reinterpret_cast<uint8_t*>(workspace), st};
  if (weight_int8(*desc)) {
    auto* wdq = c.w<__nv_bfloat16>(c.W.off_wdq);
    POETX_TRY(dequant_weight(c.st, *desc, W0p, wdq));
    W0p = wdq;
  }
  if (desc->dtype == POETX_DTYPE_FP32)
    POETX_TRY(bwd_fp32(c, reinterpret_cast<const float*>(W0p), reinterpret_cast<const float*>(X),
                       reinterpret_cast<const float*>(dY), reinterpret_cast<const float*>(saved_h),
                       reinterpret_cast<const float*>(saved_u), T, reinterpret_cast<float*>(dX)));
  else
    POETX_TRY(bwd_bf16(c, reinterpret_cast<const __nv_bfloat16*>(W0p),
                       reinterpret_cast<const __nv_bfloat16*>(X),
                       reinterpret_cast<const __nv_bfloat16*>(dY),
                       reinterpret_cast<const __nv_bfloat16*>(saved_h),
                       reinterpret_cast<const __nv_bfloat16*>(saved_u), T,
                       reinterpret_cast<__nv_bfloat16*>(dX)));
  return bwd_common_tail(c, dGenR, dGenP, accumulate);
}

size_t poetx_merge_workspace_size(const poetx_layer_desc* desc) {
  if (check_desc(desc) != POETX_OK) return 0;
  return merge_layout(*desc, params_layout(*desc)).total;
}

poetx_status poetx_merge(const poetx_layer_desc* desc, const void* params, void* W0p,
                         uint64_t new_seed_R, uint64_t new_seed_P, void* workspace, void* stream) {
  POETX_TRY(check_desc(desc));
  if (!params || !workspace) return POETX_ERR_INVALID_ARG;
  POETX_TRY(check_tensor(W0p));
  if (!aligned(params, kAlign) || !aligned(workspace, kAlign)) return POETX_ERR_MISALIGNED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int m = desc->m, n = desc->n;
  const ParamsLayout L = params_layout(*desc);
  const MergeLayout ML = merge_layout(*desc, L);
  const uint8_t* pb = reinterpret_cast<const uint8_t*>(params);
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  int32_t* rhoR = reinterpret_cast<int32_t*>(ws + ML.off_rhoR);
  int32_t* rhoP = reinterpret_cast<int32_t*>(ws + ML.off_rhoP);
  ProfScope prof(POETX_KIND_MERGE, st);
  const bool bf16 = desc->dtype == POETX_DTYPE_BF16;
  float* T1 = reinterpret_cast<float*>(ws + ML.off_T1);
  float* K = reinterpret_cast<float*>(ws + ML.off_K);
  auto* Kb = reinterpret_cast<__nv_bfloat16*>(ws + ML.off_Kb);
  if (bf16) {
    // Tensor-core passes with the identity split (tc_merge.cuh):
    //   W1 = (W0' B_P)^T as hi/lo, then K = (W1 B_R^T)^T = B_R W0' B_P.
    auto* W1hi = reinterpret_cast<__nv_bfloat16*>(ws + ML.off_W1hi);
    auto* W1lo = reinterpret_cast<__nv_bfloat16*>(ws + ML.off_W1lo);
    auto* DPhi = reinterpret_cast<__nv_bfloat16*>(ws + ML.off_DPhi);
    auto* DPlo = reinterpret_cast<__nv_bfloat16*>(ws + ML.off_DPlo);
    auto* DRhi = reinterpret_cast<__nv_bfloat16*>(ws + ML.off_DRhi);
    auto* DRlo = reinterpret_cast<__nv_bfloat16*>(ws + ML.off_DRlo);
    const float* BP = reinterpret_cast<const float*>(pb + L.P.off_B);
    const float* BR = reinterpret_cast<const float*>(pb + L.R.off_B);
    delta_superblock_kernel<<<grid_for(static_cast<int64_t>(L.P.nsb) * L.P.sb * L.P.sb), 256, 0, st>>>(
        BP, L.P.g, L.P.sb, L.P.nsb, 1, DPhi, DPlo);
    POETX_LAUNCHED();
    delta_superblock_kernel<<<grid_for(static_cast<int64_t>(L.R.nsb) * L.R.sb * L.R.sb), 256, 0, st>>>(
        BR, L.R.g, L.R.sb, L.R.nsb, 0, DRhi, DRlo);
    POETX_LAUNCHED();
    const bool q8 = weight_int8(*desc);
    auto* Klo = q8 ? reinterpret_cast<__nv_bfloat16*>(ws + ML.off_Klo) : nullptr;
    if (q8) {
      // the exact scale * code as a hi + lo pair: the first pass then splits A too
      auto* Wdq = reinterpret_cast<__nv_bfloat16*>(ws + ML.off_Wdq);
      auto* Wdqlo = reinterpret_cast<__nv_bfloat16*>(ws + ML.off_Wdqlo);
      POETX_TRY(dequant_weight(st, *desc, W0p, Wdq, Wdqlo));
      POETX_TRY(tc_merge_pass<true>(st, Wdq, Wdqlo, m, n, L.P.sb, L.P.nsb, DPhi, DPlo, W1hi, W1lo));
    } else {
      POETX_TRY(tc_merge_pass<false>(st, reinterpret_cast<const __nv_bfloat16*>(W0p), nullptr, m, n,
                                     L.P.sb, L.P.nsb, DPhi, DPlo, W1hi, W1lo));
    }
    // int8 weights keep K as hi + lo so the codes come from the fp32-grade K
    POETX_TRY(tc_merge_pass<true>(st, W1hi, W1lo, n, m, L.R.sb, L.R.nsb, DRhi, DRlo, Kb, Klo));
  } else {
    // T1 = W0' blockdiag(B_P): row-local blocks along n (not transposed).
    POETX_TRY(simt_blocks<float, float>(st, L.P, pb, reinterpret_cast<const float*>(W0p), T1, m, n,
                                        false));
    // K = blockdiag(B_R) T1: block k of rows is B_R,k (b x b) times T1[rows of k, :].
    const SideLayout& S = L.R;
    const int b = S.g.b;
    const int64_t bb = static_cast<int64_t>(b) * b;
    const float* BR = reinterpret_cast<const float*>(pb + S.off_B);
    const int full = S.g.nblk - (S.g.last < b ? 1 : 0);
    POETX_TRY(simt_gemm<float, float, float>(st, b, n, b, full, BR, b, 1, bb, T1, n, 1,
                                             static_cast<int64_t>(b) * n, K, n, 1,
                                             static_cast<int64_t>(b) * n, 1.f, 0.f));
    if (S.g.last < b) {
      const int64_t o = static_cast<int64_t>(full) * b * n;
      POETX_TRY(simt_gemm<float, float, float>(st, S.g.last, n, S.g.last, 1, BR + full * bb, b, 1, 0,
                                               T1 + o, n, 1, 0, K + o, n, 1, 0, 1.f, 0.f));
    }
  }
  // rho = pi_old^-1 o pi_new on both sides.
  std::vector<int32_t> oR, oRi, oP, oPi, nR, nRi, nP, nPi;
  perm_and_inverse(desc->seed_R, m, oR, oRi);
  perm_and_inverse(desc->seed_P, n, oP, oPi);
  perm_and_inverse(new_seed_R, m, nR, nRi);
  perm_and_inverse(new_seed_P, n, nP, nPi);
  std::vector<int32_t> rR(m), rP(n);
  for (int i = 0; i < m; ++i) rR[i] = oRi[nR[i]];
  for (int j = 0; j < n; ++j) rP[j] = oPi[nP[j]];
  POETX_TRY(ring_upload(st, {{rR.data(), rR.size()}, {rP.data(), rP.size()}}, {rhoR, rhoP}));
  const int grid = std::min(m, device_sm_count() * 8);
  if (weight_int8(*desc))  // re-basing copy and row quantization in one pass
    return quantize_weight(st, *desc, Kb, reinterpret_cast<const __nv_bfloat16*>(ws + ML.off_Klo), rhoR,
                           rhoP, W0p);
  if (bf16)
    gather2d_kernel<__nv_bfloat16, __nv_bfloat16><<<grid, 256, 0, st>>>(
        Kb, reinterpret_cast<__nv_bfloat16*>(W0p), rhoR, rhoP, m, n);
  else
    gather2d_kernel<float, float><<<grid, 256, 0, st>>>(K, reinterpret_cast<float*>(W0p), rhoR, rhoP,
                                                        m, n);
  POETX_LAUNCHED();
  return POETX_OK;
}

}  // extern "C"

namespace {

// One non-blocking stream per device for the second host-to-device copy of
// poetx_linear_step_host, created on first use and kept for the process;
// nullptr if it cannot be created (both copies then go on the caller's
// stream).
cudaStream_t step_copy_stream() {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static cudaStream_t streams[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    (void)cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!streams[dev] && cudaStreamCreateWithFlags(&streams[dev], cudaStreamNonBlocking) != cudaSuccess) {
    (void)cudaGetLastError();
    streams[dev] = nullptr;
  }
  return streams[dev];
}

// One forward + backward step from host buffers (see poetx_linear_step_host
// and poetx_linear_step_host_async in poetx.h).
poetx_status step_host_impl(const poetx_layer_desc* desc, const void* params, const void* W0p,
                            const void* X_host, const void* dY_host, int64_t T, void* X_dev,
                            void* dY_dev, void* Y_dev, void* saved_h_dev, void* saved_u_dev,
                            void* dX_dev, float* dGenR_dev, float* dGenP_dev, float* dGenR_host,
                            float* dGenP_host, void* workspace, void* stream, bool async) {
  POETX_TRY(check_desc(desc));
  if (T < 0 || !X_host || !dY_host || !X_dev || !dY_dev || !dGenR_host || !dGenP_host)
    return POETX_ERR_INVALID_ARG;
  // the forward and backward take at most 2^31 - 256 tokens: refuse before
  // any copy is enqueued
  if (T > (int64_t(1) << 31) - 256) return POETX_ERR_UNSUPPORTED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const size_t e = desc->dtype == POETX_DTYPE_BF16 ? 2 : 4;
  const size_t xb = static_cast<size_t>(T) * desc->n * e, yb = static_cast<size_t>(T) * desc->m * e;
  cudaStream_t cs = step_copy_stream();
  Ev x_done, dy_done;
  if (async && cs) {
    // both copies on the copy stream, X first, not ordered after earlier
    // work on `stream` (the caller guarantees the device buffers are free):
    // consecutive calls keep the host link busy while earlier layers compute
    POETX_CUDA(cudaMemcpyAsync(X_dev, X_host, xb, cudaMemcpyHostToDevice, cs));
    POETX_TRY(x_done.record(cs));
    POETX_CUDA(cudaMemcpyAsync(dY_dev, dY_host, yb, cudaMemcpyHostToDevice, cs));
    POETX_TRY(dy_done.record(cs));
    POETX_TRY(x_done.wait_on(st));
  } else if (cs) {
    // dY is copied on a second stream once X has arrived, so that it crosses
    // the host link while the forward runs (the two copies would only share
    // the link if they overlapped each other); the backward waits for it.
    // The wait on an event of `st` also orders the copy after all earlier
    // work on `st`, which may still read dY_dev.
    POETX_CUDA(cudaMemcpyAsync(X_dev, X_host, xb, cudaMemcpyHostToDevice, st));
    POETX_TRY(x_done.record(st));
    POETX_TRY(x_done.wait_on(cs));
    POETX_CUDA(cudaMemcpyAsync(dY_dev, dY_host, yb, cudaMemcpyHostToDevice, cs));
    POETX_TRY(dy_done.record(cs));
  } else {
    POETX_CUDA(cudaMemcpyAsync(X_dev, X_host, xb, cudaMemcpyHostToDevice, st));
    POETX_CUDA(cudaMemcpyAsync(dY_dev, dY_host, yb, cudaMemcpyHostToDevice, st));
  }
  auto run = [&]() -> poetx_status {
    POETX_TRY(poetx_linear_fwd(desc, params, W0p, X_dev, T, Y_dev, saved_h_dev, saved_u_dev,
                               workspace, stream));
    if (cs) POETX_TRY(dy_done.wait_on(st));
    return poetx_linear_bwd(desc, params, W0p, X_dev, dY_dev, saved_h_dev, saved_u_dev, T, dX_dev,
                            dGenR_dev, dGenP_dev, 0, workspace, stream);
  };
  const poetx_status rs = run();
  if (rs != POETX_OK) {
    // the copies may still be reading the caller's host buffers: wait for the
    // copy stream, and for the caller's stream when the copies ran on it or
    // the call is synchronous (results ignored: the first error is returned)
    if (cs) (void)cudaStreamSynchronize(cs);
    if (!cs || !async) (void)cudaStreamSynchronize(st);
    return rs;
  }
  const int64_t lr = poetx_gen_length(desc->m, desc->b_R), lp = poetx_gen_length(desc->n, desc->b_P);
  if (lr > 0)
    POETX_CUDA(cudaMemcpyAsync(dGenR_host, dGenR_dev, lr * 4, cudaMemcpyDeviceToHost, st));
  if (lp > 0)
    POETX_CUDA(cudaMemcpyAsync(dGenP_host, dGenP_dev, lp * 4, cudaMemcpyDeviceToHost, st));
  if (!async) POETX_CUDA(cudaStreamSynchronize(st));
  return POETX_OK;
}

}  // namespace

extern "C" {

poetx_status poetx_linear_step_host(const poetx_layer_desc* desc, const void* params, const void* W0p,
                                    const void* X_host, const void* dY_host, int64_t T, void* X_dev,
                                    void* dY_dev, void* Y_dev, void* saved_h_dev, void* saved_u_dev,
                                    void* dX_dev, float* dGenR_dev, float* dGenP_dev,
                                    float* dGenR_host, float* dGenP_host, void* workspace,
                                    void* stream) {
  return step_host_impl(desc, params, W0p, X_host, dY_host, T, X_dev, dY_dev, Y_dev, saved_h_dev,
                        saved_u_dev, dX_dev, dGenR_dev, dGenP_dev, dGenR_host, dGenP_host, workspace,
                        stream, false);
}

poetx_status poetx_linear_step_host_async(const poetx_layer_desc* desc, const void* params,
                                          const void* W0p, const void* X_host, const void* dY_host,
                                          int64_t T, void* X_dev, void* dY_dev, void* Y_dev,
                                          void* saved_h_dev, void* saved_u_dev, void* dX_dev,
                                          float* dGenR_dev, float* dGenP_dev, float* dGenR_host,
                                          float* dGenP_host, void* workspace, void* stream) {
  return step_host_impl(desc, params, W0p, X_host, dY_host, T, X_dev, dY_dev, Y_dev, saved_h_dev,
                        saved_u_dev, dX_dev, dGenR_dev, dGenP_dev, dGenR_host, dGenP_host, workspace,
                        stream, true);
}

poetx_status poetx_generator_adamw(float* gen, const float* grad, float* m1, float* m2, int64_t len,
                                   int64_t step, float lr, float beta1, float beta2, float eps,
                                   float weight_decay, void* stream) {
  if (len < 0 || step < 1) return POETX_ERR_INVALID_ARG;
  if (len == 0) return POETX_OK;
  if (!gen || !grad || !m1 || !m2) return POETX_ERR_INVALID_ARG;
  if (!(beta1 >= 0.f && beta1 < 1.f && beta2 >= 0.f && beta2 < 1.f && eps >= 0.f))
    return POETX_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const double bc1 = 1.0 - std::pow(static_cast<double>(beta1), static_cast<double>(step));
  const double bc2 = 1.0 - std::pow(static_cast<double>(beta2), static_cast<double>(step));
  const float step_size = static_cast<float>(static_cast<double>(lr) / bc1);
  const float inv_sqrt_bc2 = static_cast<float>(1.0 / std::sqrt(bc2));
  const float decay = static_cast<float>(1.0 - static_cast<double>(lr) * weight_decay);
  return launch_dep(adamw_kernel, grid_for(len), 256, 0, st, 0, gen, grad, m1, m2, len, beta1, beta2, eps,
                    decay, step_size, inv_sqrt_bc2);
}

poetx_status poetx_device_status(int32_t reset) {
  POETX_CUDA(cudaDeviceSynchronize());
  unsigned int w = 0;
  POETX_CUDA(cudaMemcpyFromSymbol(&w, g_status_word, sizeof(w)));
  if (reset) {
    const unsigned int zero = 0;
    POETX_CUDA(cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero)));
  }
  if (w & kStatusTimeout) return POETX_ERR_TIMEOUT;
  if (w & kStatusBadArgs) return POETX_ERR_INVALID_ARG;
  return POETX_OK;
}

}  // extern "C"

namespace {
__device__ int g_selftest_result;
}

extern "C" {

poetx_status poetx_selftest_bounded_wait(uint64_t timeout_ns, void* stream) {
  if (timeout_ns < 1000ull || timeout_ns > 10000000000ull) return POETX_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  POETX_CUDA(cudaStreamSynchronize(st));
  unsigned int before = 0;
  POETX_CUDA(cudaMemcpyFromSymbol(&before, g_status_word, sizeof(before)));
  int* result = nullptr;
  POETX_CUDA(cudaGetSymbolAddress(reinterpret_cast<void**>(&result), g_selftest_result));
  POETX_CUDA(cudaMemsetAsync(result, 0, sizeof(int), st));
  bounded_wait_selftest_kernel<<<1, 32, 0, st>>>(timeout_ns, result);
  POETX_LAUNCHED();
  POETX_CUDA(cudaStreamSynchronize(st));
  int r = 0;
  unsigned int after = 0;
  POETX_CUDA(cudaMemcpyFromSymbol(&r, g_selftest_result, sizeof(r)));
  POETX_CUDA(cudaMemcpyFromSymbol(&after, g_status_word, sizeof(after)));
  // leave the status word as it was: this timeout was requested
  POETX_CUDA(cudaMemcpyToSymbol(g_status_word, &before, sizeof(before)));
  if (r == 2 && (after & kStatusTimeout)) return POETX_ERR_TIMEOUT;
  if (r == 1) return POETX_OK;
  return POETX_ERR_CUDA;
}

void poetx_set_wait_timeout_ns(uint64_t timeout_ns) {
  g_timeout_ns = timeout_ns ? timeout_ns : kDefaultTimeoutNs;
}

void poetx_set_dependent_launch(int32_t on) {
  g_dependent_launch.store(on != 0, std::memory_order_relaxed);
}

void poetx_set_fused_gather_max_features(int32_t max_features) {
  g_gbd_max_cols.store(max_features < 0 ? kGbdDefaultMaxCols : max_features, std::memory_order_relaxed);
}

}  // extern "C"

extern "C" {

void poetx_profile_enable(int32_t on) {
  std::lock_guard<std::mutex> lock(g_prof.mu);
  g_prof.on = on != 0;
}

void poetx_profile_reset(void) {
  std::lock_guard<std::mutex> lock(g_prof.mu);
  for (auto& r : g_prof.recs) {
    g_prof.pool.push_back(r.start);
    g_prof.pool.push_back(r.stop);
  }
  g_prof.recs.clear();
}

poetx_status poetx_profile_read(int32_t kind, int64_t* groups, double* total_ms) {
  if (kind < 0 || kind >= POETX_NUM_KINDS || !groups || !total_ms) return POETX_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_prof.mu);
  int64_t n = 0;
  double ms = 0.0;
  for (auto& r : g_prof.recs) {
    if (r.kind != kind) continue;
    if (cudaEventSynchronize(r.stop) != cudaSuccess) return POETX_ERR_CUDA;
    float t = 0.f;
    if (cudaEventElapsedTime(&t, r.start, r.stop) != cudaSuccess) return POETX_ERR_CUDA;
    ms += t;
    ++n;
  }
  *groups = n;
  *total_ms = ms;
  return POETX_OK;
}

const char* poetx_profile_kind_name(int32_t kind) {
  static const char* names[POETX_NUM_KINDS] = {"gemm_fwd", "gemm_dgrad", "blockdiag", "gradred",
                                               "gather", "build", "genbwd", "merge", "simt",
                                               "dequant"};
  return (kind >= 0 && kind < POETX_NUM_KINDS) ? names[kind] : "unknown";
}

int64_t poetx_launch_count(void) { return g_launches.load(); }

}  // extern "C"

// ====================================================================== allocation-free forward
// Scratch for poetx_linear_fwd_noalloc: a fixed device array in this module.
// In host code its name is only a host-side stand-in, so the device address
// is looked up once per device with cudaGetSymbolAddress and cached.
static __device__ __align__(256) unsigned char g_noalloc_scratch[POETX_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kNoAllocMaxDevices] = {};
}  // namespace

extern "C" poetx_status poetx_linear_fwd_noalloc(const poetx_layer_desc* desc, const void* params,
                                                 const void* W0p, const void* X, int64_t T, void* Y,
                                                 void* saved_h, void* saved_u, void* stream) {
  POETX_TRY(check_desc(desc));
  if (T < 0) return POETX_ERR_INVALID_ARG;
  if (T == 0) return POETX_OK;
  const size_t need = poetx_workspace_size(desc, T);
  if (need == 0 || need > POETX_NOALLOC_SCRATCH_BYTES) return POETX_ERR_UNSUPPORTED;
  int dev = 0;
  POETX_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kNoAllocMaxDevices) return POETX_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
      void* addr = nullptr;
      POETX_CUDA(cudaGetSymbolAddress(&addr, g_noalloc_scratch));
      g_noalloc_addr[dev] = addr;
    }
    scratch = g_noalloc_addr[dev];
  }
  return poetx_linear_fwd(desc, params, W0p, X, T, Y, saved_h, saved_u, scratch, stream);
}
