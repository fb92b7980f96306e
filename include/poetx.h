/*
 * poetx.h -- C ABI of the POET-X orthogonal-equivalence linear layer on one
 * NVIDIA B300 (sm_103a).
 *
 * The layer.  W = R W0 P with W0 (m x n) frozen and R (m x m), P (n x n)
 * orthogonal ("POET-X: Memory-efficient LLM Training by Scaling Orthogonal
 * Transformation", gist.science summary, Methodologie §1: the update
 * W <- R_i W P_i rewritten as linear maps on the input).  R and P are
 * block-diagonal in a permuted basis (Methodologie §2: permutations as index
 * maps, two of the four folded into the weight ahead of time; §3: blocks
 * handled as independent matrices).  Each block B is the Cayley image of a
 * skew matrix Q, B = (I+Q)(I-Q)^-1 ("POET-X：基于正交变换缩放的内存高效LLM训练方法",
 * ai-stack.site, 实践 2), or its truncated Neumann form (Methodologie §4);
 * only the strict upper triangle of Q is stored (Methodologie §4).
 *
 * Conventions fixed by this library (the pages leave them open):
 *   - Activations are row-major: X is T x n, Y is T x m, Y = X W^T.
 *   - A permutation is an int32 array pi with (Pi x)_j = x_{pi(j)}.
 *     R = Pi_R^T blockdiag(B_R) Pi_R and P = Pi_P^T blockdiag(B_P) Pi_P.
 *   - pi is splitmix64(seed) driving a Fisher-Yates shuffle (i from d-1 down
 *     to 1, j uniform in [0, i] by rejection of the top partial bucket).
 *   - Blocks are contiguous in the permuted basis; if b does not divide d the
 *     last block has size d mod b and its own generator.
 *   - Packed generator: blocks concatenated; in a block of size s entry
 *     (i, j), i < j, sits at i*s - i*(i+1)/2 + (j-i-1); Q = U - U^T.
 *   - Neumann mode of order k: B = (I+Q)(I + Q + ... + Q^k).
 *   - W0' = Pi_R W0 Pi_P^T (W0'[i][j] = W0[pi_R(i)][pi_P(j)]) is the weight
 *     the forward and backward passes consume.
 *
 * Memory.  Every pointer argument is DEVICE memory owned by the caller
 * unless its comment says HOST.  The library allocates no device memory on
 * any path; per-call scratch comes from the caller's `workspace`, sized by
 * the matching *_workspace_size function, 256-byte aligned.  The one
 * exception is a fixed module array of POETX_NOALLOC_SCRATCH_BYTES that
 * every device loading the library holds from module load until exit, the
 * scratch of poetx_linear_fwd_noalloc (and of nothing else).  Layer state
 * (block matrices, permutations) lives in the caller's `params` buffer of
 * poetx_params_size() bytes, 256-byte aligned.
 *
 * Streams.  `stream` is a cudaStream_t passed as void*; NULL means the legacy
 * default stream.  Every call is asynchronous on that stream unless stated.
 * The host waits only in poetx_device_status, poetx_linear_step_host, and
 * the two calls that copy host-generated permutations (poetx_params_build,
 * poetx_merge).  Those stage the indices in a process-wide ring of 32 pinned
 * HOST slots: a call waits for the copy issued 32 such calls earlier if it
 * is still pending, and the first call for a wider layer than any before
 * replaces the ring (after its pending copies finish).
 *
 * Devices and threads.  A process uses the library on one device: the
 * device current at the first call fixes the SM count that sizes grids and
 * workspaces, and each kernel's shared-memory limit is raised once, on that
 * device.  Calls for another device in the same process are not supported
 * (their launches may fail with POETX_ERR_CUDA).  Entry points may be called
 * from several host threads; calls that share a workspace, params buffer or
 * output must be ordered by the caller (same stream, or events).
 *
 * Errors.  Argument errors return a status before any launch and leave all
 * outputs untouched.  A failed launch returns POETX_ERR_CUDA.  Kernels that
 * wait on a barrier give up after a bounded time, record the fact in a
 * device status word and return; poetx_device_status() reports it as
 * POETX_ERR_TIMEOUT.  No function throws across this boundary.
 *
 * Precision.  dtype FP32: every step in fp32 on CUDA cores.  dtype BF16:
 * X, Y, dX, dY, W0' and the saved h are bf16; block matrices are built in
 * fp32 and rounded to bf16 for the tensor-core contractions, which
 * accumulate in fp32; generator gradients are reduced and returned in fp32.
 * Generators are always fp32.
 */
#ifndef POETX_H
#define POETX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum poetx_status {
  POETX_OK = 0,
  POETX_ERR_INVALID_ARG = 1,  /* null pointer, bad size, bad enum value      */
  POETX_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. dims % 8)   */
  POETX_ERR_MISALIGNED = 3,   /* a pointer is not 256-byte (buffers) or
                                 16-byte (tensors) aligned                    */
  POETX_ERR_CUDA = 4,         /* a CUDA call or launch failed                */
  POETX_ERR_TIMEOUT = 5       /* a device-side bounded wait ran out          */
} poetx_status;

enum { POETX_MODE_CAYLEY = 0, POETX_MODE_NEUMANN = 1 };
enum { POETX_DTYPE_FP32 = 0, POETX_DTYPE_BF16 = 1 };

/* Storage of the pre-merged base weight W0p.
 *   POETX_WEIGHT_DENSE: m x n values of the layer dtype.
 *   POETX_WEIGHT_INT8:  POET-XQ (Methodologie §5: the base weights are stored
 *     quantized, e.g. INT8, and dequantized on the fly).  The scheme is a
 *     reading, as the pages give none: symmetric per row, scale_i =
 *     max_j |W0p[i][j]| / 127 and code_ij = round-half-to-even(W0p[i][j] /
 *     scale_i) clamped to [-127, 127], computed in float32; a zero row has
 *     scale 0.  The layer computes with scale_i * code_ij.  Buffer layout:
 *     m x n int8 codes (row-major), then, at the next multiple of 256 bytes,
 *     m float32 scales; poetx_weight_size gives the total.  bf16 layers only. */
enum { POETX_WEIGHT_DENSE = 0, POETX_WEIGHT_INT8 = 1 };

/* Geometry and options of one layer.  m, n >= 1; 1 <= b_R <= m and
 * 1 <= b_P <= n.  BF16 additionally needs m and n multiples of 8 (16-byte
 * rows for the tensor-memory-accelerator copies) and b_R, b_P in
 * {32, 64, 128, 256, 512}.  neumann_k >= 1 is read in Neumann mode only.
 * weight_format is POETX_WEIGHT_DENSE or (bf16 only) POETX_WEIGHT_INT8. */
typedef struct poetx_layer_desc {
  int32_t m, n;
  int32_t b_R, b_P;
  uint64_t seed_R, seed_P;
  int32_t mode;
  int32_t neumann_k;
  int32_t dtype;
  int32_t weight_format;
} poetx_layer_desc;

/* Human-readable name of a status code (static storage). */
const char* poetx_status_string(int32_t status);

/* Library ABI version (major*1000 + minor). */
int32_t poetx_version(void);

/* HOST.  Writes the permutation of 0..d-1 generated from `seed` (the
 * Fisher-Yates/splitmix64 recipe above) into host_out[0..d-1].
 * Source: Methodologie §2 (permutations realised as index maps).
 * Errors: INVALID_ARG if d < 1 or host_out is NULL. */
poetx_status poetx_perm_generate(uint64_t seed, int32_t d, int32_t* host_out);

/* Number of fp32 entries in the packed generator of a d-dimensional side
 * with block size b (sum over blocks of s(s-1)/2).  Methodologie §4.
 * Returns -1 on invalid arguments. */
int64_t poetx_gen_length(int32_t d, int32_t b);

/* Bytes of the params buffer for `desc`; 0 if desc is invalid. */
size_t poetx_params_size(const poetx_layer_desc* desc);

/* Builds the layer state into `params` (caller-owned device memory of
 * poetx_params_size bytes, 256-byte aligned): the permutations pi_R, pi_P
 * and their inverses (generated on the host and copied on `stream`), and
 * per block B = (I+Q)(I-Q)^-1 (exact Cayley, fp32 Gauss-Jordan) or the
 * Neumann polynomial, plus the backward's auxiliaries.
 * genR: device fp32[poetx_gen_length(m, b_R)]; genP: [poetx_gen_length(n, b_P)].
 * Source: Methodologie §2 and §4; 实践 2.
 * Errors: INVALID_ARG, UNSUPPORTED, MISALIGNED, CUDA. */
poetx_status poetx_params_build(const poetx_layer_desc* desc, const float* genR,
                                const float* genP, void* params, void* stream);

/* Bytes of the pre-merged weight buffer W0p in the desc's weight format
 * (0 for an invalid desc). */
size_t poetx_weight_size(const poetx_layer_desc* desc);

/* Rebuilds only the block matrices of params from new generators (the
 * builder step of poetx_params_build), leaving the permutations that
 * poetx_params_build wrote for the desc's seeds untouched.  It launches
 * device work only (no host-to-device copies and no host synchronisation),
 * so a training step that changes the generators but not the seeds can be
 * captured in a CUDA graph with it.  Arguments and errors as for
 * poetx_params_build; params must already hold the permutations of the
 * desc's seeds. */
poetx_status poetx_blocks_build(const poetx_layer_desc* desc, const float* genR,
                                const float* genP, void* params, void* stream);

/* Pre-merges the two permutations adjacent to W0 into it:
 * W0p[i][j] = W0[pi_R(i)][pi_P(j)].  W0 is row-major m x n of the layer
 * dtype; W0p is in the desc's weight format (for POETX_WEIGHT_INT8 the
 * permuted rows are quantized as described there; the codes depend only on
 * W0 and the permutations).  W0 and W0p must not overlap.  params must come
 * from poetx_params_build with the same desc.  Source: Methodologie §2 (two
 * of the four forward permutations merged into the weight ahead of time). */
poetx_status poetx_weight_premerge(const poetx_layer_desc* desc, const void* params,
                                   const void* W0, void* W0p, void* stream);

/* Scratch bytes that poetx_linear_fwd / poetx_linear_bwd need for T tokens. */
size_t poetx_workspace_size(const poetx_layer_desc* desc, int64_t T);

/* Forward, input-centric: Y = R(W0(P x)) for each of the T rows of X,
 * never forming R W0 P (Methodologie §1, §2, §3):
 *   u = X[:, pi_P];  v_k = u_k B_P,k^T;  h = v W0'^T;  z_k = h_k B_R,k^T;
 *   Y[:, pi_R] = z.
 * W0p is in the desc's weight format; an int8 weight is dequantized into the
 * workspace (scale_i * code_ij rounded to bf16) at the start of each call.
 * X: T x n, Y: T x m (dtype).  saved_h: T x m (dtype) receives h, or NULL
 * for activation recompute in the backward (Methodologie §5, POET-Xmem).
 * saved_u: T x n (dtype) receives the permuted input u, or NULL; the
 * backward reads it instead of permuting X again.  Both are caller-owned and
 * must not alias X, Y or each other.
 * T = 0 is a no-op.  Errors: INVALID_ARG, MISALIGNED, CUDA. */
poetx_status poetx_linear_fwd(const poetx_layer_desc* desc, const void* params,
                              const void* W0p, const void* X, int64_t T, void* Y,
                              void* saved_h, void* saved_u, void* workspace, void* stream);

/* Backward of L with upstream gradient dY (T x m):
 *   dz = dY[:, pi_R];  G_R,k = dz_k^T h_k;  dh_k = dz_k B_R,k;
 *   dv = dh W0';       G_P,k = dv_k^T u_k;  du_k = dv_k B_P,k;
 *   dX[:, pi_P] = du;
 * then per block the Cayley backward dL/dQ = 2 M^T G M^T with
 * M = (I-Q)^-1 (or the Neumann chain rule) and the packed gradient
 * g_ij = dL/dQ[i][j] - dL/dQ[j][i] for i < j.
 * saved_h: the h written by poetx_linear_fwd, or NULL to recompute v and h.
 * saved_u: the u written by poetx_linear_fwd, or NULL to permute X again;
 * X may be NULL when saved_u is given (it is then not read).  Whatever is
 * saved is reused and whatever is not is recomputed, so the four
 * combinations trade memory (T x m and T x n per saved tensor) against
 * recompute (a GEMM for h, one permutation pass for u).
 * dX: T x n or NULL to skip it.  dGenR/dGenP: fp32 packed
 * gradients (lengths as for the generators); accumulate != 0 adds into them.
 * Errors: INVALID_ARG, MISALIGNED, CUDA. */
poetx_status poetx_linear_bwd(const poetx_layer_desc* desc, const void* params,
                              const void* W0p, const void* X, const void* dY,
                              const void* saved_h, const void* saved_u, int64_t T, void* dX,
                              float* dGenR, float* dGenP, int32_t accumulate, void* workspace,
                              void* stream);

/* Scratch bytes that poetx_merge needs. */
size_t poetx_merge_workspace_size(const poetx_layer_desc* desc);

/* Merge (Methodologie §1, W <- R W P): folds the current R and P into the
 * base weight and re-expresses it under the permutations of
 * (new_seed_R, new_seed_P): with K = blockdiag(B_R) W0p blockdiag(B_P),
 * W0p_new[i][j] = K[pi_R^-1(pi'_R(i))][pi_P^-1(pi'_P(j))], accumulated in fp32
 * and rounded once to dtype.  An int8 weight (POET-XQ) is dequantized, merged
 * and quantized again per row from the fp32-grade K (each code then lies
 * within one step of the exact result).  W0p is updated in place.  The caller then
 * resets the generators to zero and rebuilds params with the new seeds;
 * the layer then computes the same map as before the merge.
 * Errors: INVALID_ARG, MISALIGNED, CUDA. */
poetx_status poetx_merge(const poetx_layer_desc* desc, const void* params, void* W0p,
                         uint64_t new_seed_R, uint64_t new_seed_P, void* workspace,
                         void* stream);

/* One forward+backward step from HOST buffers: copies X_host (T x n) and
 * dY_host (T x m) into the device buffers X_dev / dY_dev, runs
 * poetx_linear_fwd (into Y_dev, saved_h_dev, saved_u_dev) and
 * poetx_linear_bwd (into dX_dev, dGenR_dev, dGenP_dev, overwriting), and
 * copies the generator gradients back into dGenR_host / dGenP_host.  Host
 * buffers should be pinned for asynchronous copies.  Synchronises `stream`
 * before returning.  saved_h_dev and saved_u_dev may be NULL (recompute).
 * dY is copied on a second stream of the library once X has arrived, so that
 * it overlaps the forward; both copies stay ordered after earlier work on
 * `stream`.  Errors (returned before any copy): INVALID_ARG for T < 0 or a
 * NULL host buffer, device input buffer or host gradient; UNSUPPORTED for
 * T > 2^31 - 256; then the errors of poetx_linear_fwd / poetx_linear_bwd,
 * after which the call waits for its own copies before returning. */
poetx_status poetx_linear_step_host(const poetx_layer_desc* desc, const void* params,
                                    const void* W0p, const void* X_host,
                                    const void* dY_host, int64_t T, void* X_dev,
                                    void* dY_dev, void* Y_dev, void* saved_h_dev,
                                    void* saved_u_dev, void* dX_dev, float* dGenR_dev,
                                    float* dGenP_dev, float* dGenR_host, float* dGenP_host,
                                    void* workspace, void* stream);

/* Asynchronous form of poetx_linear_step_host: the same copies, forward,
 * backward and gradient copies, enqueued without synchronising.  Both host
 * to device copies run on a copy stream of the library (X first) and are NOT
 * ordered after earlier work on `stream`, so that a sequence of calls keeps
 * the host link busy with later layers' inputs while earlier layers compute.
 * The caller guarantees that X_dev and dY_dev are not in use by earlier,
 * unfinished work (give each call in flight its own device buffers, or
 * synchronise first).  The forward waits for X and the backward for dY on
 * `stream`; the gradient copies follow on `stream`.  The host gradients are
 * valid, and the host input buffers may be reused, once `stream` has been
 * synchronised.  Errors: as poetx_linear_step_host (on an error the call
 * waits for its own copies to finish before returning). */
poetx_status poetx_linear_step_host_async(const poetx_layer_desc* desc, const void* params,
                                          const void* W0p, const void* X_host,
                                          const void* dY_host, int64_t T, void* X_dev,
                                          void* dY_dev, void* Y_dev, void* saved_h_dev,
                                          void* saved_u_dev, void* dX_dev, float* dGenR_dev,
                                          float* dGenP_dev, float* dGenR_host,
                                          float* dGenP_host, void* workspace, void* stream);

/* One AdamW step on a packed generator array (the step after the backward).
 * The pages train the generators with an optimizer they do not name; the
 * reading is AdamW with decoupled weight decay (Loshchilov & Hutter, ICLR
 * 2019) and bias-corrected moments.  For e < len, in fp32:
 *   m1 = beta1 m1 + (1 - beta1) g;   m2 = beta2 m2 + (1 - beta2) g^2;
 *   gen = gen (1 - lr weight_decay)
 *         - (lr / (1 - beta1^step)) m1 / (sqrt(m2 / (1 - beta2^step)) + eps)
 * with g = grad[e].  gen, grad, m1, m2: device float arrays of len entries
 * (m1 and m2 zero before step 1); step >= 1; the bias corrections are
 * computed on the host in double.  len = 0 is a no-op.
 * Errors: INVALID_ARG, CUDA. */
poetx_status poetx_generator_adamw(float* gen, const float* grad, float* m1, float* m2, int64_t len,
                                   int64_t step, float lr, float beta1, float beta2, float eps,
                                   float weight_decay, void* stream);

/* Reads (and with reset != 0 clears) the device status word that bounded
 * waits write.  Synchronises the device.  Returns POETX_OK, POETX_ERR_TIMEOUT
 * if any kernel gave up on a wait since the last reset, or POETX_ERR_CUDA. */
poetx_status poetx_device_status(int32_t reset);

/* Self-test of the bounded-wait machinery: launches one kernel that waits
 * on a shared-memory barrier nothing will ever complete, with a deadline of
 * timeout_ns nanoseconds (1 us .. 10 s); the kernel must record the timeout
 * and return.  Returns the kernel's status (POETX_ERR_TIMEOUT when the
 * machinery works).  Synchronises `stream`. */
poetx_status poetx_selftest_bounded_wait(uint64_t timeout_ns, void* stream);

/* Sets the deadline (nanoseconds) of every bounded device wait in later
 * launches; 0 restores the default (2 s). */
void poetx_set_wait_timeout_ns(uint64_t timeout_ns);

/* Programmatic dependent launch of the forward, backward and optimizer
 * kernels (on by default; on != 0 turns it on).  When on, each of those
 * kernels may start on the GPU while the kernel before it on the same stream
 * finishes: it sets up its shared memory, barriers and tensor memory, then
 * waits for that kernel to complete before reading or writing global
 * memory, so results are identical either way; only the gaps between
 * launches change.  Applies to launches issued after the call (a captured
 * CUDA graph keeps the setting it was captured with). */
void poetx_set_dependent_launch(int32_t on);

/* Column permutation inside the block transform ("POET-X: Memory-efficient
 * LLM Training by Scaling Orthogonal Transformation", Methodologie §1-§2:
 * the permutations are index maps applied to the input).  For bf16 layers
 * with 128-wide super-blocks (b <= 128) whose permuted side has 256 to
 * max_features features, the forward gathers X -> u inside the P-side block
 * transform (one kernel writes u and v) and the backward gathers dY -> dz
 * inside the R-side transform + token reduction (dz is never written);
 * other sides run the separate gather pass.  Results are identical either
 * way (same bf16 values, same fp32 accumulation order).  Off by default (0):
 * on B300 the separate passes, launched as programmatic dependents from a
 * CUDA graph, were as fast or faster at every width measured.  A negative
 * value restores the default.  Applies to launches issued after the call (a
 * captured graph keeps its setting). */
void poetx_set_fused_gather_max_features(int32_t max_features);

/* Forward for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot call cudaMalloc or grow a memory pool at the point of use (for
 * example inference runtimes that own every byte of device memory in a fixed
 * arena, plugins whose host forbids device allocation inside its execution
 * callbacks, or hosts whose allocator belongs to another framework).  It computes exactly what
 * poetx_linear_fwd computes, with the same arguments except `workspace`:
 * its scratch is a fixed, file-scope device array of
 * POETX_NOALLOC_SCRATCH_BYTES bytes inside the library, which every GPU that
 * loads the library holds until the process exits.
 *
 * Limits and behaviour:
 *   - Sizes whose poetx_workspace_size(desc, T) exceeds
 *     POETX_NOALLOC_SCRATCH_BYTES are rejected with POETX_ERR_UNSUPPORTED
 *     before any launch (use poetx_linear_fwd with your own workspace).
 *   - It calls no cudaMalloc, cudaFree or other allocating routine (with
 *     the profiling counters off, as they are by default: when on, they
 *     create timing events).  The first call on each device looks up the
 *     array's device address (cudaGetSymbolAddress, with that device
 *     current) and caches it for the life of the process; make that first
 *     call outside any stream capture, and do not reset the device
 *     (cudaDeviceReset) after it, since the cached address would then name
 *     released module memory.
 *   - Every call on a device shares the same scratch and leaves its contents
 *     behind; the forward writes every scratch byte it reads, so nothing
 *     needs to start at zero.  Calls whose executions overlap on the GPU
 *     (different streams without ordering between them) race on the scratch:
 *     order them on one stream or with events.
 *   - Other arguments, errors and precision are those of poetx_linear_fwd. */
#define POETX_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
poetx_status poetx_linear_fwd_noalloc(const poetx_layer_desc* desc, const void* params,
                                      const void* W0p, const void* X, int64_t T, void* Y,
                                      void* saved_h, void* saved_u, void* stream);

/* Kernel classes reported by the profiling counters below. */
enum {
  POETX_KIND_GEMM_FWD = 0,    /* h = v W0'^T on tcgen05 (forward and recompute)   */
  POETX_KIND_GEMM_DGRAD = 1,  /* dv = dh W0' on tcgen05                            */
  POETX_KIND_BLOCKDIAG = 2,   /* block-diagonal transforms on tcgen05              */
  POETX_KIND_GRADRED = 3,     /* per-block token reductions dz^T h, dv^T u        */
  POETX_KIND_GATHER = 4,      /* feature permutations (gather / scatter)           */
  POETX_KIND_BUILD = 5,       /* Cayley / Neumann block builder                    */
  POETX_KIND_GENBWD = 6,      /* partial reduction, Cayley backward, packing       */
  POETX_KIND_MERGE = 7,       /* merge and weight pre-merge                        */
  POETX_KIND_SIMT = 8,        /* fp32 CUDA-core path of the layer                  */
  POETX_KIND_DEQUANT = 9,     /* int8 weight dequantization (POET-XQ)              */
  POETX_NUM_KINDS = 10
};

/* Profiling.  While enabled, each group of launches of one kernel class is
 * bracketed by CUDA events recorded on the launching stream (for the tensor-
 * core classes a group is a single launch).  Inside a stream capture the
 * events become event-record nodes of the graph, so a replay of the graph
 * times the captured launches (read after the replay; a later replay
 * overwrites the times).  poetx_profile_read synchronises
 * on those events and returns, for `kind`, the number of groups and their
 * summed device time in milliseconds.  poetx_profile_reset forgets all
 * records.  poetx_launch_count returns the number of kernel launches the
 * library has made since the process started (always counted). */
void poetx_profile_enable(int32_t on);
void poetx_profile_reset(void);
poetx_status poetx_profile_read(int32_t kind, int64_t* groups, double* total_ms);
const char* poetx_profile_kind_name(int32_t kind);
int64_t poetx_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* POETX_H */
