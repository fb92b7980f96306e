"""fp64 CPU oracle of the POET-X orthogonal-equivalence linear layer.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the package's smoke check
(``__graft_entry__.smoke``) and the benchmark's CPU-baseline leg may import
this module.  The CUDA library never calls it and shares no code with it.

What it computes, and where the pages define it
-----------------------------------------------
Sources (page title, then section):

* [X-nl]  "POET-X: Memory-efficient LLM Training by Scaling Orthogonal
  Transformation" (gist.science summary of arXiv 2603.05500), sections
  "Probleemstelling" and "Methodologie: POET-X" items 1-5.
* [X-zh]  "POET-X：基于正交变换缩放的内存高效LLM训练方法" (ai-stack.site),
  "实践 2：采用 Cayley 变换进行参数化" (the Cayley map of a skew matrix).
* [POET-zh] "POET方法：重塑大型语言模型训练新篇章" (showapi.com), §1.2
  (orthogonal transforms leave the spectrum unchanged).

The layer weight is W = R W0 P with W0 frozen and R, P orthogonal
([X-nl] Methodologie §1, the update W <- R_i W P_i).  R and P are
block-diagonal in a permuted basis ([X-nl] §2 permutations as index maps,
§3 block-diagonal blocks handled as independent matrices); every block is
the Cayley image of a skew matrix Q, B = (I+Q)(I-Q)^-1 ([X-zh] 实践 2;
[X-nl] §4 Cayley-Neumann parameterisation), or, in Neumann mode, the same
map with the inverse replaced by a truncated series ([X-nl] §4, which names
the highest terms Q^3 and Q^4).  Only the strict upper triangle of Q is
stored ([X-nl] §4).

Readings where the pages are silent (each is listed in the design notes):

* Activations are row-major X (T x n), Y (T x m), Y = X W^T.
* A permutation is an index array pi with (Pi x)_j = x_{pi(j)}; the layer
  uses R = Pi_R^T blockdiag(B_R) Pi_R and P = Pi_P^T blockdiag(B_P) Pi_P.
* Permutations come from splitmix64(seed) driving a Fisher-Yates shuffle
  with an unbiased bounded draw (rejection of the top partial bucket).
* Blocks are contiguous in the permuted index space; when b does not divide
  the dimension the last block is ragged, of size d mod b, with its own
  generator.
* Packed generator: blocks concatenated; inside a block of size s, entry
  (i, j), i < j, sits at i*s - i*(i+1)/2 + (j - i - 1) (row-major strict upper
  triangle), and Q = U - U^T.
* Neumann order k: B = (I+Q) * sum_{i=0..k} Q^i; k = 3 makes Q^3 and Q^4 the
  highest terms, as [X-nl] §4 names them.
* Merge folds R and P into the base weight and moves it to fresh
  permutations; the caller then resets the generators to zero.
* POET-XQ ([X-nl] Methodologie §5: base weights stored quantized, e.g. INT8,
  and dequantized on the fly; the scheme is not given): symmetric int8 per
  output row, scale = max|row| / 127, code = round-half-to-even(w / scale)
  clamped to [-127, 127], computed in float32 (the arithmetic that decides
  an integer code is the kernel's); an all-zero row has scale 0 and codes 0.
  The dequantized weight is scale * code.
* Generator optimizer step (the pages train with an optimizer they do not
  name): AdamW with decoupled weight decay (Loshchilov & Hutter, "Decoupled
  Weight Decay Regularization", ICLR 2019, Algorithm 2, with bias-corrected
  moments as in Adam).

Every function here is the plain definition: dense matrices, library
matmuls as single steps, no blocking or fusion beyond what the definition
states.
"""
from __future__ import annotations

import dataclasses
from typing import List, Sequence, Tuple

import numpy as np

__all__ = [
    "MASK64", "splitmix64", "bounded_draw", "permutation", "inverse_permutation",
    "perm_matrix", "block_sizes", "packed_length", "unpack_skew", "pack_antisym",
    "inverse_gauss_jordan", "cayley", "neumann", "LayerSpec", "blocks_of",
    "orthogonal_factor", "dense_weight", "premerged_weight", "forward_dense",
    "forward_input_centric", "backward", "merge", "loss_for_fd",
    "quantize_rows_int8", "dequantize_rows_int8", "adamw_step",
]

MASK64 = (1 << 64) - 1
_GAMMA = 0x9E3779B97F4A7C15


# --------------------------------------------------------------------------
# Permutations ([X-nl] Methodologie §2: permutations applied as index maps)
# --------------------------------------------------------------------------

def splitmix64(seed: int):
    """The splitmix64 generator (Steele, Lea & Flood, OOPSLA 2014): a 64-bit
    counter advanced by the golden-ratio gamma, each output a fixed mix of
    the counter.  State starts at ``seed``."""
    state = seed & MASK64
    while True:
        state = (state + _GAMMA) & MASK64
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
        yield z ^ (z >> 31)


def bounded_draw(gen, bound: int) -> int:
    """Uniform integer in [0, bound): draws at or above the largest multiple
    of ``bound`` that fits in 2^64 are rejected, the rest are reduced mod
    ``bound``."""
    limit = (1 << 64) - ((1 << 64) % bound)
    while True:
        r = next(gen)
        if r < limit:
            return r % bound


def permutation(seed: int, d: int) -> np.ndarray:
    """Fisher-Yates shuffle of 0..d-1 driven by splitmix64(seed).

    For i = d-1 down to 1: j = bounded_draw(i+1); swap entries i and j.
    """
    p = list(range(d))
    g = splitmix64(seed)
    for i in range(d - 1, 0, -1):
        j = bounded_draw(g, i + 1)
        p[i], p[j] = p[j], p[i]
    return np.array(p, dtype=np.int64)


def inverse_permutation(pi: np.ndarray) -> np.ndarray:
    inv = np.empty_like(pi)
    inv[pi] = np.arange(len(pi), dtype=pi.dtype)
    return inv


def perm_matrix(pi: np.ndarray) -> np.ndarray:
    """Dense Pi with (Pi x)_j = x_{pi(j)}, i.e. Pi[j, pi(j)] = 1."""
    d = len(pi)
    P = np.zeros((d, d))
    P[np.arange(d), pi] = 1.0
    return P


# --------------------------------------------------------------------------
# Generators and blocks ([X-nl] §3 block-diagonal, §4 packed upper triangle)
# --------------------------------------------------------------------------

def block_sizes(d: int, b: int) -> List[int]:
    """Sizes of the diagonal blocks: full blocks of b, then a ragged d mod b."""
    if b <= 0 or d <= 0:
        raise ValueError("d and b must be positive")
    sizes = [b] * (d // b)
    if d % b:
        sizes.append(d % b)
    return sizes


def packed_length(d: int, b: int) -> int:
    return sum(s * (s - 1) // 2 for s in block_sizes(d, b))


def unpack_skew(packed: np.ndarray, s: int) -> np.ndarray:
    """Q = U - U^T where U's strict upper triangle holds ``packed`` row by row."""
    U = np.zeros((s, s))
    k = 0
    for i in range(s):
        for j in range(i + 1, s):
            U[i, j] = packed[k]
            k += 1
    return U - U.T


def pack_antisym(G: np.ndarray) -> np.ndarray:
    """Gradient with respect to the packed entries: for a loss L(Q) with
    Q[i,j] = p and Q[j,i] = -p, dL/dp = G[i,j] - G[j,i] (i < j)."""
    s = G.shape[0]
    out = []
    for i in range(s):
        for j in range(i + 1, s):
            out.append(G[i, j] - G[j, i])
    return np.array(out)


# --------------------------------------------------------------------------
# Cayley map ([X-zh] 实践 2) and its truncated Neumann form ([X-nl] §4)
# --------------------------------------------------------------------------

def inverse_gauss_jordan(A: np.ndarray) -> np.ndarray:
    """Textbook Gauss-Jordan inversion with partial pivoting, fp64."""
    n = A.shape[0]
    M = np.hstack([np.array(A, dtype=np.float64), np.eye(n)])
    for k in range(n):
        p = k + int(np.argmax(np.abs(M[k:, k])))
        if M[p, k] == 0.0:
            raise np.linalg.LinAlgError("singular matrix")
        if p != k:
            M[[k, p]] = M[[p, k]]
        M[k] = M[k] / M[k, k]
        f = M[:, k].copy()
        f[k] = 0.0
        M -= np.outer(f, M[k])
    return M[:, n:]


def cayley(Q: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Exact Cayley map.  Returns (B, M) with M = (I - Q)^-1 and
    B = (I + Q) M; M is what the backward pass needs."""
    I = np.eye(Q.shape[0])
    M = inverse_gauss_jordan(I - Q)
    return (I + Q) @ M, M


def neumann(Q: np.ndarray, k: int) -> np.ndarray:
    """Cayley map with (I - Q)^-1 replaced by sum_{i=0..k} Q^i."""
    I = np.eye(Q.shape[0])
    S = np.zeros_like(Q)
    Qi = I
    for _ in range(k + 1):
        S = S + Qi
        Qi = Qi @ Q
    return (I + Q) @ S


@dataclasses.dataclass(frozen=True)
class LayerSpec:
    m: int
    n: int
    b_R: int
    b_P: int
    seed_R: int
    seed_P: int
    mode: str = "exact"        # "exact" | "neumann"
    neumann_k: int = 3


def blocks_of(packed: np.ndarray, d: int, b: int, mode: str, k: int):
    """Per block: (Q, B, aux) where aux is M = (I-Q)^-1 (exact) or None."""
    out = []
    off = 0
    packed = np.asarray(packed, dtype=np.float64)
    if len(packed) != packed_length(d, b):
        raise ValueError("packed generator has the wrong length")
    for s in block_sizes(d, b):
        L = s * (s - 1) // 2
        Q = unpack_skew(packed[off:off + L], s)
        off += L
        if mode == "exact":
            B, M = cayley(Q)
            out.append((Q, B, M))
        elif mode == "neumann":
            out.append((Q, neumann(Q, k), None))
        else:
            raise ValueError(mode)
    return out


def _block_diag(mats: Sequence[np.ndarray]) -> np.ndarray:
    d = sum(a.shape[0] for a in mats)
    out = np.zeros((d, d))
    o = 0
    for a in mats:
        s = a.shape[0]
        out[o:o + s, o:o + s] = a
        o += s
    return out


def orthogonal_factor(pi: np.ndarray, Bs: Sequence[np.ndarray]) -> np.ndarray:
    """Dense Pi^T blockdiag(B) Pi."""
    Pi = perm_matrix(pi)
    return Pi.T @ _block_diag(Bs) @ Pi


# --------------------------------------------------------------------------
# Forward ([X-nl] Methodologie §1 input-centric evaluation, §2, §3)
# --------------------------------------------------------------------------

def _layer(spec: LayerSpec, genR, genP, piR=None, piP=None):
    piR = permutation(spec.seed_R, spec.m) if piR is None else np.asarray(piR)
    piP = permutation(spec.seed_P, spec.n) if piP is None else np.asarray(piP)
    bR = blocks_of(genR, spec.m, spec.b_R, spec.mode, spec.neumann_k)
    bP = blocks_of(genP, spec.n, spec.b_P, spec.mode, spec.neumann_k)
    return piR, piP, bR, bP


def dense_weight(spec: LayerSpec, W0, genR, genP, piR=None, piP=None) -> np.ndarray:
    """W = R W0 P, formed densely (allowed in the oracle only)."""
    piR, piP, bR, bP = _layer(spec, genR, genP, piR, piP)
    R = orthogonal_factor(piR, [B for _, B, _ in bR])
    P = orthogonal_factor(piP, [B for _, B, _ in bP])
    return R @ np.asarray(W0, dtype=np.float64) @ P


def premerged_weight(W0, piR, piP) -> np.ndarray:
    """W0' = Pi_R W0 Pi_P^T, i.e. W0'[i, j] = W0[pi_R(i), pi_P(j)]: the two
    permutations adjacent to W0 folded in ahead of time ([X-nl] §2)."""
    W0 = np.asarray(W0, dtype=np.float64)
    return W0[np.asarray(piR)][:, np.asarray(piP)]


def forward_dense(spec: LayerSpec, W0, X, genR, genP, piR=None, piP=None) -> np.ndarray:
    """Y = X W^T with W = R W0 P."""
    W = dense_weight(spec, W0, genR, genP, piR, piP)
    return np.asarray(X, dtype=np.float64) @ W.T


def _apply_blocks(A: np.ndarray, blocks, transpose: bool) -> np.ndarray:
    """Columns of A grouped by block; block k maps a_k -> a_k B_k^T
    (transpose=True) or a_k -> a_k B_k (transpose=False)."""
    out = np.empty_like(A)
    o = 0
    for _, B, _ in blocks:
        s = B.shape[0]
        out[:, o:o + s] = A[:, o:o + s] @ (B.T if transpose else B)
        o += s
    return out


def forward_input_centric(spec: LayerSpec, W0, X, genR, genP, piR=None, piP=None):
    """Y = R(W0(P x)) per token, never forming R W0 P.

    u = X[:, pi_P]          (gather: Pi_P applied to each token)
    v = u blockdiag(B_P)^T  (P's blocks)
    h = v W0'^T             (W0' = Pi_R W0 Pi_P^T)
    z = h blockdiag(B_R)^T  (R's blocks)
    Y[:, pi_R] = z          (scatter: Pi_R^T)
    Returns (Y, dict of intermediates).
    """
    piR, piP, bR, bP = _layer(spec, genR, genP, piR, piP)
    X = np.asarray(X, dtype=np.float64)
    u = X[:, piP]
    v = _apply_blocks(u, bP, transpose=True)
    W0p = premerged_weight(W0, piR, piP)
    h = v @ W0p.T
    z = _apply_blocks(h, bR, transpose=True)
    Y = np.empty_like(z)
    Y[:, piR] = z
    return Y, dict(u=u, v=v, h=h, z=z, W0p=W0p, piR=piR, piP=piP, bR=bR, bP=bP)


# --------------------------------------------------------------------------
# Backward (chain rule of the forward above)
# --------------------------------------------------------------------------

def _generator_grad(blocks, G_blocks, mode: str, k: int) -> np.ndarray:
    """dL/d(packed) from dL/dB per block.

    Exact: B = 2M - I with M = (I-Q)^-1, dB = 2 M dQ M, so
    dL/dQ = 2 M^T G M^T.  Neumann: B = sum_p c_p Q^p with c_0 = 1,
    c_1..c_k = 2, c_{k+1} = 1, so dL/dQ = sum_p c_p sum_{a+b=p-1}
    (Q^T)^a G (Q^T)^b.  Then pack_antisym.
    """
    out = []
    for (Q, _, M), G in zip(blocks, G_blocks):
        if mode == "exact":
            GQ = 2.0 * M.T @ G @ M.T
        else:
            s = Q.shape[0]
            c = [1.0] + [2.0] * k + [1.0]
            Qt = Q.T
            pw = [np.eye(s)]
            for _ in range(k + 1):
                pw.append(pw[-1] @ Qt)
            GQ = np.zeros_like(G)
            for p in range(1, k + 2):
                for a in range(p):
                    GQ += c[p] * pw[a] @ G @ pw[p - 1 - a]
        out.append(pack_antisym(GQ))
    return np.concatenate(out) if out else np.zeros(0)


def backward(spec: LayerSpec, W0, X, dY, genR, genP, piR=None, piP=None):
    """Gradients of L = <dY, Y>: returns (dX, dgenR, dgenP, extras).

    dz = dY[:, pi_R];  G_R,k = dz_k^T h_k;  dh_k = dz_k B_R,k
    dv = dh W0';       G_P,k = dv_k^T u_k;  du_k = dv_k B_P,k
    dX[:, pi_P] = du
    """
    Y, it = forward_input_centric(spec, W0, X, genR, genP, piR, piP)
    dY = np.asarray(dY, dtype=np.float64)
    bR, bP = it["bR"], it["bP"]
    dz = dY[:, it["piR"]]
    GR, o = [], 0
    for _, B, _ in bR:
        s = B.shape[0]
        GR.append(dz[:, o:o + s].T @ it["h"][:, o:o + s])
        o += s
    dh = _apply_blocks(dz, bR, transpose=False)
    dv = dh @ it["W0p"]
    GP, o = [], 0
    for _, B, _ in bP:
        s = B.shape[0]
        GP.append(dv[:, o:o + s].T @ it["u"][:, o:o + s])
        o += s
    du = _apply_blocks(dv, bP, transpose=False)
    dX = np.empty_like(du)
    dX[:, it["piP"]] = du
    dgenR = _generator_grad(bR, GR, spec.mode, spec.neumann_k)
    dgenP = _generator_grad(bP, GP, spec.mode, spec.neumann_k)
    return dX, dgenR, dgenP, dict(Y=Y, GR=GR, GP=GP, dz=dz, dh=dh, dv=dv, du=du, **it)


def loss_for_fd(spec: LayerSpec, W0, X, dY, genR, genP, piR=None, piP=None) -> float:
    """L = <dY, Y> through the dense product: what finite differences probe."""
    Y = forward_dense(spec, W0, X, genR, genP, piR, piP)
    return float(np.sum(np.asarray(dY, dtype=np.float64) * Y))


# --------------------------------------------------------------------------
# Merge ([X-nl] Methodologie §1: W <- R_i W P_i)
# --------------------------------------------------------------------------

def merge(spec: LayerSpec, W0, genR, genP, new_seed_R: int, new_seed_P: int,
          piR=None, piP=None) -> np.ndarray:
    """Fold R and P into the base weight and re-express it under fresh
    permutations: W0_new = R W0 P, returned pre-merged for the new seeds,
    W0'_new = W0_new[pi'_R, :][:, pi'_P].  With the generators reset to zero
    and seeds (new_seed_R, new_seed_P) the layer computes the same map."""
    Wn = dense_weight(spec, W0, genR, genP, piR, piP)
    return premerged_weight(Wn, permutation(new_seed_R, spec.m),
                            permutation(new_seed_P, spec.n))


def quantize_rows_int8(W) -> Tuple[np.ndarray, np.ndarray]:
    """POET-XQ storage of a weight ([X-nl] Methodologie §5): per row i,
    scale_i = max_j |W[i, j]| / 127 and code_ij = round-half-to-even(
    W[i, j] / scale_i), clamped to [-127, 127].  All of it in float32, the
    precision in which the integer decision is taken; a zero row gets scale 0
    and codes 0.  Returns (codes int8 m x n, scales float32 m)."""
    W32 = np.asarray(W, dtype=np.float32)
    amax = np.max(np.abs(W32), axis=1)
    scale = (amax / np.float32(127.0)).astype(np.float32)
    safe = np.where(scale > 0, scale, np.float32(1.0)).astype(np.float32)
    q = np.rint(W32 / safe[:, None])          # float32 division; rint rounds half to even
    q = np.clip(q, -127, 127)
    q[scale == 0, :] = 0
    return q.astype(np.int8), scale


def dequantize_rows_int8(codes, scales) -> np.ndarray:
    """The weight a POET-XQ layer computes with: scale_i * code_ij (exact)."""
    return np.asarray(scales, dtype=np.float64)[:, None] * np.asarray(codes, dtype=np.float64)


def adamw_step(theta, grad, m1, m2, step: int, lr: float, beta1: float, beta2: float, eps: float,
               weight_decay: float):
    """One AdamW step (decoupled weight decay), step counted from 1:
        m1 <- beta1 m1 + (1 - beta1) g,     m2 <- beta2 m2 + (1 - beta2) g^2
        mhat = m1 / (1 - beta1^step),        vhat = m2 / (1 - beta2^step)
        theta <- theta - lr (mhat / (sqrt(vhat) + eps) + weight_decay theta)
    Returns (theta, m1, m2) as new float64 arrays."""
    th = np.asarray(theta, dtype=np.float64)
    g = np.asarray(grad, dtype=np.float64)
    m1 = beta1 * np.asarray(m1, dtype=np.float64) + (1.0 - beta1) * g
    m2 = beta2 * np.asarray(m2, dtype=np.float64) + (1.0 - beta2) * g * g
    mhat = m1 / (1.0 - beta1 ** step)
    vhat = m2 / (1.0 - beta2 ** step)
    th = th - lr * (mhat / (np.sqrt(vhat) + eps) + weight_decay * th)
    return th, m1, m2
