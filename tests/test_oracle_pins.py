"""Pins of the fp64 oracle against facts fixed outside it (CPU only).

Each check compares the oracle with something it does not compute itself:
known-answer values of the permutation generator, hand-derived closed forms
of the Cayley map, library routines (numpy solve/svd), invariants the pages
state (orthogonality, spectrum invariance), the dense product, and central
finite differences.  The mutation tests at the end plant plausible mistakes
in copies of the oracle and confirm that one of these pins fails.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle as O
from tests.conftest import read_golden


def _frac(s):
    return float(Fraction(s))


def _rng(seed):
    return np.random.default_rng(seed)


def _spec(m, n, bR, bP, mode="exact", k=3, sR=11, sP=12):
    return O.LayerSpec(m=m, n=n, b_R=bR, b_P=bP, seed_R=sR, seed_P=sP, mode=mode, neumann_k=k)


def _rand_layer(spec, T, seed=0, gstd=0.05):
    r = _rng(seed)
    W0 = r.standard_normal((spec.m, spec.n)) * 0.3
    X = r.standard_normal((T, spec.n))
    dY = r.standard_normal((T, spec.m))
    gR = r.standard_normal(O.packed_length(spec.m, spec.b_R)) * gstd
    gP = r.standard_normal(O.packed_length(spec.n, spec.b_P)) * gstd
    return W0, X, dY, gR, gP


# ---------------------------------------------------------------- permutations

def test_splitmix64_known_answers():
    want = [int(r[0], 16) for r in read_golden("splitmix64_seed0.txt")]
    g = O.splitmix64(0)
    assert [next(g) for _ in range(len(want))] == want


@pytest.mark.parametrize("d", [4, 5])
def test_permutation_hand_derived_seed0(d):
    want = [int(x) for x in read_golden(f"perm_seed0_d{d}.txt")[0]]
    assert O.permutation(0, d).tolist() == want


def test_bounded_draw_rejects_top_bucket():
    # 2^64 mod 3 == 1, so 2^64-1 lies in the partial top bucket and is redrawn.
    def fake():
        yield (1 << 64) - 1
        yield 5
    assert O.bounded_draw(fake(), 3) == 2
    def fake2():
        yield (1 << 64) - 2     # below the limit: accepted, (2^64-2) mod 3 == 2
    assert O.bounded_draw(fake2(), 3) == ((1 << 64) - 2) % 3


@pytest.mark.parametrize("d", [1, 2, 3, 17, 256, 1376, 11008])
def test_permutation_is_bijection(d):
    p = O.permutation(1234 + d, d)
    assert sorted(p.tolist()) == list(range(d))
    inv = O.inverse_permutation(p)
    assert np.array_equal(p[inv], np.arange(d))


def test_permutation_uniform_brute_force():
    # All 24 permutations of 4 items, over 9600 seeds: chi-square with 23 dof.
    from collections import Counter
    cnt = Counter(tuple(O.permutation(s, 4).tolist()) for s in range(9600))
    assert len(cnt) == 24
    exp = 9600 / 24
    chi2 = sum((c - exp) ** 2 / exp for c in cnt.values())
    assert chi2 < 60.0      # p ~ 4e-5 under uniformity


def test_perm_matrix_gather_convention():
    p = np.array([2, 0, 1])
    x = np.array([10.0, 20.0, 30.0])
    assert (O.perm_matrix(p) @ x).tolist() == [30.0, 10.0, 20.0]


# ---------------------------------------------------------------- generators

def test_packing_order_and_ragged_blocks():
    assert O.block_sizes(11008, 512) == [512] * 21 + [256]
    assert O.block_sizes(1376, 32) == [32] * 43
    assert O.block_sizes(7, 4) == [4, 3]
    assert O.packed_length(7, 4) == 6 + 3
    Q = O.unpack_skew(np.array([1.0, 2.0, 3.0, 4.0, 5.0, 6.0]), 4)
    # row-major strict upper: (0,1)(0,2)(0,3)(1,2)(1,3)(2,3)
    assert Q[0, 1] == 1 and Q[0, 3] == 3 and Q[1, 2] == 4 and Q[2, 3] == 6
    assert np.array_equal(Q, -Q.T)
    # pack_antisym is the adjoint of unpack_skew: <G, unpack(p)> = <pack(G), p>
    r = _rng(3)
    G = r.standard_normal((4, 4))
    p = r.standard_normal(6)
    assert np.isclose(np.sum(G * O.unpack_skew(p, 4)), O.pack_antisym(G) @ p, rtol=1e-14)


# ---------------------------------------------------------------- Cayley / Neumann

def test_cayley_2x2_closed_form():
    for row in read_golden("cayley_2x2.txt"):
        s = _frac(row[0])
        want = np.array([_frac(x) for x in row[1:]]).reshape(2, 2)
        B, _ = O.cayley(np.array([[0.0, s], [-s, 0.0]]))
        assert np.abs(B - want).max() < 1e-15


def test_cayley_3x3_closed_form_pins_packing_sign_and_side():
    rows = read_golden("cayley_3x3.txt")
    packed = np.array([float(x) for x in rows[0][1:]])
    want = np.array([[_frac(x) for x in r] for r in rows[1:]])
    (Q, B, M), = O.blocks_of(packed, 3, 3, "exact", 3)
    assert np.abs(B - want).max() < 1e-15


@pytest.mark.parametrize("s", [1, 2, 7, 32, 64, 128])
def test_cayley_orthogonal_and_identities(s):
    r = _rng(s)
    Q = O.unpack_skew(r.standard_normal(s * (s - 1) // 2) * 0.05, s)
    B, M = O.cayley(Q)
    I = np.eye(s)
    assert np.abs(B.T @ B - I).max() <= 1e-12
    assert np.abs(B @ B.T - I).max() <= 1e-12
    assert np.abs(B - (2 * M - I)).max() <= 1e-12
    # library cross-check: B (I-Q) = I+Q solved by LAPACK
    B_lapack = np.linalg.solve((I - Q).T, (I + Q).T).T
    assert np.abs(B - B_lapack).max() <= 1e-12


def test_gauss_jordan_matches_lapack_with_pivoting():
    r = _rng(5)
    A = r.standard_normal((9, 9))
    A[0, 0] = 0.0      # forces a row exchange
    assert np.abs(O.inverse_gauss_jordan(A) - np.linalg.inv(A)).max() < 1e-10


def test_neumann_expanded_polynomial_and_residual():
    r = _rng(7)
    s = 16
    Q = O.unpack_skew(r.standard_normal(s * (s - 1) // 2) * 0.1, s)
    I = np.eye(s)
    Q2, Q3 = Q @ Q, Q @ Q @ Q
    Q4 = Q2 @ Q2
    assert np.abs(O.neumann(Q, 3) - (I + 2 * Q + 2 * Q2 + 2 * Q3 + Q4)).max() < 1e-14
    for k in (1, 2, 3, 5):
        B, M = O.cayley(Q)
        resid = (I + Q) @ np.linalg.matrix_power(Q, k + 1) @ M
        assert np.abs((B - O.neumann(Q, k)) - resid).max() < 1e-13
    assert np.array_equal(O.neumann(np.zeros((5, 5)), 3), np.eye(5))


# ---------------------------------------------------------------- forward

LAYERS = [
    _spec(16, 16, 4, 4), _spec(12, 20, 4, 8), _spec(7, 9, 4, 4),
    _spec(24, 24, 24, 24), _spec(10, 10, 3, 5, mode="neumann"),
]


@pytest.mark.parametrize("spec", LAYERS)
def test_input_centric_equals_dense(spec):
    W0, X, dY, gR, gP = _rand_layer(spec, 5)
    Yd = O.forward_dense(spec, W0, X, gR, gP)
    Yi, _ = O.forward_input_centric(spec, W0, X, gR, gP)
    assert np.abs(Yd - Yi).max() <= 1e-12 * max(1.0, np.abs(Yd).max())


def test_premerged_weight_matches_permutation_matrices():
    r = _rng(9)
    W0 = r.standard_normal((6, 5))
    piR, piP = O.permutation(1, 6), O.permutation(2, 5)
    want = O.perm_matrix(piR) @ W0 @ O.perm_matrix(piP).T
    assert np.array_equal(O.premerged_weight(W0, piR, piP), want)


@pytest.mark.parametrize("spec", [_spec(32, 24, 8, 6), _spec(40, 40, 16, 16)])
def test_spectrum_invariance(spec):
    W0, X, dY, gR, gP = _rand_layer(spec, 1, gstd=0.3)
    W = O.dense_weight(spec, W0, gR, gP)
    sv = np.linalg.svd(W, compute_uv=False)
    sv0 = np.linalg.svd(W0, compute_uv=False)
    assert np.allclose(sv, sv0, rtol=1e-10, atol=0)
    assert not np.allclose(W, W0, atol=1e-3)


def test_zero_generators_identity_perms_is_plain_gemm():
    spec = _spec(12, 8, 4, 4)
    W0, X, dY, gR, gP = _rand_layer(spec, 6)
    Y, _ = O.forward_input_centric(spec, W0, X, np.zeros_like(gR), np.zeros_like(gP),
                                   piR=np.arange(12), piP=np.arange(8))
    assert np.abs(Y - X @ W0.T).max() < 1e-13


def test_block_size_one_is_plain_gemm_under_any_perms():
    spec = _spec(9, 7, 1, 1)
    W0, X, dY, gR, gP = _rand_layer(spec, 4)
    assert len(gR) == 0 and len(gP) == 0
    Y, _ = O.forward_input_centric(spec, W0, X, gR, gP)
    assert np.abs(Y - X @ W0.T).max() < 1e-13


def test_norm_preservation_with_orthogonal_base():
    spec = _spec(16, 16, 4, 8)
    r = _rng(11)
    W0, _ = np.linalg.qr(r.standard_normal((16, 16)))
    _, X, _, gR, gP = _rand_layer(spec, 7, gstd=0.5)
    Y, _ = O.forward_input_centric(spec, W0, X, gR, gP)
    assert np.isclose(np.linalg.norm(Y), np.linalg.norm(X), rtol=1e-12)


# ---------------------------------------------------------------- backward

def _fd_grad(spec, W0, X, dY, gR, gP, which, h=1e-6):
    g = gR if which == "R" else gP
    out = np.zeros_like(g)
    for i in range(len(g)):
        gp, gm = g.copy(), g.copy()
        gp[i] += h
        gm[i] -= h
        if which == "R":
            lp = O.loss_for_fd(spec, W0, X, dY, gp, gP)
            lm = O.loss_for_fd(spec, W0, X, dY, gm, gP)
        else:
            lp = O.loss_for_fd(spec, W0, X, dY, gR, gp)
            lm = O.loss_for_fd(spec, W0, X, dY, gR, gm)
        out[i] = (lp - lm) / (2 * h)
    return out


@pytest.mark.parametrize("spec", [
    _spec(8, 8, 4, 4), _spec(7, 9, 4, 4), _spec(8, 8, 4, 4, mode="neumann"),
    _spec(6, 10, 3, 5, mode="neumann", k=2), _spec(6, 6, 3, 3, mode="neumann", k=1),
    _spec(6, 6, 3, 3, mode="neumann", k=6)])
def test_generator_grad_matches_finite_differences(spec):
    W0, X, dY, gR, gP = _rand_layer(spec, 3, gstd=0.2)
    dX, dgR, dgP, _ = O.backward(spec, W0, X, dY, gR, gP)
    for which, ana in (("R", dgR), ("P", dgP)):
        fd = _fd_grad(spec, W0, X, dY, gR, gP, which)
        assert np.linalg.norm(ana - fd) <= 1e-7 * np.linalg.norm(fd)


@pytest.mark.parametrize("spec", LAYERS)
def test_dX_equals_dY_times_dense_weight(spec):
    W0, X, dY, gR, gP = _rand_layer(spec, 5)
    dX, _, _, _ = O.backward(spec, W0, X, dY, gR, gP)
    W = O.dense_weight(spec, W0, gR, gP)
    assert np.abs(dX - dY @ W).max() < 1e-12


def test_generator_grad_is_additive_over_token_shards():
    spec = _spec(12, 10, 4, 5)
    W0, X, dY, gR, gP = _rand_layer(spec, 8)
    _, a_R, a_P, _ = O.backward(spec, W0, X, dY, gR, gP)
    _, b_R, b_P, _ = O.backward(spec, W0, X[:3], dY[:3], gR, gP)
    _, c_R, c_P, _ = O.backward(spec, W0, X[3:], dY[3:], gR, gP)
    assert np.abs(a_R - (b_R + c_R)).max() < 1e-12
    assert np.abs(a_P - (b_P + c_P)).max() < 1e-12


# ---------------------------------------------------------------- merge

@pytest.mark.parametrize("spec", [_spec(12, 10, 4, 5), _spec(9, 9, 4, 4, mode="neumann")])
def test_merge_preserves_the_layer_map(spec):
    W0, X, dY, gR, gP = _rand_layer(spec, 6, gstd=0.3)
    Y_old = O.forward_dense(spec, W0, X, gR, gP)
    W0p_new = O.merge(spec, W0, gR, gP, 77, 78)
    spec_new = _spec(spec.m, spec.n, spec.b_R, spec.b_P, spec.mode, spec.neumann_k, 77, 78)
    piR, piP = O.permutation(77, spec.m), O.permutation(78, spec.n)
    # recover the un-premerged base weight from W0' = W0[piR][:, piP]
    W0_new = np.empty_like(W0p_new)
    W0_new[np.ix_(piR, piP)] = W0p_new
    Y_new = O.forward_dense(spec_new, W0_new, X, np.zeros_like(gR), np.zeros_like(gP))
    assert np.abs(Y_old - Y_new).max() < 1e-12


# ---------------------------------------------------------------- planted mistakes

# ------------------------------------------------------------------ POET-XQ int8 rows

def test_int8_quantization_golden_rows():
    rows = read_golden("quant_int8_rows.txt")
    ws = [np.array([float(x) for x in r[1:]]) for r in rows if r[0] == "w:"]
    qs = [np.array([int(x) for x in r[1:]]) for r in rows if r[0] == "q:"]
    W = np.stack(ws)
    codes, scales = O.quantize_rows_int8(W)
    assert codes.dtype == np.int8
    assert np.array_equal(codes.astype(np.int64), np.stack(qs))
    amax = np.abs(W.astype(np.float32)).max(axis=1)
    assert np.array_equal(scales, (amax / np.float32(127)).astype(np.float32))


def test_int8_quantization_properties():
    rng = np.random.default_rng(11)
    W = (rng.standard_normal((37, 53)) * 0.02).astype(np.float32)
    W[5] = 0.0                      # an all-zero row
    W[7, 3] = 0.5                   # a row dominated by one entry
    codes, scales = O.quantize_rows_int8(W)
    deq = O.dequantize_rows_int8(codes, scales)
    # within half a quantization step of the input (plus float32 round-off)
    err = np.abs(deq - W.astype(np.float64))
    assert np.all(err <= scales[:, None].astype(np.float64) * (0.5 + 1e-5) + 1e-12)
    # every nonzero row reaches the full code range at its largest entry
    nz = scales > 0
    assert np.all(np.abs(codes[nz]).max(axis=1) == 127)
    assert np.all(codes[~nz] == 0) and np.all(scales[~nz] == 0)
    assert np.all(np.abs(codes.astype(np.int64)) <= 127)
    # per-row: permuting rows permutes the result; permuting columns permutes codes
    pr, pc = rng.permutation(37), rng.permutation(53)
    c2, s2 = O.quantize_rows_int8(W[pr][:, pc])
    assert np.array_equal(c2, codes[pr][:, pc]) and np.array_equal(s2, scales[pr])


# ------------------------------------------------------------------ AdamW on the generators

def test_adamw_first_step_closed_form():
    # zero moments: mhat = g and vhat = g^2, so each entry moves by
    # -lr (g / (|g| + eps) + wd theta): about -lr sign(g) for |g| >> eps
    th = np.array([0.5, -0.25, 0.0, 1.0])
    g = np.array([2.0, -1e-3, 0.5, 0.0])
    lr, wd, eps = 0.1, 0.01, 1e-8
    t1, m1, m2 = O.adamw_step(th, g, np.zeros(4), np.zeros(4), 1, lr, 0.9, 0.999, eps, wd)
    want = th - lr * (g / (np.abs(g) + eps) + wd * th)
    assert np.allclose(t1, want, rtol=0, atol=1e-15)
    assert np.allclose(m1, 0.1 * g) and np.allclose(m2, 0.001 * g * g)


def test_adamw_matches_torch_optim_adamw_over_steps():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    th0 = rng.standard_normal(50) * 0.01
    grads = [rng.standard_normal(50) for _ in range(6)]
    hp = dict(lr=3e-3, betas=(0.9, 0.95), eps=1e-8, weight_decay=0.1)
    p = torch.nn.Parameter(torch.tensor(th0, dtype=torch.float64))
    opt = torch.optim.AdamW([p], **hp)
    th, m1, m2 = th0.copy(), np.zeros(50), np.zeros(50)
    for t, g in enumerate(grads, start=1):
        p.grad = torch.tensor(g, dtype=torch.float64)
        opt.step()
        th, m1, m2 = O.adamw_step(th, g, m1, m2, t, hp["lr"], *hp["betas"], hp["eps"],
                                  hp["weight_decay"])
    assert np.allclose(th, p.detach().numpy(), rtol=1e-12, atol=1e-15)


def _pins_fail(monkeypatch, name, replacement, checks):
    monkeypatch.setattr(O, name, replacement)
    failed = 0
    for chk in checks:
        try:
            chk()
        except AssertionError:
            failed += 1
    monkeypatch.undo()
    return failed


def test_planted_mistakes_are_caught(monkeypatch):
    orig_cayley, orig_neumann = O.cayley, O.neumann
    orig_unpack, orig_apply = O.unpack_skew, O._apply_blocks
    orig_ggrad = O._generator_grad
    orig_quant = O.quantize_rows_int8
    orig_adamw = O.adamw_step
    orig_perm = O.permutation

    def cayley_transposed(Q):
        B, M = orig_cayley(Q)
        return B.T, M.T

    def neumann_k_off_by_one(Q, k):
        return orig_neumann(Q, k + 1)

    def unpack_column_major(p, s):
        U = np.zeros((s, s))
        k = 0
        for j in range(s):
            for i in range(j):
                U[i, j] = p[k]
                k += 1
        return U - U.T

    def apply_blocks_untransposed(A, blocks, transpose):
        return orig_apply(A, blocks, not transpose)

    def ggrad_dropped_two(blocks, G, mode, k):
        return 0.5 * orig_ggrad(blocks, G, mode, k)

    def perm_reversed_loop(seed, d):
        p = list(range(d))
        g = O.splitmix64(seed)
        for i in range(1, d):
            j = O.bounded_draw(g, i + 1)
            p[i], p[j] = p[j], p[i]
        return np.array(p, dtype=np.int64)

    three = lambda: test_cayley_3x3_closed_form_pins_packing_sign_and_side()
    two = lambda: test_cayley_2x2_closed_form()
    poly = lambda: test_neumann_expanded_polynomial_and_residual()
    fd = lambda: test_generator_grad_matches_finite_differences(_spec(8, 8, 4, 4))
    fdn = lambda: test_generator_grad_matches_finite_differences(_spec(8, 8, 4, 4, mode="neumann"))
    dense = lambda: test_input_centric_equals_dense(_spec(12, 20, 4, 8))
    permk = lambda: test_permutation_hand_derived_seed0(5)

    assert _pins_fail(monkeypatch, "cayley", cayley_transposed, [three, two]) >= 1
    assert _pins_fail(monkeypatch, "neumann", neumann_k_off_by_one, [poly]) >= 1
    pack4 = lambda: test_packing_order_and_ragged_blocks()
    # (for s = 3 both orders coincide; the 4x4 packing pin separates them)
    assert _pins_fail(monkeypatch, "unpack_skew", unpack_column_major, [three, pack4]) >= 1
    assert _pins_fail(monkeypatch, "_apply_blocks", apply_blocks_untransposed, [dense, fd]) >= 1
    assert _pins_fail(monkeypatch, "_generator_grad", ggrad_dropped_two, [fd, fdn]) >= 1
    assert _pins_fail(monkeypatch, "permutation", perm_reversed_loop, [permk]) >= 1

    def quant_per_column(W):
        c, s_ = orig_quant(np.asarray(W).T)
        return c.T, s_
    def quant_over_128(W):
        W32 = np.asarray(W, dtype=np.float32)
        sc = (np.abs(W32).max(axis=1) / np.float32(128)).astype(np.float32)
        safe = np.where(sc > 0, sc, np.float32(1))
        return np.clip(np.rint(W32 / safe[:, None]), -127, 127).astype(np.int8), sc
    def quant_truncating(W):
        W32 = np.asarray(W, dtype=np.float32)
        sc = (np.abs(W32).max(axis=1) / np.float32(127)).astype(np.float32)
        safe = np.where(sc > 0, sc, np.float32(1))
        return np.clip(np.trunc(W32 / safe[:, None]), -127, 127).astype(np.int8), sc
    qgold = lambda: test_int8_quantization_golden_rows()
    for bad in (quant_per_column, quant_over_128, quant_truncating):
        assert _pins_fail(monkeypatch, "quantize_rows_int8", bad, [qgold]) >= 1

    def adamw_no_bias_correction(th, g, m1, m2, step, lr, b1, b2, eps, wd):
        m1 = b1 * np.asarray(m1) + (1 - b1) * np.asarray(g)
        m2 = b2 * np.asarray(m2) + (1 - b2) * np.asarray(g) ** 2
        return np.asarray(th) - lr * (m1 / (np.sqrt(m2) + eps) + wd * np.asarray(th)), m1, m2
    def adamw_coupled_decay(th, g, m1, m2, step, lr, b1, b2, eps, wd):
        return orig_adamw(th, np.asarray(g) + wd * np.asarray(th), m1, m2, step, lr, b1, b2, eps, 0.0)
    first = lambda: test_adamw_first_step_closed_form()
    vs_torch = lambda: test_adamw_matches_torch_optim_adamw_over_steps()
    for bad in (adamw_no_bias_correction, adamw_coupled_decay):
        assert _pins_fail(monkeypatch, "adamw_step", bad, [first, vs_torch]) >= 1
