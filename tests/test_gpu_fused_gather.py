"""The column permutation fused into the block transform (needs a B300).

With poetx_set_fused_gather_max_features(1536) (off by default), for bf16
sides with 128-wide super-blocks and 256 to 1536 features, the forward
gathers X -> u inside the P-side transform (one kernel writes u and v) and
the backward gathers dY -> dz inside the R-side transform + token
reduction.  Each case checks the fused form against the fp64 oracle (the
usual bf16 bound, also per row and per block, and the saved u bit for bit
against X[:, pi_P]) and against the separate gather passes (the default,
poetx_set_fused_gather_max_features(0)): both forms round the same products
in the same order, so every output must be bit-identical.

Cases: ragged token tails, a ragged last super-block (1376 = 10 * 128 + 96
features), b = 32, 64, 128, recompute mode (the backward regathers u with
the fused kernel), a single token (most CTAs own no token tile), the width
bound itself, and a token count with many tiles per CTA.
"""
import numpy as np
import pytest
import torch

import oracle as O
from tests.gpu_cases import make_inputs, parity_errors, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2


@pytest.fixture(scope="module")
def px():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import orthogonal_equivalence_reparameterized_poetx_b300 as m
    yield m
    m.poetx_set_fused_gather_max_features(-1)


@pytest.mark.parametrize("m,n,b,T,recompute,save_u", [
    (512, 512, 32, 1000, False, True),      # LLaMA-60M attention shape, ragged tokens
    (1376, 512, 32, 777, False, False),     # R side 1376 wide: ragged last super-block
    (512, 1376, 32, 300, True, False),      # P side 1376 wide, recompute: u and v regathered
    (1024, 1024, 64, 4097, True, True),     # b = 64, 33 token tiles
    (640, 384, 128, 1, False, False),       # one token: CTAs without a token tile
    (256, 1536, 128, 129, False, True),     # the width bound itself
    (512, 512, 32, 40000, False, True),     # many token tiles per CTA, the staging ring reused
])
def test_fused_gather_matches_oracle_and_separate_passes(px, m, n, b, T, recompute, save_u):
    inp = make_inputs(m, n, b, b, T, "bf16", index=31, gstd=0.01)
    desc = px.make_desc(m, n, b, b, inp.seed_R, inp.seed_P, dtype="bf16")
    spec = O.LayerSpec(m, n, b, b, inp.seed_R, inp.seed_P, "exact", 3)

    px.poetx_set_fused_gather_max_features(1536)
    try:
        g = run_gpu(px, desc, inp, recompute, save_u=save_u)
    finally:
        px.poetx_set_fused_gather_max_features(-1)
    if T <= 4097:
        o = run_oracle(spec, inp)
        errs = parity_errors(g, o, m, n, b, b)
        for k, e in errs.items():
            assert e <= TOL_BF16, f"{k}: rel Frobenius {e:.3e} > {TOL_BF16:.0e} ({errs})"
    if save_u:
        u_o = inp.X.double().numpy()[:, O.permutation(inp.seed_P, n)]
        assert np.array_equal(g["u"], u_o), "saved u must be the permuted input, bit for bit"

    px.poetx_set_fused_gather_max_features(0)
    s = run_gpu(px, desc, inp, recompute, save_u=save_u)
    for k in ("Y", "dX", "dgR", "dgP", "u"):
        if g[k] is None:
            continue
        assert np.array_equal(g[k], s[k]), f"{k} differs between the fused and separate gathers"
