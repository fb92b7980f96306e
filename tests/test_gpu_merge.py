"""GPU parity of the merge W0 <- R W0 P and of the weight pre-merge (needs a B300).

The merge folds the current orthogonal factors into the base weight and
re-expresses it under fresh permutations ("POET-X: Memory-efficient LLM
Training by Scaling Orthogonal Transformation", Methodologie §1, the update
W <- R_i W P_i).  Checked against the oracle's dense R W0 P, re-based under
the new permutations, and by the invariance that defines it: with the
generators reset to zero and the new seeds, the merged layer computes the
same Y as the layer before the merge.
"""
import numpy as np
import pytest
import torch

import oracle as O
from tests.gpu_cases import make_inputs, rel_fro

pytestmark = pytest.mark.gpu

TOL = {"fp32": 1e-5, "bf16": 2e-2}


@pytest.fixture(scope="module")
def px():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import orthogonal_equivalence_reparameterized_poetx_b300 as m
    return m


@pytest.mark.parametrize("dtype,m,n,bR,bP,mode", [
    ("fp32", 128, 96, 32, 32, "cayley"),
    ("fp32", 200, 136, 64, 48, "cayley"),      # ragged blocks on both sides
    ("bf16", 384, 256, 64, 64, "cayley"),
    ("bf16", 768, 512, 512, 256, "cayley"),    # cluster builders, ragged R block
    ("bf16", 256, 256, 128, 128, "neumann"),
])
def test_merge_matches_oracle_and_preserves_the_map(px, dtype, m, n, bR, bP, mode):
    T = 200
    inp = make_inputs(m, n, bR, bP, T, dtype, index=5, gstd=0.05)
    desc = px.make_desc(m, n, bR, bP, inp.seed_R, inp.seed_P, dtype=dtype, mode=mode)
    layer = px.Layer(desc, T)
    layer.build(inp.genR.cuda(), inp.genP.cuda())
    layer.premerge(inp.W0.cuda())
    X = inp.X.cuda()
    Y_old = torch.empty(T, m, dtype=layer.dtype, device="cuda")
    layer.forward(X, Y_old)
    new_R, new_P = 8101, 9102
    layer.merge(new_R, new_P)
    torch.cuda.synchronize()
    W0p_new = layer.W0p.double().cpu().numpy()

    spec = O.LayerSpec(m, n, bR, bP, inp.seed_R, inp.seed_P,
                       "neumann" if mode == "neumann" else "exact", 3)
    want = O.merge(spec, inp.W0.double().numpy(), inp.genR.double().numpy(),
                   inp.genP.double().numpy(), new_R, new_P)
    assert rel_fro(W0p_new, want) <= TOL[dtype]

    # the merged layer with zero generators under the new seeds computes the same map
    d2 = px.make_desc(m, n, bR, bP, new_R, new_P, dtype=dtype, mode=mode)
    l2 = px.Layer(d2, T)
    l2.build(torch.zeros_like(inp.genR).cuda(), torch.zeros_like(inp.genP).cuda())
    l2.W0p.copy_(layer.W0p)
    Y_new = torch.empty(T, m, dtype=layer.dtype, device="cuda")
    l2.forward(X, Y_new)
    torch.cuda.synchronize()
    assert px.poetx_device_status(reset=True) == px.POETX_OK
    assert rel_fro(Y_new.double().cpu().numpy(), Y_old.double().cpu().numpy()) <= TOL[dtype]


def test_premerge_is_an_exact_permutation_copy(px):
    m, n = 1376, 512
    inp = make_inputs(m, n, 32, 32, 1, "bf16", index=6)
    desc = px.make_desc(m, n, 32, 32, inp.seed_R, inp.seed_P, dtype="bf16")
    layer = px.Layer(desc, 1)
    layer.build(inp.genR.cuda(), inp.genP.cuda())
    layer.premerge(inp.W0.cuda())
    torch.cuda.synchronize()
    piR, piP = O.permutation(inp.seed_R, m), O.permutation(inp.seed_P, n)
    want = inp.W0.float().numpy()[piR][:, piP]
    assert np.array_equal(layer.W0p.float().cpu().numpy(), want)


@pytest.mark.parametrize("m,n,b,mode,k", [
    (384, 256, 32, "cayley", 3), (512, 640, 128, "cayley", 3), (768, 512, 256, "cayley", 3),
    (768, 512, 512, "cayley", 3),
    # Neumann blocks built by the fused tensor-core builder: B itself must be
    # fp32-grade for the merged weight to stay within half an ulp
    (512, 640, 128, "neumann", 3), (768, 512, 256, "neumann", 2), (768, 512, 512, "neumann", 3),
    (512, 384, 256, "neumann", 6),
])
def test_bf16_merge_is_rounded_once_from_a_near_exact_product(px, m, n, b, mode, k):
    """The bf16 merge runs on the tensor cores with bf16 operands, splitting
    B - I and the intermediate into hi + lo bf16 pairs; the result must still
    be the exact R W0 P (re-based) rounded once to bf16: every element within
    half a bf16 ulp of the fp64 oracle's value, plus slack at the fp32 level
    (the blocks themselves are built to fp32 accuracy)."""
    # Neumann blocks with the workloads' generator scale (||Q|| < 1, where the
    # series is a good orthogonal approximation); Cayley blocks larger
    gstd = 0.01 if mode == "neumann" else 0.05
    inp = make_inputs(m, n, b, b, 1, "bf16", index=7, gstd=gstd)
    desc = px.make_desc(m, n, b, b, inp.seed_R, inp.seed_P, dtype="bf16", mode=mode, neumann_k=k)
    layer = px.Layer(desc, 1)
    layer.build(inp.genR.cuda(), inp.genP.cuda())
    layer.premerge(inp.W0.cuda())
    new_R, new_P = 8303, 9304
    layer.merge(new_R, new_P)
    torch.cuda.synchronize()
    assert px.poetx_device_status(reset=True) == px.POETX_OK
    got = layer.W0p.double().cpu().numpy()
    spec = O.LayerSpec(m, n, b, b, inp.seed_R, inp.seed_P,
                       "neumann" if mode == "neumann" else "exact", k)
    want = O.merge(spec, inp.W0.double().numpy(), inp.genR.double().numpy(),
                   inp.genP.double().numpy(), new_R, new_P)
    a = np.abs(want)
    tiny = np.finfo(np.float64).tiny
    half_ulp = 2.0 ** (np.floor(np.log2(np.maximum(a, tiny))) - 8)   # bf16: 8 significant bits
    slack = 2e-5 * a + 1e-5 * a.max()
    err = np.abs(got - want)
    bad = err > half_ulp + slack
    assert not bad.any(), (f"{bad.sum()} elements beyond half an ulp; worst excess "
                           f"{(err - half_ulp - slack).max():.3e}")
