"""POET-XQ: int8 base weights, dequantized on the fly (needs a B300).

"POET-X: Memory-efficient LLM Training by Scaling Orthogonal Transformation",
Methodologie §5, stores the base weights quantized (e.g. INT8) and
dequantizes them on the fly.  The scheme is a reading (symmetric per-row
absmax, scale = max|row| / 127, round half to even, float32), implemented by
the oracle's ``quantize_rows_int8``.  Checked here:

* the pre-merge writes exactly the oracle's codes and scales (the integer
  decisions are taken in float32 on both sides);
* forward and backward of an int8 layer match the oracle computing with the
  dequantized weight (scale * code) within the bf16 tolerance;
* the merge re-quantizes the fp32-grade merged weight: every dequantized
  element lies within half a quantization step of the fp64 merge of the
  dequantized weight, and the merged layer computes the same map;
* one full-size linear of the d = 2048 block.
"""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from tests.gpu_cases import make_inputs, rel_fro

pytestmark = pytest.mark.gpu

TOL = 2e-2


@pytest.fixture(scope="module")
def px():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import orthogonal_equivalence_reparameterized_poetx_b300 as m
    return m


def _split(buf, m, n):
    """(codes m x n int8, scales m float32) of an int8 weight buffer."""
    raw = buf.cpu().numpy()
    cb = (m * n + 255) // 256 * 256
    return raw[:m * n].view(np.int8).reshape(m, n), raw[cb:cb + 4 * m].view(np.float32)


def _original_basis(Wp, piR, piP):
    """W0 with W0[pi_R(i)][pi_P(j)] = Wp[i][j] (inverse of the pre-merge)."""
    W = np.zeros_like(Wp)
    W[np.ix_(piR, piP)] = Wp
    return W


def _layer(px, m, n, b, T, index, gstd=0.01, tokens=None, mode="cayley"):
    inp = make_inputs(m, n, b, b, T, "bf16", index=index, gstd=gstd)
    desc = px.make_desc(m, n, b, b, inp.seed_R, inp.seed_P, dtype="bf16", weight="int8", mode=mode)
    layer = px.Layer(desc, T)
    layer.build(inp.genR.cuda(), inp.genP.cuda())
    layer.premerge(inp.W0.cuda())
    return inp, desc, layer


@pytest.mark.parametrize("m,n,b", [(384, 256, 32), (1376, 512, 32), (256, 2816, 64)])
def test_premerge_quantizes_exactly_like_the_oracle(px, m, n, b):
    inp, desc, layer = _layer(px, m, n, b, 1, index=2)
    torch.cuda.synchronize()
    assert px.poetx_device_status(reset=True) == px.POETX_OK
    codes, scales = _split(layer.W0p, m, n)
    piR, piP = O.permutation(inp.seed_R, m), O.permutation(inp.seed_P, n)
    want_c, want_s = O.quantize_rows_int8(O.premerged_weight(inp.W0.double().numpy(), piR, piP))
    assert np.array_equal(scales, want_s)
    assert np.array_equal(codes, want_c)


@pytest.mark.parametrize("m,n,b,T,recompute,mode", [
    (512, 384, 128, 300, False, "cayley"),
    (1376, 1032, 64, 777, True, "cayley"),    # CTA-pair GEMMs, ragged tiles and blocks
    (640, 384, 128, 300, False, "neumann"),   # int8 weights with Neumann blocks
])
def test_int8_layer_matches_the_oracle_on_the_dequantized_weight(px, m, n, b, T, recompute, mode):
    inp, desc, layer = _layer(px, m, n, b, T, index=4, mode=mode)
    X, dY = inp.X.cuda(), inp.dY.cuda()
    Y = torch.empty(T, m, dtype=torch.bfloat16, device="cuda")
    h = None if recompute else torch.empty(T, m, dtype=torch.bfloat16, device="cuda")
    u = None if recompute else torch.empty(T, n, dtype=torch.bfloat16, device="cuda")
    layer.forward(X, Y, saved_h=h, saved_u=u)
    dX = torch.empty(T, n, dtype=torch.bfloat16, device="cuda")
    dgR = torch.empty(layer.len_R, device="cuda")
    dgP = torch.empty(layer.len_P, device="cuda")
    layer.backward(X, dY, dX, dgR, dgP, saved_h=h, saved_u=u)
    torch.cuda.synchronize()
    assert px.poetx_device_status(reset=True) == px.POETX_OK
    codes, scales = _split(layer.W0p, m, n)
    piR, piP = O.permutation(inp.seed_R, m), O.permutation(inp.seed_P, n)
    W0q = _original_basis(O.dequantize_rows_int8(codes, scales), piR, piP)
    spec = O.LayerSpec(m, n, b, b, inp.seed_R, inp.seed_P, "neumann" if mode == "neumann" else "exact", 3)
    dX_o, dgR_o, dgP_o, ex = O.backward(spec, W0q, inp.X.double().numpy(), inp.dY.double().numpy(),
                                        inp.genR.double().numpy(), inp.genP.double().numpy())
    errs = {"Y": rel_fro(Y.double().cpu().numpy(), ex["Y"]),
            "dX": rel_fro(dX.double().cpu().numpy(), dX_o),
            "dgR": rel_fro(dgR.double().cpu().numpy(), dgR_o),
            "dgP": rel_fro(dgP.double().cpu().numpy(), dgP_o)}
    assert all(e <= TOL for e in errs.values()), errs


@pytest.mark.parametrize("m,n,b", [(384, 256, 64), (640, 512, 256)])
def test_int8_merge_requantizes_within_half_a_step(px, m, n, b):
    T = 200
    inp, desc, layer = _layer(px, m, n, b, T, index=6, gstd=0.05)
    X = inp.X.cuda()
    Y_old = torch.empty(T, m, dtype=torch.bfloat16, device="cuda")
    layer.forward(X, Y_old)
    torch.cuda.synchronize()
    codes0, scales0 = _split(layer.W0p, m, n)
    new_R, new_P = 8505, 9506
    layer.merge(new_R, new_P)
    torch.cuda.synchronize()
    assert px.poetx_device_status(reset=True) == px.POETX_OK
    codes1, scales1 = _split(layer.W0p, m, n)

    piR, piP = O.permutation(inp.seed_R, m), O.permutation(inp.seed_P, n)
    W0q = _original_basis(O.dequantize_rows_int8(codes0, scales0), piR, piP)
    spec = O.LayerSpec(m, n, b, b, inp.seed_R, inp.seed_P)
    K = O.merge(spec, W0q, inp.genR.double().numpy(), inp.genP.double().numpy(), new_R, new_P)
    amax = np.abs(K).max(axis=1)
    assert np.allclose(scales1, amax / 127.0, rtol=1e-4, atol=0)
    err = np.abs(O.dequantize_rows_int8(codes1, scales1) - K)
    assert np.all(err <= scales1[:, None] * (0.5 + 5e-3) + 1e-9)

    # the merged layer (zero generators, new seeds) computes the same map
    d2 = px.make_desc(m, n, b, b, new_R, new_P, dtype="bf16", weight="int8")
    l2 = px.Layer(d2, T)
    l2.build(torch.zeros_like(inp.genR).cuda(), torch.zeros_like(inp.genP).cuda())
    l2.W0p.copy_(layer.W0p)
    Y_new = torch.empty(T, m, dtype=torch.bfloat16, device="cuda")
    l2.forward(X, Y_new)
    torch.cuda.synchronize()
    assert rel_fro(Y_new.double().cpu().numpy(), Y_old.double().cpu().numpy()) <= TOL


def test_int8_full_size_gate_linear(px):
    """d = 2048 block, gate 2048 -> 5632, b = 128, 65536 tokens with h and u
    saved: sampled rows of Y and dX against the oracle, generator gradients on
    the first 2048 tokens."""
    wl = synth.WORKLOADS["d2048_block"]
    li, b = 4, 128
    lin = wl.linears[li]
    T, m, n = wl.tokens, lin.m, lin.n
    lr, lp = O.packed_length(m, b), O.packed_length(n, b)
    inp = synth.layer_inputs(lin, li, T, "bf16", lr, lp)
    desc = px.make_desc(m, n, b, b, inp.seed_R, inp.seed_P, dtype="bf16", weight="int8")
    layer = px.Layer(desc, T)
    layer.build(inp.genR.cuda(), inp.genP.cuda())
    layer.premerge(inp.W0.cuda())
    X, dY = inp.X.cuda(), inp.dY.cuda()

    def run(Tn, want_out):
        Y = torch.empty(Tn, m, dtype=torch.bfloat16, device="cuda")
        h = torch.empty(Tn, m, dtype=torch.bfloat16, device="cuda")
        u = torch.empty(Tn, n, dtype=torch.bfloat16, device="cuda")
        dX = torch.empty(Tn, n, dtype=torch.bfloat16, device="cuda") if want_out else None
        dgR, dgP = torch.empty(lr, device="cuda"), torch.empty(lp, device="cuda")
        layer.forward(X[:Tn], Y, saved_h=h, saved_u=u)
        layer.backward(X[:Tn], dY[:Tn], dX, dgR, dgP, saved_h=h, saved_u=u)
        torch.cuda.synchronize()
        assert px.poetx_device_status(reset=True) == px.POETX_OK
        return Y, dX, dgR, dgP

    Y, dX, _, _ = run(T, True)
    codes, scales = _split(layer.W0p, m, n)
    piR, piP = O.permutation(inp.seed_R, m), O.permutation(inp.seed_P, n)
    W0q = _original_basis(O.dequantize_rows_int8(codes, scales), piR, piP)
    spec = O.LayerSpec(m, n, b, b, inp.seed_R, inp.seed_P)
    gR, gP = inp.genR.double().numpy(), inp.genP.double().numpy()
    rows = np.unique(np.concatenate([[0, 1, 255, 256, T // 2, T - 1],
                                     np.random.default_rng(3).integers(0, T, 10)]))
    dX_o, _, _, ex = O.backward(spec, W0q, inp.X[rows].double().numpy(),
                                inp.dY[rows].double().numpy(), gR, gP)
    assert rel_fro(Y[rows].double().cpu().numpy(), ex["Y"]) <= TOL
    assert rel_fro(dX[rows].double().cpu().numpy(), dX_o) <= TOL
    Ts = 2048
    _, _, sR, sP = run(Ts, False)
    _, dgR_o, dgP_o, _ = O.backward(spec, W0q, inp.X[:Ts].double().numpy(),
                                    inp.dY[:Ts].double().numpy(), gR, gP)
    assert rel_fro(sR.double().cpu().numpy(), dgR_o) <= TOL
    assert rel_fro(sP.double().cpu().numpy(), dgP_o) <= TOL
