"""Checkpoint and resume of a layer.

A layer's whole state is its descriptor (sizes, block sizes, permutation
seeds, mode, dtype, weight format), its packed fp32 generators and its
pre-merged base weight W0'.  The permutations and block matrices in `params`
are functions of the seeds and generators, so they are rebuilt on resume
rather than saved.  The state goes through torch.save / torch.load.

The CPU test checks the round trip of that state.  The GPU test runs a layer
through a merge under fresh seeds ("POET-X: Memory-efficient LLM Training by
Scaling Orthogonal Transformation", Methodologie §1, W <- R W P), continues it
with other generators, saves it, resumes it into new buffers, and requires
the resumed forward and backward to equal the original's bit for bit.
"""
import io

import pytest
import torch

from tests.gpu_cases import make_inputs

DESC_FIELDS = ("m", "n", "b_R", "b_P", "seed_R", "seed_P", "mode", "neumann_k", "dtype",
               "weight_format")


def save_state(desc, genR, genP, W0p) -> bytes:
    state = {f: int(getattr(desc, f)) for f in DESC_FIELDS}
    state.update(genR=genR.detach().cpu(), genP=genP.detach().cpu(), W0p=W0p.detach().cpu())
    buf = io.BytesIO()
    torch.save(state, buf)
    return buf.getvalue()


def load_state(px, blob: bytes):
    s = torch.load(io.BytesIO(blob))
    desc = px.poetx_layer_desc(*(s[f] for f in DESC_FIELDS))
    return desc, s["genR"], s["genP"], s["W0p"]


def test_state_round_trip_on_the_host():
    import orthogonal_equivalence_reparameterized_poetx_b300 as px
    desc = px.make_desc(416, 256, 64, 32, (1 << 64) - 5, 12345, dtype="bf16", mode="neumann",
                        neumann_k=6, weight="int8")
    g = torch.Generator().manual_seed(3)
    genR = torch.randn(px.poetx_gen_length(416, 64), generator=g)
    genP = torch.randn(px.poetx_gen_length(256, 32), generator=g)
    W0p = torch.randint(0, 256, (px.poetx_weight_size(desc),), dtype=torch.uint8, generator=g)
    d2, gR, gP, W = load_state(px, save_state(desc, genR, genP, W0p))
    assert all(getattr(d2, f) == getattr(desc, f) for f in DESC_FIELDS), (desc, d2)
    assert d2.seed_R == (1 << 64) - 5
    assert torch.equal(gR, genR) and torch.equal(gP, genP) and torch.equal(W, W0p)
    assert W.dtype == torch.uint8 and gR.dtype == torch.float32


@pytest.fixture(scope="module")
def px():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import orthogonal_equivalence_reparameterized_poetx_b300 as m
    return m


def _step(px, layer, X, dY):
    """Forward (recomputing h in the backward) and backward; CPU copies."""
    T = X.shape[0]
    Y = torch.empty(T, layer.desc.m, dtype=layer.dtype, device="cuda")
    dX = torch.empty(T, layer.desc.n, dtype=layer.dtype, device="cuda")
    dgR = torch.empty(layer.len_R, dtype=torch.float32, device="cuda")
    dgP = torch.empty(layer.len_P, dtype=torch.float32, device="cuda")
    layer.forward(X, Y)
    layer.backward(X, dY, dX, dgR, dgP)
    torch.cuda.synchronize()
    assert px.poetx_device_status(reset=True) == px.POETX_OK
    return [t.cpu() for t in (Y, dX, dgR, dgP)]


@pytest.mark.gpu
@pytest.mark.parametrize("m,n,b,mode,weight", [
    (384, 256, 64, "cayley", "dense"),
    (384, 256, 64, "cayley", "int8"),       # POET-XQ weight: codes and row scales
    (256, 256, 128, "neumann", "dense"),
])
def test_resumed_layer_equals_the_original_bit_for_bit(px, m, n, b, mode, weight):
    T = 300
    inp = make_inputs(m, n, b, b, T, "bf16", index=21, gstd=0.05)
    later = make_inputs(m, n, b, b, T, "bf16", index=22, gstd=0.05)
    desc = px.make_desc(m, n, b, b, inp.seed_R, inp.seed_P, dtype="bf16", mode=mode, weight=weight)
    layer = px.Layer(desc, T)
    layer.build(inp.genR.cuda(), inp.genP.cuda())
    layer.premerge(inp.W0.cuda())
    # fold R and P into W0' under fresh seeds, then continue with other generators
    layer.merge(8301, 9302)
    layer.desc.seed_R, layer.desc.seed_P = 8301, 9302
    genR, genP = later.genR.cuda(), later.genP.cuda()
    layer.build(genR, genP)
    X, dY = later.X.cuda(), later.dY.cuda()
    want = _step(px, layer, X, dY)

    d2, gR, gP, W0p = load_state(px, save_state(layer.desc, genR, genP, layer.W0p))
    resumed = px.Layer(d2, T)
    resumed.build(gR.cuda(), gP.cuda())
    resumed.W0p.copy_(W0p.cuda())
    got = _step(px, resumed, X, dY)
    for name, g_, w_ in zip(("Y", "dX", "dgR", "dgP"), got, want):
        assert torch.equal(g_, w_), name
