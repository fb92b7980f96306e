"""CUDA-graph capture of a training step (needs a B300).

A step whose generators change but whose permutation seeds do not can be
captured once and replayed: poetx_blocks_build rebuilds the blocks with
device work only, and the forward and backward launch no host copies and
allocate nothing.  Checked here: blocks_build after params_build equals a
fresh params_build, and a captured (rebuild, forward, backward) replays to
bit-identical results of the eager calls, including after the generators
are overwritten in place between replays.
"""
import pytest
import torch

from tests.gpu_cases import make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def px():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import orthogonal_equivalence_reparameterized_poetx_b300 as m
    return m


def _setup(px, m, n, b, T, dtype="bf16", mode="cayley"):
    inp = make_inputs(m, n, b, b, T, dtype, index=8, gstd=0.02)
    desc = px.make_desc(m, n, b, b, inp.seed_R, inp.seed_P, dtype=dtype, mode=mode)
    layer = px.Layer(desc, T)
    layer.build(inp.genR.cuda(), inp.genP.cuda())
    layer.premerge(inp.W0.cuda())
    dt = layer.dtype
    bufs = dict(X=inp.X.cuda(), dY=inp.dY.cuda(), Y=torch.empty(T, m, dtype=dt, device="cuda"),
                h=torch.empty(T, m, dtype=dt, device="cuda"), u=torch.empty(T, n, dtype=dt, device="cuda"),
                dX=torch.empty(T, n, dtype=dt, device="cuda"),
                dgR=torch.empty(layer.len_R, device="cuda"), dgP=torch.empty(layer.len_P, device="cuda"))
    return inp, desc, layer, bufs


def _step(layer, genR, genP, B):
    layer.rebuild(genR, genP)
    layer.forward(B["X"], B["Y"], saved_h=B["h"], saved_u=B["u"])
    layer.backward(B["X"], B["dY"], B["dX"], B["dgR"], B["dgP"], saved_h=B["h"], saved_u=B["u"])


def _snapshot(B):
    return [B[k].clone() for k in ("Y", "dX", "dgR", "dgP")]


@pytest.mark.parametrize("b,mode", [(64, "cayley"), (256, "cayley"), (128, "neumann"), (256, "neumann")])
def test_blocks_build_equals_params_build(px, b, mode):
    m, n, T = 512, 384, 200
    inp, desc, layer, B = _setup(px, m, n, b, T, mode=mode)
    g2R, g2P = (inp.genR * 1.5).cuda(), (inp.genP * -0.5).cuda()
    _step(layer, g2R, g2P, B)
    torch.cuda.synchronize()
    a = _snapshot(B)
    fresh = px.Layer(desc, T)
    fresh.build(g2R, g2P)
    fresh.premerge(inp.W0.cuda())
    fresh.forward(B["X"], B["Y"], saved_h=B["h"], saved_u=B["u"])
    fresh.backward(B["X"], B["dY"], B["dX"], B["dgR"], B["dgP"], saved_h=B["h"], saved_u=B["u"])
    torch.cuda.synchronize()
    assert px.poetx_device_status(reset=True) == px.POETX_OK
    for x, y in zip(a, _snapshot(B)):
        assert torch.equal(x, y)


@pytest.mark.parametrize("m,n,b,mode", [
    (512, 1376, 32, "cayley"), (2048, 1024, 128, "cayley"),
    (768, 512, 512, "cayley"),      # cluster Gauss-Jordan builder, ragged block
    (640, 384, 128, "neumann"),     # tensor-core Neumann builder and backward
    (512, 768, 256, "neumann"),     # tensor-core Neumann builder, batched backward
])
def test_captured_step_replays_bit_identically(px, m, n, b, mode):
    T = 1000
    inp, desc, layer, B = _setup(px, m, n, b, T, mode=mode)
    genR, genP = inp.genR.cuda().clone(), inp.genP.cuda().clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _step(layer, genR, genP, B)          # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager1 = _snapshot(B)

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _step(layer, genR, genP, B)
    for k in ("Y", "dX", "dgR", "dgP"):
        B[k].zero_()
    g.replay()
    torch.cuda.synchronize()
    for x, y in zip(eager1, _snapshot(B)):
        assert torch.equal(x, y)

    # new generators written into the captured tensors: the replay rebuilds
    genR.mul_(0.5)
    genP.mul_(2.0)
    g.replay()
    torch.cuda.synchronize()
    replayed = _snapshot(B)
    _step(layer, genR, genP, B)
    torch.cuda.synchronize()
    assert px.poetx_device_status(reset=True) == px.POETX_OK
    for x, y in zip(replayed, _snapshot(B)):
        assert torch.equal(x, y)
    assert not torch.equal(replayed[2], eager1[2])   # the gradients did change
