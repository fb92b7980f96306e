"""Programmatic dependent launch of the pass kernels (needs a B300).

With dependent launch on, each forward, backward and optimizer kernel may
start while the kernel before it on the stream drains, and waits for that
kernel's completion before its first global-memory access.  A missing or
misplaced wait would let a kernel read its input before the producer has
written it.  Checked here on a chain of three layers (layer i's output is
layer i+1's input, and the backward runs the chain in reverse, so every
kernel reads what the kernel right before it wrote), with every output
poisoned with NaN just before the step: eager on, eager off and a captured
CUDA graph with it on give bit-identical results, covering each family of
kernels that takes the wait (gathers, block transforms with and without the
fused reduction, both GEMM forms, every generator-backward variant, the fp32
path and AdamW).
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
    yield m
    m.poetx_set_dependent_launch(True)


def _chain(px, d, b, T, dtype, mode, depth=3):
    layers = []
    for i in range(depth):
        inp = make_inputs(d, d, b, b, T, dtype, index=20 + i, gstd=0.02)
        desc = px.make_desc(d, d, b, b, inp.seed_R, inp.seed_P, dtype=dtype, mode=mode)
        L = px.Layer(desc, T)
        L.build(inp.genR.cuda(), inp.genP.cuda())
        L.premerge(inp.W0.cuda())
        dt = L.dtype
        st = dict(L=L, genR=inp.genR.cuda(), genP=inp.genP.cuda(),
                  Y=torch.empty(T, d, dtype=dt, device="cuda"),
                  h=torch.empty(T, d, dtype=dt, device="cuda"),
                  u=torch.empty(T, d, dtype=dt, device="cuda"),
                  dX=torch.empty(T, d, dtype=dt, device="cuda"),
                  dgR=torch.empty(L.len_R, device="cuda"), dgP=torch.empty(L.len_P, device="cuda"))
        st["mom"] = [torch.zeros_like(st[k]) for k in ("genR", "genR", "genP", "genP")]
        layers.append(st)
    X0 = make_inputs(d, d, b, b, T, dtype, index=19).X.cuda()
    dY = make_inputs(d, d, b, b, T, dtype, index=18).dY.cuda()
    return layers, X0, dY


def _poison(layers):
    for st in layers:
        for k in ("Y", "h", "u", "dX", "dgR", "dgP"):
            st[k].fill_(float("nan"))


def _step(px, layers, X0, dY):
    _poison(layers)
    x = X0
    for st in layers:
        st["L"].rebuild(st["genR"], st["genP"])
        st["L"].forward(x, st["Y"], saved_h=st["h"], saved_u=st["u"])
        x = st["Y"]
    g = dY
    for i in reversed(range(len(layers))):
        st = layers[i]
        xin = X0 if i == 0 else layers[i - 1]["Y"]
        st["L"].backward(xin, g, st["dX"], st["dgR"], st["dgP"], saved_h=st["h"], saved_u=st["u"])
        mR, vR, mP, vP = st["mom"]
        px.poetx_generator_adamw(st["genR"], st["dgR"], mR, vR, st["L"].len_R, 1, 1e-3,
                                 0.9, 0.999, 1e-8, 0.0)
        px.poetx_generator_adamw(st["genP"], st["dgP"], mP, vP, st["L"].len_P, 1, 1e-3,
                                 0.9, 0.999, 1e-8, 0.0)
        g = st["dX"]


def _state(layers):
    return [st[k].clone() for st in layers for k in ("Y", "dX", "dgR", "dgP", "genR", "genP")]


def _restore(layers, gens):
    for st, (gR, gP) in zip(layers, gens):
        st["genR"].copy_(gR)
        st["genP"].copy_(gP)
        for t in st["mom"]:
            t.zero_()


@pytest.mark.parametrize("d,b,T,dtype,mode", [
    (512, 32, 1000, "bf16", "cayley"),     # narrow rows: pair-interleaved gather, b = 32 backward
    (1024, 64, 777, "bf16", "cayley"),
    (2048, 128, 600, "bf16", "cayley"),    # pipelined gather, fused reduction, cluster backward
    (512, 256, 300, "bf16", "cayley"),     # 256-wide fused reduction, fp32-grade GEMM backward
    (640, 128, 333, "bf16", "neumann"),    # tensor-core Neumann backward
    (256, 32, 512, "fp32", "cayley"),      # fp32 path
])
def test_dependent_launch_bit_identical(px, d, b, T, dtype, mode):
    layers, X0, dY = _chain(px, d, b, T, dtype, mode)
    gens = [(st["genR"].clone(), st["genP"].clone()) for st in layers]

    px.poetx_set_dependent_launch(False)
    _step(px, layers, X0, dY)
    torch.cuda.synchronize()
    ref = _state(layers)
    assert all(torch.isfinite(t).all() for t in ref)

    px.poetx_set_dependent_launch(True)
    _restore(layers, gens)
    _step(px, layers, X0, dY)
    torch.cuda.synchronize()
    for x, y in zip(ref, _state(layers)):
        assert torch.equal(x, y)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _restore(layers, gens)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            _step(px, layers, X0, dY)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(2):
        _restore(layers, gens)
        g.replay()
        torch.cuda.synchronize()
        for x, y in zip(ref, _state(layers)):
            assert torch.equal(x, y)
    assert px.poetx_device_status(reset=True) == px.POETX_OK
