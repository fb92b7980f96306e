"""Independent linears on parallel streams (needs a B300).

A transformer block applies q, k and v (and gate and up) to the same input,
so their forward and backward calls can run on parallel streams, each with
its own workspace; the benchmark's step does so.  Every call keeps its
scratch in its own workspace and its state in its own params, so running
them concurrently must not change a bit: checked here against the same
calls run one after another on one stream, eagerly and from a captured CUDA
graph whose branches are the parallel streams, with every output poisoned
with NaN first.  The layers differ in shape and block size so that their
kernels (and grids) differ while they overlap.
"""
import pytest
import torch

from tests.gpu_cases import make_inputs

pytestmark = pytest.mark.gpu

SHAPES = [  # (m, n, b, T): share T so that the layers read one block input
    (512, 512, 32, 1000),
    (1376, 512, 32, 1000),
    (1024, 512, 128, 1000),
]


@pytest.fixture(scope="module")
def px():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import orthogonal_equivalence_reparameterized_poetx_b300 as m
    return m


def _layers(px, recompute):
    out = []
    X = make_inputs(512, 512, 32, 32, 1000, "bf16", index=40).X.cuda()
    for i, (m, n, b, T) in enumerate(SHAPES):
        inp = make_inputs(m, n, b, b, T, "bf16", index=41 + i, gstd=0.02)
        desc = px.make_desc(m, n, b, b, inp.seed_R, inp.seed_P, dtype="bf16")
        L = px.Layer(desc, T)
        L.build(inp.genR.cuda(), inp.genP.cuda())
        L.premerge(inp.W0.cuda())
        st = dict(L=L, X=X, dY=inp.dY.cuda(),
                  Y=torch.empty(T, m, dtype=torch.bfloat16, device="cuda"),
                  h=None if recompute else torch.empty(T, m, dtype=torch.bfloat16, device="cuda"),
                  u=None if recompute else torch.empty(T, n, dtype=torch.bfloat16, device="cuda"),
                  dX=torch.empty(T, n, dtype=torch.bfloat16, device="cuda"),
                  dgR=torch.empty(L.len_R, device="cuda"), dgP=torch.empty(L.len_P, device="cuda"))
        out.append(st)
    return out


def _poison(layers):
    for st in layers:
        for k in ("Y", "h", "u", "dX", "dgR", "dgP"):
            if st[k] is not None:
                st[k].fill_(float("nan"))
    torch.cuda.synchronize()   # the fills (current stream) land before any other stream runs


def _run(st, stream):
    L = st["L"]   # each Layer owns its workspace
    L.forward(st["X"], st["Y"], saved_h=st["h"], saved_u=st["u"], stream=stream)
    L.backward(st["X"], st["dY"], st["dX"], st["dgR"], st["dgP"], saved_h=st["h"], saved_u=st["u"],
               stream=stream)


def _state(layers):
    return [st[k].clone() for st in layers for k in ("Y", "dX", "dgR", "dgP")]


def _concurrent(layers, main, side):
    fork = torch.cuda.Event()
    fork.record(main)
    joins = []
    for st, s in zip(layers, [main] + side):
        if s is not main:
            s.wait_event(fork)
        _run(st, s)
        if s is not main:
            e = torch.cuda.Event()
            e.record(s)
            joins.append(e)
    for e in joins:
        main.wait_event(e)


@pytest.mark.parametrize("recompute", [False, True])
def test_parallel_streams_bit_identical(px, recompute):
    layers = _layers(px, recompute)
    main = torch.cuda.Stream()
    side = [torch.cuda.Stream() for _ in layers[1:]]
    torch.cuda.synchronize()   # builds and pre-merges ran on the current stream

    _poison(layers)
    for st in layers:
        _run(st, main)
    torch.cuda.synchronize()
    ref = _state(layers)
    assert all(torch.isfinite(t).all() for t in ref)

    for _ in range(2):
        _poison(layers)
        _concurrent(layers, main, side)
        torch.cuda.synchronize()
        for x, y in zip(ref, _state(layers)):
            assert torch.equal(x, y)

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=main):
        _concurrent(layers, main, side)
    for _ in range(2):
        _poison(layers)
        g.replay()
        torch.cuda.synchronize()
        for x, y in zip(ref, _state(layers)):
            assert torch.equal(x, y)
    assert px.poetx_device_status(reset=True) == px.POETX_OK
