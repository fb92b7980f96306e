"""One training step from host buffers (poetx_linear_step_host; needs a B300).

The call copies X and dY from host memory, runs the forward and the backward
and copies the packed generator gradients back, synchronising before it
returns.  Its results are those of the device calls on the same inputs, bit
for bit (the same kernels in the same order; every reduction is
deterministic), and they match the oracle within the bf16 / fp32 tolerances.
Checked for pinned and pageable host buffers, with and without saved
activations, and for two calls in a row that reuse the device buffers with
different host inputs (the second copy of dY must not overtake the first
call's backward, which reads the same device buffer).
"""
import pytest
import torch

import oracle as O
from tests.gpu_cases import make_inputs, rel_fro, run_oracle

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-2, "fp32": 1e-5}


@pytest.fixture(scope="module")
def px():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import orthogonal_equivalence_reparameterized_poetx_b300 as m
    return m


def _layer(px, m, n, b, T, dtype, index):
    inp = make_inputs(m, n, b, b, T, dtype, index=index)
    desc = px.make_desc(m, n, b, b, inp.seed_R, inp.seed_P, dtype=dtype)
    layer = px.Layer(desc, T)
    layer.build(inp.genR.cuda(), inp.genP.cuda())
    layer.premerge(inp.W0.cuda())
    return inp, desc, layer


def _device_bufs(layer, T, saved):
    m, n, dt = layer.desc.m, layer.desc.n, layer.dtype
    e = lambda *s, **k: torch.empty(*s, device="cuda", **k)
    return dict(X=e(T, n, dtype=dt), dY=e(T, m, dtype=dt), Y=e(T, m, dtype=dt),
                h=e(T, m, dtype=dt) if saved else None, u=e(T, n, dtype=dt) if saved else None,
                dX=e(T, n, dtype=dt), dgR=e(layer.len_R), dgP=e(layer.len_P))


def _step_host(px, layer, Xh, dYh, T, B, pinned=True):
    gR = torch.empty(layer.len_R, dtype=torch.float32, pin_memory=pinned)
    gP = torch.empty(layer.len_P, dtype=torch.float32, pin_memory=pinned)
    px.poetx_linear_step_host(layer.desc, layer.params, layer.W0p, Xh, dYh, T, B["X"], B["dY"],
                              B["Y"], B["h"], B["u"], B["dX"], B["dgR"], B["dgP"], gR, gP,
                              layer.workspace)
    assert px.poetx_device_status(reset=True) == px.POETX_OK
    return dict(Y=B["Y"].cpu(), dX=B["dX"].cpu(), dgR=gR.clone(), dgP=gP.clone(),
                dgR_dev=B["dgR"].cpu(), dgP_dev=B["dgP"].cpu())


def _device_step(px, layer, X, dY, T, saved):
    B = _device_bufs(layer, T, saved)
    X, dY = X.cuda(), dY.cuda()
    layer.forward(X, B["Y"], saved_h=B["h"], saved_u=B["u"])
    layer.backward(X, dY, B["dX"], B["dgR"], B["dgP"], saved_h=B["h"], saved_u=B["u"])
    torch.cuda.synchronize()
    assert px.poetx_device_status(reset=True) == px.POETX_OK
    return dict(Y=B["Y"].cpu(), dX=B["dX"].cpu(), dgR=B["dgR"].cpu(), dgP=B["dgP"].cpu())


def _host(t, pinned):
    out = torch.empty(t.shape, dtype=t.dtype, pin_memory=pinned)
    out.copy_(t)
    return out


@pytest.mark.parametrize("m,n,b,T,dtype,saved,pinned", [
    (512, 384, 64, 300, "bf16", True, True),
    (1376, 1032, 128, 777, "bf16", False, True),   # recompute, CTA-pair GEMMs, ragged tiles
    (512, 384, 64, 300, "bf16", True, False),      # pageable host memory
    (256, 256, 32, 200, "fp32", False, True),
])
def test_step_host_equals_device_calls_and_oracle(px, m, n, b, T, dtype, saved, pinned):
    inp, desc, layer = _layer(px, m, n, b, T, dtype, index=11)
    B = _device_bufs(layer, T, saved)
    got = _step_host(px, layer, _host(inp.X, pinned), _host(inp.dY, pinned), T, B, pinned)
    want = _device_step(px, layer, inp.X, inp.dY, T, saved)
    for k in ("Y", "dX", "dgR", "dgP"):
        assert torch.equal(got[k], want[k]), k
    assert torch.equal(got["dgR"], got["dgR_dev"]) and torch.equal(got["dgP"], got["dgP_dev"])

    ref = run_oracle(O.LayerSpec(m, n, b, b, inp.seed_R, inp.seed_P), inp)
    errs = {k: rel_fro(got[k].double().numpy(), ref[k]) for k in ("Y", "dX", "dgR", "dgP")}
    assert all(e <= TOL[dtype] for e in errs.values()), errs


def test_two_calls_reuse_device_buffers(px):
    """Back-to-back calls with different host inputs on one set of device
    buffers: each call's results are those of its own inputs."""
    m, n, b, T = 640, 512, 64, 400
    inp, desc, layer = _layer(px, m, n, b, T, "bf16", index=12)
    second = make_inputs(m, n, b, b, T, "bf16", index=13)
    B = _device_bufs(layer, T, True)
    first_out = _step_host(px, layer, _host(inp.X, True), _host(inp.dY, True), T, B)
    second_out = _step_host(px, layer, _host(second.X, True), _host(second.dY, True), T, B)
    want1 = _device_step(px, layer, inp.X, inp.dY, T, True)
    want2 = _device_step(px, layer, second.X, second.dY, T, True)
    for k in ("Y", "dX", "dgR", "dgP"):
        assert torch.equal(first_out[k], want1[k]), k
        assert torch.equal(second_out[k], want2[k]), k
    assert not torch.equal(first_out["dgR"], second_out["dgR"])


def test_step_host_zero_tokens(px):
    """T = 0: nothing is copied in, and the host gradients come back zero."""
    m, n, b = 256, 256, 32
    inp, desc, layer = _layer(px, m, n, b, 1, "bf16", index=14)
    B = _device_bufs(layer, 1, True)
    gR = torch.full((layer.len_R,), 3.0, pin_memory=True)
    gP = torch.full((layer.len_P,), 3.0, pin_memory=True)
    px.poetx_linear_step_host(desc, layer.params, layer.W0p, _host(inp.X, True), _host(inp.dY, True),
                              0, B["X"], B["dY"], B["Y"], B["h"], B["u"], B["dX"], B["dgR"],
                              B["dgP"], gR, gP, layer.workspace)
    assert px.poetx_device_status(reset=True) == px.POETX_OK
    assert float(gR.abs().max()) == 0.0 and float(gP.abs().max()) == 0.0


def test_async_steps_in_flight_equal_synchronous_steps(px):
    """Two layers' asynchronous host steps enqueued back to back, each with
    its own device buffers, then one synchronisation: the same results, bit
    for bit, as the synchronous calls."""
    cases = [(640, 512, 64, 400, 15), (512, 1376, 128, 300, 16)]
    setups = []
    for m, n, b, T, index in cases:
        inp, desc, layer = _layer(px, m, n, b, T, "bf16", index=index)
        setups.append((inp, layer, T, _device_bufs(layer, T, True), _device_bufs(layer, T, True)))
    want = [_step_host(px, layer, _host(inp.X, True), _host(inp.dY, True), T, Bs)
            for inp, layer, T, Bs, _ in setups]
    hosts = []
    for inp, layer, T, _, Ba in setups:
        Xh, dYh = _host(inp.X, True), _host(inp.dY, True)
        gR = torch.empty(layer.len_R, dtype=torch.float32, pin_memory=True)
        gP = torch.empty(layer.len_P, dtype=torch.float32, pin_memory=True)
        px.poetx_linear_step_host_async(layer.desc, layer.params, layer.W0p, Xh, dYh, T, Ba["X"],
                                        Ba["dY"], Ba["Y"], Ba["h"], Ba["u"], Ba["dX"], Ba["dgR"],
                                        Ba["dgP"], gR, gP, layer.workspace)
        hosts.append((Xh, dYh, gR, gP))
    torch.cuda.synchronize()
    assert px.poetx_device_status(reset=True) == px.POETX_OK
    for (inp, layer, T, _, Ba), (_, _, gR, gP), w in zip(setups, hosts, want):
        assert torch.equal(Ba["Y"].cpu(), w["Y"]) and torch.equal(Ba["dX"].cpu(), w["dX"])
        assert torch.equal(gR, w["dgR"]) and torch.equal(gP, w["dgP"])
