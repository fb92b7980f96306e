"""The allocation-free forward entry point (needs a B300).

poetx_linear_fwd_noalloc serves callers that cannot allocate device memory
where they call the layer: runtimes that hand out every byte from a fixed
arena, plugins whose host forbids device allocation in its callbacks, or
hosts whose allocator belongs to someone else.  Instead of a caller-provided workspace it uses a fixed
device array inside the library.  These tests call it through the C ABI and
compare it with the ordinary forward (caller-provided workspace) on the same
inputs.  Both run the same deterministic kernels, so the outputs must be
identical bit for bit.  Before the compared calls, a call on another layer
shape fills the shared scratch with a different layout, and the compared
call is made twice in a row, so a stale-scratch bug cannot pass.  Oversized
requests must be refused before any launch.  This file is collected last so a stop-at-first-failure run has
already run every other test.
"""
import numpy as np
import pytest
import torch

import oracle as O
from tests.gpu_cases import make_inputs, rel_fro

pytestmark = pytest.mark.gpu

TOL = 2e-2   # the bf16 tolerance the parity tests use (for the oracle check)


def _dirty_the_scratch(px):
    """One allocation-free forward of a different layer shape and token count,
    so the compared calls start from scratch laid out by another call."""
    m, n, b, T = 640, 256, 32, 129
    inp = make_inputs(m, n, b, b, T, "bf16", index=5)
    desc = px.make_desc(m, n, b, b, inp.seed_R, inp.seed_P, dtype="bf16")
    layer = px.Layer(desc, T)
    layer.build(inp.genR.cuda(), inp.genP.cuda())
    layer.premerge(inp.W0.cuda())
    Y = torch.empty(T, m, dtype=torch.bfloat16, device="cuda")
    h = torch.empty(T, m, dtype=torch.bfloat16, device="cuda")
    px.poetx_linear_fwd_noalloc(desc, layer.params, layer.W0p, inp.X.cuda(), T, Y, h, None)
    torch.cuda.synchronize()
    assert px.poetx_device_status(reset=True) == px.POETX_OK


@pytest.fixture(scope="module")
def px():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import orthogonal_equivalence_reparameterized_poetx_b300 as m
    return m


@pytest.mark.parametrize("keep_h", [True, False])
def test_noalloc_forward_matches_workspace_forward_twice(px, keep_h):
    m, n, b, T = 512, 384, 64, 300
    inp = make_inputs(m, n, b, b, T, "bf16", index=3)
    desc = px.make_desc(m, n, b, b, inp.seed_R, inp.seed_P, dtype="bf16")
    assert px.poetx_workspace_size(desc, T) <= px.NOALLOC_SCRATCH_BYTES
    layer = px.Layer(desc, T)
    layer.build(inp.genR.cuda(), inp.genP.cuda())
    layer.premerge(inp.W0.cuda())
    X = inp.X.cuda()
    Y_ref = torch.empty(T, m, dtype=torch.bfloat16, device="cuda")
    h_ref = torch.empty(T, m, dtype=torch.bfloat16, device="cuda")
    layer.forward(X, Y_ref, saved_h=h_ref)
    _dirty_the_scratch(px)
    for call in range(2):
        Y = torch.full((T, m), float("nan"), dtype=torch.bfloat16, device="cuda")
        h = torch.empty(T, m, dtype=torch.bfloat16, device="cuda") if keep_h else None
        px.poetx_linear_fwd_noalloc(desc, layer.params, layer.W0p, X, T, Y, h, None)
        torch.cuda.synchronize()
        assert px.poetx_device_status(reset=True) == px.POETX_OK
        assert torch.isfinite(Y.float()).all(), f"call {call}: unwritten outputs"
        assert torch.equal(Y, Y_ref), f"call {call}: Y differs from the workspace forward"
        if keep_h:
            assert torch.equal(h, h_ref), f"call {call}: h differs from the workspace forward"
    # and the result is the layer's: compare once with the oracle as well
    spec = O.LayerSpec(m, n, b, b, inp.seed_R, inp.seed_P)
    Y_o, _ = O.forward_input_centric(spec, inp.W0.double().numpy(), inp.X.double().numpy(),
                                     inp.genR.double().numpy(), inp.genP.double().numpy())
    assert rel_fro(Y.double().cpu().numpy(), Y_o) <= TOL


def test_noalloc_forward_refuses_oversized_requests(px):
    m, n, b = 2048, 2048, 128
    desc = px.make_desc(m, n, b, b, 1, 2, dtype="bf16")
    T = 65536
    assert px.poetx_workspace_size(desc, T) > px.NOALLOC_SCRATCH_BYTES
    with pytest.raises(px.PoetxError) as ei:
        px.poetx_linear_fwd_noalloc(desc, 256, 256, 256, T, 256, None, None)
    assert ei.value.status == px.POETX_ERR_UNSUPPORTED
