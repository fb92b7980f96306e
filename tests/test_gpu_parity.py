"""GPU parity of the CUDA path against the fp64 oracle (needs a B300).

Every case runs forward + backward through the C ABI and through the oracle
on identical seeded inputs (the oracle consumes the already-rounded values)
and compares Y, dX and both packed generator gradients by relative Frobenius
error: <= 1e-5 for fp32, <= 2e-2 for bf16 with fp32 accumulation.  The same
bound holds for the worst single row of Y and dX and for the worst single
block of each generator gradient, so a local error cannot hide in the
aggregate.  The
pre-merged weight W0' is a pure permutation copy and must match bit for bit,
which also checks the device permutations against the oracle's.

Shapes span several 128-token tiles with a ragged token tail, ragged last
blocks (b not dividing the dimension), every bf16 block size, m != n, both
Cayley and Neumann modes, and stored-h versus recompute.
"""
import numpy as np
import pytest
import torch

import oracle as O
from tests.gpu_cases import make_inputs, parity_errors, rel_fro, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

TOL = {"fp32": 1e-5, "bf16": 2e-2}


@pytest.fixture(scope="module")
def px():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import orthogonal_equivalence_reparameterized_poetx_b300 as m
    return m


def _case(px, m, n, bR, bP, T, dtype, mode="cayley", k=3, recompute=False, index=0, gstd=0.01,
          save_u=False):
    inp = make_inputs(m, n, bR, bP, T, dtype, index=index, gstd=gstd)
    desc = px.make_desc(m, n, bR, bP, inp.seed_R, inp.seed_P, dtype=dtype, mode=mode, neumann_k=k)
    spec = O.LayerSpec(m, n, bR, bP, inp.seed_R, inp.seed_P,
                       "neumann" if mode == "neumann" else "exact", k)
    g = run_gpu(px, desc, inp, recompute, save_u=save_u)
    o = run_oracle(spec, inp)
    assert np.array_equal(g["W0p"], o["W0p"]), "pre-merged weight must be a bit-exact copy"
    if save_u:
        # u = X[:, pi_P] is a permutation copy of the input: bit-exact
        u_o = inp.X.double().numpy()[:, O.permutation(inp.seed_P, n)]
        assert np.array_equal(g["u"], u_o), "saved u must be the permuted input, bit for bit"
    tol = TOL[dtype]
    errs = parity_errors(g, o, m, n, bR, bP)
    for k_, e in errs.items():
        assert e <= tol, f"{k_}: rel Frobenius {e:.3e} > {tol:.0e} ({errs})"
    return errs


# ------------------------------------------------------------------ fp32 path

def test_fp32_workload_256(px):
    # single POET-X linear 256 -> 256, b = 32, 512 tokens, stored h
    _case(px, 256, 256, 32, 32, 512, "fp32")


def test_fp32_ragged_blocks_and_tokens_recompute(px):
    _case(px, 200, 136, 64, 48, 77, "fp32", recompute=True, gstd=0.05)


def test_fp32_neumann(px):
    _case(px, 128, 128, 32, 32, 100, "fp32", mode="neumann", gstd=0.05)


def test_fp32_neumann_b256_ragged(px):
    # fp32 layers keep CUDA-core products for the Neumann build and chain rule
    _case(px, 512, 384, 256, 256, 64, "fp32", mode="neumann", gstd=0.02)


def test_fp32_cluster_builder_b256(px):
    # 256-wide blocks: one cluster of two 1024-thread CTAs per block
    _case(px, 512, 384, 256, 128, 64, "fp32", gstd=0.02)


@pytest.mark.parametrize("gstd", [0.02, 0.1])
def test_fp32_cluster_builder_b512_ragged(px, gstd):
    # 768 = 512 + 256 and 640 = 512 + 128: ragged last blocks inverted as the
    # identity-padded 512 x 512 matrix; gstd = 0.1 gives ||Q|| of several units
    _case(px, 768, 640, 512, 512, 64, "fp32", gstd=gstd)


def test_fp32_blocked_builder_b384(px):
    # a block size that is neither <= 128 nor 256 / 512: the panel-wise
    # Gauss-Jordan builder with batched products
    _case(px, 768, 384, 384, 384, 64, "fp32", gstd=0.02)


# ------------------------------------------------------------------ bf16 path

@pytest.mark.parametrize("recompute", [False, True])
def test_bf16_b32_ragged_tokens(px, recompute):
    _case(px, 384, 256, 32, 32, 1000, "bf16", recompute=recompute)


@pytest.mark.parametrize("dtype,recompute", [("fp32", False), ("fp32", True),
                                             ("bf16", False), ("bf16", True)])
def test_saved_u_replaces_the_input_in_the_backward(px, dtype, recompute):
    """The forward keeps u = X[:, pi_P]; the backward gets it instead of X
    (X is NULL there), with h saved or recomputed."""
    bs = 32 if dtype == "fp32" else 128
    _case(px, 384, 256, bs, bs, 300, dtype, recompute=recompute, save_u=True)


def test_bf16_b64(px):
    _case(px, 256, 640, 64, 64, 300, "bf16")


@pytest.mark.parametrize("T", [777, 12289])
def test_bf16_cta_pair_gemms_with_ragged_tiles(px, T):
    # m = 1376 and n = 1032 are wide enough for the CTA-pair GEMMs (256 x 256
    # tiles split over two CTAs) in the dgrad, and at T = 12289 (outputs above
    # 32 MB) in the forward too, where T = 777 takes the fused R epilogue;
    # neither m, n nor T are multiples of 256, and b = 64 leaves a ragged
    # last block
    _case(px, 1376, 1032, 64, 64, T, "bf16")


def test_bf16_b128(px):
    _case(px, 512, 512, 128, 128, 513, "bf16")


def test_bf16_b128_ragged_last_blocks(px):
    # 456 = 3 x 128 + 72 and 328 = 2 x 128 + 72: a short last block on both
    # sides in the fused transform + reduction and the clustered Cayley backward
    _case(px, 456, 328, 128, 128, 300, "bf16", gstd=0.03)


def test_bf16_neumann_b256_tensor_core_builder(px):
    # Neumann blocks of 256 (built and differentiated with tensor-core products)
    _case(px, 512, 640, 256, 256, 200, "bf16", mode="neumann", gstd=0.02)


def test_bf16_b256_ragged_last_blocks(px):
    # 640 = 2 x 256 + 128 and 328 = 256 + 72: short last blocks on both sides
    # in the clustered 256-wide Cayley backward
    _case(px, 640, 328, 256, 256, 300, "bf16", gstd=0.02)


def test_bf16_b512_ragged_block_and_b256(px):
    # 768 = 512 + ragged 256 on the R side; P side b = 256
    _case(px, 768, 512, 512, 256, 260, "bf16", recompute=True)


@pytest.mark.parametrize("m,n,b,T", [(1280, 1024, 512, 700), (1024, 1536, 256, 333)])
def test_bf16_wide_superblocks_on_cta_pairs(px, m, n, b, T):
    # outputs of at least 1024 with 256- and 512-wide super-blocks: the block
    # transforms (K = sb) and, at b = 512, the token reductions run on CTA
    # pairs with 256 x 256 tiles; 1280 = 2 x 512 + 256 ends in a partial
    # super-block
    _case(px, m, n, b, b, T, "bf16", gstd=0.02, index=5)


def test_bf16_ragged_superblock(px):
    # 1376 = 10 x 128 + 96: the last 128-wide super-block is partial
    _case(px, 1376, 512, 32, 32, 128, "bf16")
    _case(px, 512, 1376, 32, 32, 128, "bf16", index=1)


def test_bf16_neumann(px):
    _case(px, 256, 256, 128, 128, 200, "bf16", mode="neumann", gstd=0.05)


@pytest.mark.parametrize("k", [1, 2, 6])
def test_bf16_neumann_fused_builder_orders(px, k):
    # the fused tensor-core builder runs k products; 384 = 256 + 128 ragged
    _case(px, 512, 384, 256, 256, 200, "bf16", mode="neumann", k=k, gstd=0.02)


def test_bf16_neumann_b512_ragged(px):
    # eight-CTA clusters per 512-wide block; 768 = 512 + 256 ragged
    _case(px, 768, 512, 512, 512, 130, "bf16", mode="neumann", gstd=0.01)


@pytest.mark.parametrize("m,b,recompute", [(200, 64, False), (200, 64, True), (1000, 32, False),
                                         (896, 128, True)])
def test_bf16_r_transform_in_the_gemm_epilogue(px, m, b, recompute):
    # outputs narrower than 1024 take the forward GEMM whose epilogue applies
    # the R blocks (h written only when kept); 200 = 128 + 72 and 1000 =
    # 7 x 128 + 104 end in a partial super-block, and 777 tokens in a partial
    # token tile
    _case(px, m, 320, b, b, 777, "bf16", recompute=recompute, index=3)


def test_bf16_single_token_and_single_block(px):
    _case(px, 128, 128, 128, 128, 1, "bf16")


@pytest.mark.parametrize("recompute", [False, True])
def test_bf16_long_tokens_many_tiles(px, recompute):
    # 9617 tokens (ragged tail of 17 after 150 tiles of 64): the persistent
    # kernels cycle through many tiles per CTA, with every row still checked
    _case(px, 2048, 1024, 128, 128, 64 * 150 + 17, "bf16", recompute=recompute, index=7)


# ------------------------------------------------------------------ other ABI behaviour

@pytest.mark.parametrize("m,n,b,mode", [
    (256, 256, 64, "cayley"),
    (384, 256, 128, "neumann"),     # fused tensor-core Neumann backward (b = 128)
    (512, 384, 256, "cayley"),
    (768, 512, 512, "neumann"),     # batched Neumann chain rule
])
def test_accumulate_adds_into_generator_gradients(px, m, n, b, mode):
    inp = make_inputs(m, n, b, b, 200, "bf16")
    desc = px.make_desc(m, n, b, b, inp.seed_R, inp.seed_P, dtype="bf16", mode=mode)
    g = run_gpu(px, desc, inp, recompute=True)
    layer = g["layer"]
    dev = "cuda"
    X, dY = inp.X.to(dev), inp.dY.to(dev)
    dgR = torch.from_numpy(g["dgR"]).float().to(dev)
    dgP = torch.from_numpy(g["dgP"]).float().to(dev)
    layer.backward(X, dY, None, dgR, dgP, accumulate=True)
    torch.cuda.synchronize()
    assert rel_fro(dgR.double().cpu().numpy(), 2 * g["dgR"]) < 1e-6
    assert rel_fro(dgP.double().cpu().numpy(), 2 * g["dgP"]) < 1e-6


def test_zero_tokens(px):
    desc = px.make_desc(128, 128, 32, 32, 1, 2, dtype="bf16")
    layer = px.Layer(desc, 1)
    X = torch.empty(0, 128, dtype=torch.bfloat16, device="cuda")
    Y = torch.empty(0, 128, dtype=torch.bfloat16, device="cuda")
    layer.forward(X, Y)
    dgR = torch.full((layer.len_R,), 3.0, device="cuda")
    dgP = torch.full((layer.len_P,), 3.0, device="cuda")
    layer.backward(X, Y, None, dgR, dgP)
    torch.cuda.synchronize()
    assert float(dgR.abs().max()) == 0.0 and float(dgP.abs().max()) == 0.0


def test_bounded_wait_gives_up_and_reports_timeout(px):
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    st = px.poetx_selftest_bounded_wait(2_000_000)      # 2 ms deadline on a barrier nobody completes
    t1.record()
    torch.cuda.synchronize()
    assert st == px.POETX_ERR_TIMEOUT
    assert t0.elapsed_time(t1) < 2000.0
    # the self-test restores the status word; the context stays usable
    assert px.poetx_device_status(reset=False) == px.POETX_OK
    x = torch.ones(4, device="cuda")
    assert float((x * 2).sum()) == 8.0


# ------------------------------------------------------------------ degenerate cases

@pytest.mark.parametrize("m,n,b,mode,dtype", [
    (1376, 1032, 64, "cayley", "bf16"), (768, 640, 256, "neumann", "bf16"),
    (512, 384, 512 // 4, "cayley", "fp32"),
])
def test_zero_generators_reduce_to_the_plain_linear(px, m, n, b, mode, dtype):
    """With zero generators every block is the identity (Cayley and Neumann
    alike), so under any permutations the layer is Y = X W0^T and dX = dY W0,
    and the generator gradients are the skew part of the token reductions.
    Checked against torch's own matmul, independently of the oracle: this
    pins the gathers and scatters as exact inverses of each other."""
    T = 333
    inp = make_inputs(m, n, b, b, T, dtype, index=21)
    desc = px.make_desc(m, n, b, b, inp.seed_R, inp.seed_P, dtype=dtype, mode=mode)
    layer = px.Layer(desc, T)
    layer.build(torch.zeros_like(inp.genR).cuda(), torch.zeros_like(inp.genP).cuda())
    layer.premerge(inp.W0.cuda())
    X, dY = inp.X.cuda(), inp.dY.cuda()
    Y = torch.empty(T, m, dtype=layer.dtype, device="cuda")
    dX = torch.empty(T, n, dtype=layer.dtype, device="cuda")
    dgR = torch.empty(layer.len_R, device="cuda")
    dgP = torch.empty(layer.len_P, device="cuda")
    layer.forward(X, Y)
    layer.backward(X, dY, dX, dgR, dgP)
    torch.cuda.synchronize()
    assert px.poetx_device_status(reset=True) == px.POETX_OK
    W0 = inp.W0.double()
    Y_ref = inp.X.double() @ W0.T
    dX_ref = inp.dY.double() @ W0
    tol = TOL[dtype]
    assert rel_fro(Y.double().cpu().numpy(), Y_ref.numpy()) <= tol
    assert rel_fro(dX.double().cpu().numpy(), dX_ref.numpy()) <= tol
