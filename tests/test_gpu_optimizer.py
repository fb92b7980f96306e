"""AdamW step on packed generators (needs a B300).

The optimizer the pages train with is not named; the reading is AdamW with
decoupled weight decay (see the oracle's ``adamw_step``).  The kernel runs
in fp32 and must follow the fp64 oracle over several steps with changing
gradients, including weight decay and a bias correction that changes each
step.
"""
import numpy as np
import pytest
import torch

import oracle as O
from tests.gpu_cases import rel_fro

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def px():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import orthogonal_equivalence_reparameterized_poetx_b300 as m
    return m


@pytest.mark.parametrize("length", [1, 1000, O.packed_length(2048, 128)])
def test_adamw_follows_the_oracle_over_steps(px, length):
    rng = np.random.default_rng(length)
    th = (rng.standard_normal(length) * 0.01).astype(np.float32)
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.05)
    gen = torch.tensor(th, device="cuda")
    m1 = torch.zeros(length, device="cuda")
    m2 = torch.zeros(length, device="cuda")
    o_th, o_m1, o_m2 = th.astype(np.float64), np.zeros(length), np.zeros(length)
    for step in range(1, 6):
        g = (rng.standard_normal(length) * 10.0 ** rng.integers(-3, 2)).astype(np.float32)
        px.poetx_generator_adamw(gen, torch.tensor(g, device="cuda"), m1, m2, length, step, **hp)
        o_th, o_m1, o_m2 = O.adamw_step(o_th, g, o_m1, o_m2, step, hp["lr"], hp["beta1"],
                                        hp["beta2"], hp["eps"], hp["weight_decay"])
    torch.cuda.synchronize()
    assert px.poetx_device_status(reset=True) == px.POETX_OK
    assert rel_fro(gen.double().cpu().numpy(), o_th) <= 1e-6
    assert rel_fro(m1.double().cpu().numpy(), o_m1) <= 1e-6
    assert rel_fro(m2.double().cpu().numpy(), o_m2) <= 1e-6
    # and the update itself (theta_now - theta_0) to fp32 accuracy
    assert rel_fro(gen.double().cpu().numpy() - th, o_th - th) <= 1e-5


def test_adamw_argument_errors(px):
    z = torch.zeros(4, device="cuda")
    with pytest.raises(px.PoetxError):
        px.poetx_generator_adamw(z, z, z, z, 4, 0, 1e-3)        # step counts from 1
    with pytest.raises(px.PoetxError):
        px.poetx_generator_adamw(z, z, z, z, 4, 1, 1e-3, beta1=1.0)
    px.poetx_generator_adamw(z, z, z, z, 0, 1, 1e-3)            # empty: no-op
