"""The seeded synthetic inputs (CPU only).

Full-size GPU parity samples rows of 65536-token inputs and regenerates only
those rows for the oracle, which is sound only if a row depends on its seed,
index and width and not on how many rows are generated around it.  The
workload shapes are those of the stated configurations.
"""
import numpy as np
import pytest
import torch

import synth


@pytest.mark.parametrize("t0,t1", [(0, 1), (255, 257), (300, 1000), (4096, 4100)])
def test_a_row_does_not_depend_on_the_rows_generated_with_it(t0, t1):
    full = synth.rows(1234, 0, 5000, 96, 1.0)
    assert np.array_equal(synth.rows(1234, t0, t1, 96, 1.0), full[t0:t1])


def test_threaded_generation_equals_sequential():
    # 20 chunks of 256 rows are filled by a thread pool, 3 chunks sequentially
    many = synth.rows(77, 0, 20 * synth.CHUNK_ROWS, 40, 0.5)
    for c in (0, 7, 19):
        lo = c * synth.CHUNK_ROWS
        assert np.array_equal(synth.rows(77, lo, lo + 3, 40, 0.5), many[lo:lo + 3])


def test_scale_and_distribution():
    x = synth.rows(5, 0, 4096, 256, 0.02)
    assert x.dtype == np.float32
    assert abs(float(x.std()) - 0.02) < 0.002 and abs(float(x.mean())) < 0.001
    assert np.array_equal(synth.rows(5, 0, 4096, 256, 1.0) * np.float32(0.02), x)
    v = synth.vector(9, 100000, 0.01)
    assert abs(float(v.std()) - 0.01) < 0.0002


def test_seeds_and_linears_draw_independent_streams():
    a = synth.rows(synth.SEED_X + 0, 0, 4, 64, 1.0)
    b = synth.rows(synth.SEED_X + 1, 0, 4, 64, 1.0)
    c = synth.rows(synth.SEED_DY + 0, 0, 4, 64, 1.0)
    assert not np.array_equal(a, b) and not np.array_equal(a, c)


def test_round_to_bf16_is_round_to_nearest_even():
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9, -2.5e-3], dtype=np.float32)
    got = synth.round_to(vals, "bf16").float().numpy()
    # bf16 keeps 8 significant bits: ties at 1 + 2^-8 and 1 + 3 * 2^-8 go to even
    assert got[0] == 1.0 and got[1] == 1.0 and got[2] == 1.0 + 2 ** -6 and got[3] == 1.0
    assert got[4] == np.float32(torch.tensor(-2.5e-3).to(torch.bfloat16).item())
    assert synth.round_to(vals, "fp32").dtype == torch.float32


def test_workload_shapes():
    w = synth.WORKLOADS
    d2048 = w["d2048_block"]
    assert d2048.tokens == 256 * 256 and list(d2048.block_sizes) == [128, 256]
    assert d2048.merge_each_step and not d2048.recompute and d2048.dtype == "bf16"
    assert [(l.n, l.m) for l in d2048.linears] == [(2048, 2048)] * 4 + [(2048, 5632)] * 2 + [(5632, 2048)]
    d4096 = w["d4096_ffn"]
    assert d4096.tokens == 65536 and d4096.recompute
    assert [(l.n, l.m) for l in d4096.linears] == [(4096, 11008), (11008, 4096)]
    assert list(d4096.block_sizes) == [32, 64, 128, 256, 512]
    d1024 = w["d1024_block"]
    assert d1024.tokens == 256 * 128 and d1024.recompute and list(d1024.block_sizes) == [64]
    assert [(l.n, l.m) for l in d1024.linears] == [(1024, 1024)] * 4 + [(1024, 2816)] * 2 + [(2816, 1024)]
    ll = w["llama60m_block"]
    assert ll.tokens == 8192 and list(ll.block_sizes) == [32]
    assert [(l.n, l.m) for l in ll.linears] == [(512, 512)] * 4 + [(512, 1376)] * 2 + [(1376, 512)]
    f = w["fp32_256"]
    assert f.dtype == "fp32" and f.tokens == 512 and [(l.n, l.m) for l in f.linears] == [(256, 256)]
