"""The benchmark's algorithmic flop and byte accounting (CPU only).

Every TFLOP/s figure and every roofline fraction the benchmark prints divides
these counts by a measured time, so they are pinned here against totals
worked out by hand for the stored workloads:

* flops of one linear, fwd + bwd: 4 T m n (forward and dgrad GEMMs) plus
  6 T (sum of b_R^2 + sum of b_P^2) (block transforms: forward 2, backward
  transform 2 and reduction 2), plus 2 T m n + 2 T sum b_P^2 with recompute;
* bytes of the memory-bound passes: each bf16 T x d operand read or written
  once per pass.
"""
import pytest

import bench
import synth

T = 65536


def test_block_square_sum_with_a_ragged_block():
    assert bench.block_square_sum(2048, 128) == 16 * 128 * 128
    assert bench.block_square_sum(11008, 512) == 21 * 512 * 512 + 256 * 256
    assert bench.block_square_sum(1376, 32) == 43 * 32 * 32


def test_d2048_block_flops():
    # q: 4 T 2048^2 = 1.09951e12; 6 T (16 + 16) 128^2 = 2.06158e11
    q = 4 * T * 2048 * 2048 + 6 * T * 32 * 128 * 128
    # gate (2048 -> 5632): 4 T 2048 * 5632 + 6 T (44 + 16) 128^2; down is its mirror
    gate = 4 * T * 2048 * 5632 + 6 * T * 60 * 128 * 128
    assert q == pytest.approx(1.3057e12, rel=1e-4)
    assert gate == pytest.approx(3.4102e12, rel=1e-4)
    wl = synth.WORKLOADS["d2048_block"]
    assert bench.step_flops(wl, 128) == pytest.approx(4 * q + 3 * gate, rel=1e-12)
    assert bench.step_flops(wl, 128) == pytest.approx(15.453e12, rel=1e-4)
    # b = 256: 8 + 8 and 22 + 8 blocks of 256^2
    q256 = 4 * T * 2048 * 2048 + 6 * T * 16 * 256 * 256
    gate256 = 4 * T * 2048 * 5632 + 6 * T * 30 * 256 * 256
    assert bench.step_flops(wl, 256) == pytest.approx(4 * q256 + 3 * gate256, rel=1e-12)
    assert bench.step_flops(wl, 256) == pytest.approx(17.438e12, rel=1e-4)


def test_recompute_adds_a_forward_gemm_and_the_p_transform():
    wl = synth.WORKLOADS["d4096_ffn"]
    b = 512
    up = 4 * T * 4096 * 11008 + 6 * T * (21 * 512 * 512 + 256 * 256 + 8 * 512 * 512)
    up += 2 * T * 4096 * 11008 + 2 * T * 8 * 512 * 512           # recompute, P side n = 4096
    down = 4 * T * 4096 * 11008 + 6 * T * (21 * 512 * 512 + 256 * 256 + 8 * 512 * 512)
    down += 2 * T * 4096 * 11008 + 2 * T * (21 * 512 * 512 + 256 * 256)   # P side n = 11008
    assert bench.step_flops(wl, b) == pytest.approx(up + down, rel=1e-12)


def test_gemm_flop_classes_partition_the_gemm_flops():
    wl = synth.WORKLOADS["d2048_block"]
    mn = 4 * 2048 * 2048 + 3 * 2048 * 5632
    assert bench.gemm_flops_per_step(wl, "gemm_fwd") == 2 * T * mn
    assert bench.gemm_flops_per_step(wl, "gemm_dgrad") == 2 * T * mn
    wl = synth.WORKLOADS["d4096_ffn"]
    assert bench.gemm_flops_per_step(wl, "gemm_fwd") == 2 * 2 * T * 2 * 4096 * 11008


def test_d2048_memory_pass_bytes():
    wl = synth.WORKLOADS["d2048_block"]
    widths = 4 * (2048 + 2048) + 3 * (2048 + 5632)       # sum of n + m over the linears
    # four permutation passes of 2 bytes in and 2 bytes out per element
    assert bench.kind_bytes_per_step(wl, 128, "gather") == 8 * T * widths
    # forward transforms read + write (4 B), fused backward reads two and writes one (6 B)
    assert bench.kind_bytes_per_step(wl, 128, "blockdiag") == 10 * T * widths
    assert bench.kind_bytes_per_step(wl, 128, "gradred") == 0
    assert bench.kind_bytes_per_step(wl, 128, "gather") == 20669530112
    assert bench.kind_bytes_per_step(wl, 128, "blockdiag") == 25836912640


def test_unfused_256_sides_are_counted_as_transform_plus_reduction():
    # at d = 11008 the 256-wide fused kernel's grid (86 CTAs per slot) does not
    # fill 80% of the SMs, so that side runs the separate transform (4 B) and
    # reduction (4 B): 2 more bytes per element than the fused 6 B
    wl = synth.WORKLOADS["d4096_ffn"]
    n, m = 4096, 11008
    gr = bench.kind_bytes_per_step(wl, 256, "gradred")
    assert gr == 2 * T * (2 * m + 2 * m)      # up: R side 11008; down: P side 11008
    bd = bench.kind_bytes_per_step(wl, 256, "blockdiag")
    per = lambda nn, mm, fm, fn: T * (2 * nn + 2 * mm + (3 if fm else 2) * mm + (3 if fn else 2) * nn
                                      + 2 * nn) * 2
    assert bd == per(n, m, False, True) + per(m, n, True, False)
