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
    sum_n = 4 * 2048 + 2 * 2048 + 5632
    sum_m = 4 * 2048 + 2 * 5632 + 2048
    assert sum_n + sum_m == widths
    # four permutation passes of 2 bytes in and 2 bytes out per element
    assert bench.kind_bytes_per_step(wl, 128, "gather") == 8 * T * widths
    # forward P transform reads + writes (4 B per element of n; the R transform
    # runs in the forward GEMM's epilogue), the fused backward transforms read
    # two operands and write one (6 B per element of m and of n)
    assert bench.kind_bytes_per_step(wl, 128, "blockdiag") == 2 * T * (5 * sum_n + 3 * sum_m)
    assert bench.kind_bytes_per_step(wl, 128, "gradred") == 0
    assert bench.kind_bytes_per_step(wl, 128, "gather") == 20669530112
    assert bench.kind_bytes_per_step(wl, 128, "blockdiag") == 20199768064


def test_epilogue_placement_follows_the_library():
    # the R transform is in the forward GEMM for b <= 128 only
    assert bench.r_in_gemm(32) and bench.r_in_gemm(128) and not bench.r_in_gemm(256)
    # the P side is in the dgrad where that GEMM is single-CTA or its output <= 32 MB
    assert bench.p_in_dgrad(8192, 512, 32)          # narrow output
    assert bench.p_in_dgrad(8192, 1376, 32)         # 22.5 MB
    assert not bench.p_in_dgrad(32768, 1024, 64)    # 64 MB on CTA pairs
    assert bench.p_in_dgrad(128, 4096, 128)         # fewer than 256 tokens: single CTA
    assert not bench.p_in_dgrad(8192, 512, 256)
    # LLaMA-60M: every P side is in the dgrad, so the blockdiag class moves the
    # forward P transform (4 B) and the fused R backward (6 B) only
    wl = synth.WORKLOADS["llama60m_block"]
    t = wl.tokens
    sum_n = 6 * 512 + 1376
    sum_m = 4 * 512 + 2 * 1376 + 512
    assert bench.kind_bytes_per_step(wl, 32, "blockdiag") == 2 * t * (2 * sum_n + 3 * sum_m)
    assert bench.kind_bytes_per_step(wl, 32, "gather") == 8 * t * (sum_n + sum_m)
    # with the permutations inside the transforms (bound 1536) the forward
    # X -> u -> v moves 6 B and the R backward gathers dY itself; the gather
    # class keeps z -> Y and du -> dX
    old = bench.FUSED_GATHER_MAX
    try:
        bench.FUSED_GATHER_MAX = 1536
        assert bench.kind_bytes_per_step(wl, 32, "blockdiag") == 2 * t * (3 * sum_n + 3 * sum_m)
        assert bench.kind_bytes_per_step(wl, 32, "gather") == 4 * t * (sum_n + sum_m)
    finally:
        bench.FUSED_GATHER_MAX = old
    # and the dgrad class carries the transform and reduction flops, 4 T sum b_P^2
    sq = lambda d: bench.block_square_sum(d, 32)
    extra = 4 * t * (6 * sq(512) + sq(1376))
    assert bench.kind_flops_per_step(wl, 32, "gemm_dgrad") == pytest.approx(
        bench.gemm_flops_per_step(wl, "gemm_dgrad") + extra, rel=1e-12)


def test_unfused_256_sides_are_counted_as_transform_plus_reduction():
    # at d = 11008 the 256-wide fused kernel's grid (86 CTAs per slot) does not
    # fill 80% of the SMs, so that side runs the separate transform (4 B) and
    # reduction (4 B): 2 more bytes per element than the fused 6 B
    wl = synth.WORKLOADS["d4096_ffn"]
    n, m = 4096, 11008
    gr = bench.kind_bytes_per_step(wl, 256, "gradred")
    assert gr == 2 * T * (2 * m + 2 * m)      # up: R side 11008; down: P side 11008
    bd = bench.kind_bytes_per_step(wl, 256, "blockdiag")
    # b = 256: the R transform stays a separate pass (2 * mm)
    per = lambda nn, mm, fm, fn: T * (2 * nn + 2 * mm + (3 if fm else 2) * mm + (3 if fn else 2) * nn
                                      + 2 * nn) * 2
    assert bd == per(n, m, False, True) + per(m, n, True, False)


def test_gather_inside_the_transform_for_narrow_sides():
    # off by default; with the bound at 1536: bf16 sides of 256 to 1536
    # features, b <= 128
    wl = synth.WORKLOADS["d1024_block"]
    assert not bench.gather_in_transform(wl, 1024, 64)
    old = bench.FUSED_GATHER_MAX
    bench.FUSED_GATHER_MAX = 1536
    try:
        _check_d1024_fused_accounting(wl)
    finally:
        bench.FUSED_GATHER_MAX = old


def _check_d1024_fused_accounting(wl):
    assert bench.gather_in_transform(wl, 1024, 64) and bench.gather_in_transform(wl, 1536, 128)
    assert not bench.gather_in_transform(wl, 2816, 64)
    assert not bench.gather_in_transform(wl, 1024, 256)
    assert not bench.gather_in_transform(synth.WORKLOADS["fp32_256"], 256, 32)
    assert not bench.gather_in_transform(wl, 200, 64)
    # d1024 (recompute, T = 32768): P sides of 1024 gather X -> u inside the
    # forward and the recompute transform (6 B each), down's 2816-wide P side
    # keeps its passes; R sides of 1024 gather dY inside the backward transform
    t = wl.tokens
    n_f = 6 * 1024             # fused P sides (q, k, v, o, gate, up)
    n_s = 2816                 # separate P side (down)
    m_f = 4 * 1024 + 1024      # fused R sides (q, k, v, o, down)
    m_s = 2 * 2816             # separate R sides (gate, up)
    assert bench.kind_bytes_per_step(wl, 64, "gather") == 4 * t * (n_f + 3 * n_s + m_f + 2 * m_s)
    pd = lambda n: bench.p_in_dgrad(t, n, 64)
    assert not pd(1024) and not pd(2816)
    # blockdiag: fwd P (6 or 4 B), R in the GEMM, bwd R (6 B) and P (6 B), recompute P (6 or 4 B)
    want = 2 * t * (3 * n_f + 2 * n_s + 3 * (m_f + m_s) + 3 * (n_f + n_s) + 3 * n_f + 2 * n_s)
    assert bench.kind_bytes_per_step(wl, 64, "blockdiag") == want
    # with the bound at 0 every side keeps its gather passes
    old = bench.FUSED_GATHER_MAX
    try:
        bench.FUSED_GATHER_MAX = 0
        assert bench.kind_bytes_per_step(wl, 64, "gather") == 4 * t * (3 * (n_f + n_s) + 2 * (m_f + m_s))
    finally:
        bench.FUSED_GATHER_MAX = old


def test_concurrent_groups_follow_the_block_structure():
    # q, k, v and gate, up read the same block input; o and down stand alone
    assert bench.concurrent_groups(synth.WORKLOADS["llama60m_block"]) == [[0, 1, 2], [3], [4, 5], [6]]
    assert bench.concurrent_groups(synth.WORKLOADS["d2048_block"]) == [[0, 1, 2], [3], [4, 5], [6]]
    assert bench.concurrent_groups(synth.WORKLOADS["d4096_ffn"]) == [[0], [1]]
    assert bench.concurrent_groups(synth.WORKLOADS["fp32_256"]) == [[0]]

    class A:
        mode, weight, optimizer, gpus, graph, concurrent = "cayley", "dense", "none", 1, "auto", "on"
    wl = synth.WORKLOADS["llama60m_block"]
    assert bench.workload_config(wl, 32, A)["linear_order"] == "q|k|v o gate|up down"
    A.concurrent = "off"
    assert bench.workload_config(wl, 32, A)["linear_order"] == "q k v o gate up down"


@pytest.mark.parametrize("key", ["llama60m_block", "d1024_block", "d2048_block", "d4096_ffn"])
@pytest.mark.parametrize("b", [32, 64, 128, 256, 512])
def test_class_flops_partition_the_step_flops(key, b):
    # the GEMM classes (with the transforms in their epilogues), the block
    # transforms and the separate reductions together are the step's
    # algorithmic flops, whatever the placement rules decide
    wl = synth.WORKLOADS[key]
    parts = sum(bench.kind_flops_per_step(wl, b, k)
                for k in ("gemm_fwd", "gemm_dgrad", "blockdiag", "gradred"))
    assert parts == pytest.approx(bench.step_flops(wl, b), rel=1e-12)
