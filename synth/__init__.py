"""Seeded synthetic inputs for the POET-X layer workloads.

This module is shared by the fp64 oracle tests, the GPU parity tests and the
benchmark.  It holds only shapes and random-number recipes: none of the
layer's arithmetic lives here.  Both sides of every parity test draw their
inputs from these functions, so they see identical values.

Workload shapes follow the LLaMA-shaped linears that "POET-X: Memory-efficient
LLM Training by Scaling Orthogonal Transformation" (gist.science summary,
"Resultaten") trains; the pages measure on C4 with Llama 3B/8B/13B, which are
not used here: seeded Gaussian stand-ins of the same shapes replace them.

Random streams
--------------
Matrices are generated in chunks of ``CHUNK_ROWS`` rows; chunk ``c`` of a
tensor with seed ``s`` is ``numpy.random.default_rng([s, c])`` drawing a
float32 standard normal block of ``CHUNK_ROWS x cols``.  Row ``t`` therefore
depends only on (seed, t, cols), never on the total row count, so a test can
regenerate a sampled row of a 65536-token input without building the rest.
"""
from __future__ import annotations

import dataclasses
import os
from typing import List, Optional, Sequence

import numpy as np

CHUNK_ROWS = 256

# Per-linear seed bases: linear l of a workload uses base + l.
SEED_W0, SEED_X, SEED_DY, SEED_GEN_R, SEED_GEN_P, SEED_PERM_R, SEED_PERM_P = (
    1000, 2000, 3000, 4000, 5000, 6000, 7000)
# Seeds of the fresh permutations that a merge moves a layer to.
SEED_MERGE_R, SEED_MERGE_P = 8000, 9000

STD_W0 = 0.02     # W0 ~ N(0, 0.02^2)
STD_ACT = 1.0     # X, dY ~ N(0, 1)
STD_GEN = 0.01    # packed skew generators ~ N(0, 0.01^2)


@dataclasses.dataclass(frozen=True)
class Linear:
    """One linear map n -> m (W0 is m x n) inside a workload."""
    name: str
    n: int
    m: int


@dataclasses.dataclass(frozen=True)
class Workload:
    key: str
    description: str
    linears: Sequence[Linear]
    tokens: int
    block_sizes: Sequence[int]     # b values swept (b_R = b_P = b)
    dtype: str                     # "fp32" or "bf16"
    recompute: bool                # activation recompute in backward
    merge_each_step: bool


def _block(d: int, f: int) -> List[Linear]:
    return [Linear("q", d, d), Linear("k", d, d), Linear("v", d, d),
            Linear("o", d, d), Linear("gate", d, f), Linear("up", d, f),
            Linear("down", f, d)]


WORKLOADS = {
    "fp32_256": Workload(
        "fp32_256", "single POET-X linear 256->256, fp32, b=32, 512 tokens",
        [Linear("lin", 256, 256)], 512, [32], "fp32", False, False),
    "llama60m_block": Workload(
        "llama60m_block", "LLaMA-60M-shaped block (q,k,v,o 512; gate/up 512->1376; "
        "down 1376->512), bf16, b=32, 8192 tokens",
        _block(512, 1376), 8192, [32], "bf16", False, False),
    "d1024_block": Workload(
        "d1024_block", "d=1024 block (gate/up 1024->2816), bf16, b=64, 32768 tokens, "
        "activation recompute",
        _block(1024, 2816), 32768, [64], "bf16", True, False),
    "d2048_block": Workload(
        "d2048_block", "d=2048 1B-class block (gate/up 2048->5632), bf16, b=128/256, "
        "65536 tokens, merge every step",
        _block(2048, 5632), 65536, [128, 256], "bf16", False, True),
    "d4096_ffn": Workload(
        "d4096_ffn", "d=4096 FFN linears 4096->11008 and 11008->4096, bf16, 65536 tokens, "
        "b in {32..512}, activation recompute",
        [Linear("up", 4096, 11008), Linear("down", 11008, 4096)], 65536,
        [32, 64, 128, 256, 512], "bf16", True, False),
}


def rows(seed: int, t0: int, t1: int, cols: int, std: float) -> np.ndarray:
    """Rows [t0, t1) of the seeded N(0, std^2) matrix with ``cols`` columns (float32)."""
    if t1 <= t0:
        return np.zeros((0, cols), dtype=np.float32)
    out = np.empty((t1 - t0, cols), dtype=np.float32)
    c0, c1 = t0 // CHUNK_ROWS, (t1 - 1) // CHUNK_ROWS

    def fill(c):
        rng = np.random.default_rng([seed, c])
        blk = rng.standard_normal((CHUNK_ROWS, cols), dtype=np.float32)
        lo, hi = max(t0, c * CHUNK_ROWS), min(t1, (c + 1) * CHUNK_ROWS)
        out[lo - t0:hi - t0] = blk[lo - c * CHUNK_ROWS:hi - c * CHUNK_ROWS]
        if std != 1.0:
            out[lo - t0:hi - t0] *= np.float32(std)

    nchunks = c1 - c0 + 1
    if nchunks >= 16:
        # chunks are independent streams, so threads change nothing in the values
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(max_workers=min(32, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, range(c0, c1 + 1)))
    else:
        for c in range(c0, c1 + 1):
            fill(c)
    return out


def matrix(seed: int, nrows: int, cols: int, std: float) -> np.ndarray:
    return rows(seed, 0, nrows, cols, std)


def vector(seed: int, length: int, std: float) -> np.ndarray:
    """A seeded N(0, std^2) float32 vector (used for packed generators)."""
    rng = np.random.default_rng([seed, 0])
    v = rng.standard_normal(length, dtype=np.float32)
    return v * np.float32(std) if std != 1.0 else v


def round_to(a: np.ndarray, dtype: str):
    """Round a float32 array to the workload dtype; returns a torch CPU tensor.

    The oracle consumes ``round_to(...).double()``, i.e. exactly the values the
    GPU path receives.
    """
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    if dtype == "bf16":
        return t.to(torch.bfloat16)
    if dtype == "fp32":
        return t.clone()
    raise ValueError(dtype)


@dataclasses.dataclass
class LayerInputs:
    """All seeded inputs of one linear: weights, activations, generators, seeds."""
    W0: object          # torch CPU tensor m x n (dtype)
    X: object           # T x n
    dY: object          # T x m
    genR: object        # torch float32, packed
    genP: object
    seed_R: int
    seed_P: int


def layer_inputs(lin: Linear, index: int, tokens: int, dtype: str,
                 gen_len_R: int, gen_len_P: int,
                 t0: int = 0, t1: Optional[int] = None) -> LayerInputs:
    """Inputs of linear ``index`` of a workload; tokens [t0, t1) of X and dY.

    ``gen_len_R``/``gen_len_P`` are the packed generator lengths, which the
    caller computes from the layer geometry.
    """
    import torch
    t1 = tokens if t1 is None else t1
    W0 = round_to(matrix(SEED_W0 + index, lin.m, lin.n, STD_W0), dtype)
    X = round_to(rows(SEED_X + index, t0, t1, lin.n, STD_ACT), dtype)
    dY = round_to(rows(SEED_DY + index, t0, t1, lin.m, STD_ACT), dtype)
    genR = torch.from_numpy(vector(SEED_GEN_R + index, gen_len_R, STD_GEN))
    genP = torch.from_numpy(vector(SEED_GEN_P + index, gen_len_P, STD_GEN))
    return LayerInputs(W0, X, dY, genR, genP, SEED_PERM_R + index, SEED_PERM_P + index)
