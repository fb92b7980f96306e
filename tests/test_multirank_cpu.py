"""Data-parallel sharding of the layer over tokens, on CPU ranks (gloo).

The layer shards by tokens: every rank holds W0', the permutation seeds and
the generators, runs forward/backward on its own tokens, and the only
exchange is a sum all-reduce of the packed generator gradients ("POET-X:
Memory-efficient LLM Training by Scaling Orthogonal Transformation",
Resultaten: plain data parallelism with no model sharding).  Here each rank
computes its shard's gradients with the oracle and the all-reduced sum must
equal the single-process gradient over all tokens.  A second case has one
rank raise before the collective and checks that the survivor sees an error
rather than hanging.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle as O

SPEC = O.LayerSpec(m=12, n=10, b_R=4, b_P=5, seed_R=21, seed_P=22)
T = 10


def _inputs():
    r = np.random.default_rng(42)
    W0 = r.standard_normal((SPEC.m, SPEC.n)) * 0.3
    X = r.standard_normal((T, SPEC.n))
    dY = r.standard_normal((T, SPEC.m))
    gR = r.standard_normal(O.packed_length(SPEC.m, SPEC.b_R)) * 0.1
    gP = r.standard_normal(O.packed_length(SPEC.n, SPEC.b_P)) * 0.1
    return W0, X, dY, gR, gP


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, outdir, fail_rank):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import datetime
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=20))
    try:
        W0, X, dY, gR, gP = _inputs()
        lo, hi = rank * T // world, (rank + 1) * T // world
        if rank == fail_rank:
            raise RuntimeError("planted rank failure before the exchange")
        _, dgR, dgP, _ = O.backward(SPEC, W0, X[lo:hi], dY[lo:hi], gR, gP)
        buf = torch.from_numpy(np.concatenate([dgR, dgP]))
        dist.all_reduce(buf, op=dist.ReduceOp.SUM)
        np.save(os.path.join(outdir, f"rank{rank}.npy"), buf.numpy())
    except Exception as e:       # record what the rank saw
        with open(os.path.join(outdir, f"rank{rank}.err"), "w") as f:
            f.write(repr(e))
    finally:
        try:
            dist.destroy_process_group()
        except Exception:
            pass


def test_token_sharded_allreduce_matches_full(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path), -1),
                       nprocs=world, start_method="spawn", join=True)
    W0, X, dY, gR, gP = _inputs()
    _, dgR, dgP, _ = O.backward(SPEC, W0, X, dY, gR, gP)
    full = np.concatenate([dgR, dgP])
    for r in range(world):
        got = np.load(tmp_path / f"rank{r}.npy")
        assert np.abs(got - full).max() < 1e-12


def test_failed_rank_surfaces_as_error_not_hang(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path), 1),
                       nprocs=world, start_method="spawn", join=True)
    assert (tmp_path / "rank1.err").exists()
    # rank 0 must not have produced a reduced result: its collective failed
    assert not (tmp_path / "rank0.npy").exists()
    assert (tmp_path / "rank0.err").exists()
