#!/usr/bin/env python
"""Benchmark of the POET-X orthogonal-equivalence linear layer on B300.

One step = the whole hot path over one batch of synthetic tokens for every
linear of the workload: build the blocks from the generators (permutations
plus Cayley builder), forward (gather, P blocks, W0' GEMM, R blocks,
scatter), backward (gather, R^T blocks, per-block token reductions, dgrad
GEMM, P^T blocks, scatter, Cayley backward and packing) and, where the
workload says so, the merge W0 <- R W0 P under fresh permutations.

Prints one JSON line.  `value` is whole-job tokens/s with inputs resident in
HBM; `e2e` is the same metric through the C ABI from pinned host buffers,
host<->device copies included; `roofline` covers the kernel class with the
largest device time; `cpu_baseline` times the fp64 oracle on a bounded token
sample on this host's cores.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload KEY] [--b B]
    python bench.py --impl reference ...      # the fp64 oracle, timed on host cores
"""
from __future__ import annotations

import argparse
import atexit
import datetime
import hashlib
import json
import tempfile
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = ("POET-X linear fwd+bwd tokens/s and TFLOP/s (fraction of bf16 peak), 1×B300")
DEFAULT_WORKLOAD = "d2048_block"
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="poetx", choices=["poetx", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--b", type=int, default=None, help="block size (default: first of the workload)")
    ap.add_argument("--mode", default="cayley", choices=["cayley", "neumann"])
    ap.add_argument("--graph", default="auto", choices=["auto", "on", "off"],
                    help="replay each timed step from a CUDA graph (auto: for workloads "
                         "without a per-step merge, whose new permutations come from the host)")
    ap.add_argument("--optimizer", default="none", choices=["none", "adamw"],
                    help="end each layer's step with an AdamW update of its generators")
    ap.add_argument("--weight", default="dense", choices=["dense", "int8"],
                    help="storage of the base weight: layer dtype, or int8 rows (POET-XQ)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-overhead", action="store_true",
                    help="skip the plain-bf16-linear comparison and the per-linear breakdown")
    ap.add_argument("--cpu-tokens", type=int, default=1536,
                    help="oracle sample tokens per linear (the cpu_baseline leg and each step of "
                         "the reference arm)")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the other workloads (measured in child processes after the main line)")
    ap.add_argument("--extra-steps", type=int, default=10,
                    help="timed steps of each other workload (3 warm-up steps each)")
    ap.add_argument("--tokens", type=int, default=None,
                    help="override the workload's token count (small profiling cases only)")
    ap.add_argument("--clock-log", default=None,
                    help="keep the raw nvidia-smi clock samples of the timed region in this file")
    ap.add_argument("--concurrent", default="on", choices=["on", "off"],
                    help="run the linears a block applies to one input (q, k, v; gate, up) "
                         "on parallel streams")
    ap.add_argument("--fused-gather-max", type=int, default=-1,
                    help="widest side whose column permutation runs inside its block transform "
                         "(0, the library's default: separate gather passes)")
    ap.add_argument("--builds-only", action="store_true",
                    help="time only the block builds (poetx_blocks_build) of each linear, "
                         "in isolation, and print one JSON line")
    return ap.parse_args()


# ---------------------------------------------------------------- workload arithmetic

def block_square_sum(d: int, b: int) -> int:
    full, last = d // b, d % b
    return full * b * b + last * last


def step_flops(wl, b: int) -> float:
    """Algorithmic tensor flops of one step over all linears.

    fwd: 2Tmn (GEMM) + 2T(sum b_P^2 + sum b_R^2) (block transforms);
    bwd: 2Tmn (dgrad) + 4T sum b_R^2 (R^T transform and dB_R) + 4T sum b_P^2;
    recompute adds 2Tmn + 2T sum b_P^2.  Builder, Cayley backward and merge
    are fp32 CUDA-core work and are not counted here.
    """
    T = wl.tokens
    f = 0.0
    for lin in wl.linears:
        sR, sP = block_square_sum(lin.m, b), block_square_sum(lin.n, b)
        f += 4.0 * T * lin.m * lin.n + 6.0 * T * (sR + sP)
        if wl.recompute:
            f += 2.0 * T * lin.m * lin.n + 2.0 * T * sP
    return f


# The library's placement of the block transforms of a bf16 layer (as its
# forward and backward decide): for b <= 128 the forward R transform runs in
# the forward GEMM's epilogue, and the backward P-side transform and token
# reduction run in the dgrad's epilogue where that GEMM is the single-CTA
# engine (outputs narrower than 1024, or fewer than 256 tokens) or its output
# is at most 32 MB.
def r_in_gemm(b: int) -> bool:
    return b <= 128


def p_in_dgrad(T: int, n: int, b: int) -> bool:
    pair = n >= 1024 and T >= 256
    return b <= 128 and (not pair or T * n * 2 <= (32 << 20))


# Widest bf16 side (b <= 128) whose column permutation runs inside its block
# transform: the forward X -> u -> v in one kernel and the backward dY -> dz
# inside the R-side transform + reduction (off by default in the library; the
# --fused-gather-max flag sets both).
FUSED_GATHER_MAX = 0


def gather_in_transform(wl, d: int, b: int) -> bool:
    return wl.dtype == "bf16" and b <= 128 and -(-d // 128) <= 148 and 256 <= d <= FUSED_GATHER_MAX


def concurrent_groups(wl):
    """Groups of consecutive linears that read the same block input in a
    transformer block (q, k, v and gate, up); the others stand alone."""
    names = [lin.name for lin in wl.linears]
    sets = ({"q", "k", "v"}, {"gate", "up"})
    groups, i = [], 0
    while i < len(names):
        g = [i]
        for st in sets:
            if names[i] in st:
                while i + len(g) < len(names) and names[i + len(g)] in st:
                    g.append(i + len(g))
        groups.append(g)
        i += len(g)
    return groups


def use_concurrent(args, wl) -> bool:
    """Parallel streams for the grouped linears (measured on B300, 20-step
    means, two runs each: LLaMA-60M 0.530 -> 0.466 ms per step, d1024 3.95-3.99
    -> 3.70-3.78 ms, d2048 16.62 -> 16.41-16.50 ms), unless turned off."""
    return args.concurrent != "off"


def gemm_flops_per_step(wl, kind: str, b: int = 0) -> float:
    """Flops of a GEMM class: the GEMMs, plus the block-transform (and
    reduction) flops that run in their epilogues when b is given."""
    T = wl.tokens
    f = 0.0
    for lin in wl.linears:
        sR = block_square_sum(lin.m, b) if b else 0
        sP = block_square_sum(lin.n, b) if b else 0
        if kind == "gemm_fwd":
            f += 2.0 * T * lin.m * lin.n * (2 if wl.recompute else 1)
            if b and wl.dtype == "bf16" and r_in_gemm(b):
                f += 2.0 * T * sR
        elif kind == "gemm_dgrad":
            f += 2.0 * T * lin.m * lin.n
            if b and wl.dtype == "bf16" and p_in_dgrad(T, lin.n, b):
                f += 4.0 * T * sP
    return f


def kind_flops_per_step(wl, b: int, kind: str) -> float:
    T = wl.tokens
    if kind in ("gemm_fwd", "gemm_dgrad"):
        return gemm_flops_per_step(wl, kind, b)
    f = 0.0
    for lin in wl.linears:
        sR, sP = block_square_sum(lin.m, b), block_square_sum(lin.n, b)
        pd = wl.dtype == "bf16" and p_in_dgrad(T, lin.n, b)
        rg = wl.dtype == "bf16" and r_in_gemm(b)
        if kind == "blockdiag":
            # fwd P (and R unless in the GEMM), bwd R^T (and P^T unless in the
            # dgrad), recompute P
            f += 2.0 * T * (sP + (0 if rg else sR) + sR + (0 if pd else sP)
                            + (sP if wl.recompute else 0))
        elif kind == "gradred":
            f += 2.0 * T * (sR + (0 if pd else sP))
    return f


def kind_bytes_per_step(wl, b: int, kind: str) -> float:
    """Algorithmic DRAM bytes of one step for the memory-bound kernel classes
    (each T x d activation operand read or written once per pass).

    gather: X -> u and z -> Y in the forward, dY -> dz and du -> dX in the
    backward, plus X -> u again when u is recomputed.  blockdiag: forward
    u -> v, and h -> z unless the R transform runs in the forward GEMM
    (b <= 128); backward dz -> dh and dv -> du, which for b <= 128 also read h
    and u (the fused transform + reduction), the latter unless it runs in the
    dgrad's epilogue; plus u -> v when recomputing.  gradred (sides whose
    reduction is not fused): dz^T h and dv^T u read two operands.  The fused
    kernels are used for b <= 128 and, when their grid fills the GPU, for
    b = 256 (as the library decides).  Where the permutation runs inside the
    transform (gather_in_transform), X -> u -> v reads X once and writes u
    and v (6 B per element instead of 4 + 4), and dY -> dz -> dh reads dY in
    place of dz (the gather pass disappears).
    """
    T = wl.tokens
    e = 2 if wl.dtype == "bf16" else 4
    r = 1 if wl.recompute else 0
    sms = 148

    def fused(d):  # the library's choice of the fused transform + reduction for one side
        if b <= 128:
            return -(-d // 128) <= sms
        if b == 256:
            cps = 2 * -(-d // 256)
            return cps <= sms and 5 * (sms // cps) * cps >= 4 * sms
        return False

    by = 0
    for lin in wl.linears:
        n, m = lin.n, lin.m
        fm, fn = fused(m), fused(n)
        pd = wl.dtype == "bf16" and p_in_dgrad(T, n, b)
        rg = wl.dtype == "bf16" and r_in_gemm(b)
        gn, gm = gather_in_transform(wl, n, b), gather_in_transform(wl, m, b)
        if kind == "gather":
            by += 2 * T * ((1 if gn else 2 + r) * n + (1 if gm else 2) * m) * e
        elif kind == "blockdiag":
            bwd = (3 if fm else 2) * m + (0 if pd else (3 if fn else 2) * n)
            pfwd = 3 if gn else 2
            by += T * (pfwd * n + (0 if rg else 2 * m) + bwd + pfwd * n * r) * e
        elif kind == "gradred":
            by += T * ((0 if fm else 2) * m + (0 if (fn or pd) else 2) * n) * e
    return float(by)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"],
                    bf16_sustained=d["bf16_tflops_sustained"], source="measured")
    return dict(hbm=6400.0, bf16=1800.0, bf16_sustained=1400.0, source="fallback")


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "orthogonal_equivalence_reparameterized_poetx_b300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh")):
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(kind: str, workload: str, b: int):
    """DRAM bytes per launch of `kind` from a committed ncu summary, or None
    when the kernels changed since the counters were taken."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        d = json.load(f)
    if d.get("kernel_source_hash") != kernel_source_hash():
        return None
    e = d.get("entries", {}).get(f"{workload}/b{b}/{kind}")
    return None if e is None else e.get("bytes_per_launch")


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling every 20 ms, started ahead of the timed region (so
    its start-up falls outside it); the summary keeps the samples whose
    timestamps fall inside the region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,timestamp")

    def __init__(self, gpu_index: int, log_path=None):
        """log_path: keep the raw samples there; default a temporary file,
        removed once the samples are summarised."""
        self.idx = gpu_index
        self.proc = None
        self.keep = log_path is not None
        if log_path is None:
            fd, log_path = tempfile.mkstemp(prefix="poetx_clocks_", suffix=".csv")
            os.close(fd)
        self.path = log_path

    def start(self):
        try:
            if os.path.dirname(self.path):
                os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
            atexit.register(self._end)  # never outlive this process
        except Exception:
            self.proc = None

    def _end(self):
        if self.proc is not None and self.proc.poll() is None:
            self.proc.kill()

    def stop(self, t0=None, t1=None):
        """Ends sampling; summarises the samples taken between host times t0
        and t1 (seconds since the epoch), widened by 0.1 s on each side when
        the region is shorter than the sampling interval."""
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        with open(self.path) as f:
            lines = f.readlines()
        summary = summarise_clock_samples(lines, t0, t1)
        if summary is None and t0 is not None:
            summary = summarise_clock_samples(lines, t0 - 0.1, t1 + 0.1)
            if summary is not None:
                summary["window"] = "timed region +- 0.1 s (shorter than the sampling interval)"
        if not self.keep:
            try:
                os.remove(self.path)
            except OSError:
                pass
        return summary


def sample_time(stamp: str):
    """Seconds since the epoch of an nvidia-smi timestamp
    ('YYYY/MM/DD HH:MM:SS.mmm', local time), or None."""
    try:
        return datetime.datetime.strptime(stamp.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
    except ValueError:
        return None


def summarise_clock_samples(lines, t0=None, t1=None):
    """Median SM clock, maximum clock, sample count and the throttle reasons
    seen active, from `nvidia-smi --query-gpu=<ClockSampler.FIELDS>
    --format=csv,noheader,nounits` lines; None without a usable sample.
    With t0 and t1 (seconds since the epoch) only samples whose timestamp
    lies in [t0, t1] count.  Lines that are not complete samples (a partial
    last line, [N/A] clocks) are skipped."""
    sm, smax, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in lines:
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 8:
            continue
        try:
            clk, clk_max = float(parts[0]), float(parts[1])
        except ValueError:
            continue
        if t0 is not None:
            ts = sample_time(parts[8]) if len(parts) > 8 else None
            if ts is None or ts < t0 or ts > t1:
                continue
        sm.append(clk)
        smax.append(clk_max)
        for nm, v in zip(names, parts[4:8]):
            if v.lower().startswith("active"):
                reasons.add(nm)
    if not sm:
        return None
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
            "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------- the fp64 oracle as baseline

def oracle_sample(wl, b: int, tokens: int, mode: str):
    """Times the oracle (fwd+bwd incl. block build) on `tokens` tokens of every
    linear; returns (seconds, threads)."""
    import oracle as O
    try:
        import threadpoolctl
        threads = max(i["num_threads"] for i in threadpoolctl.threadpool_info())
    except Exception:
        threads = os.cpu_count()
    total = 0.0
    for li, lin in enumerate(wl.linears):
        spec = O.LayerSpec(lin.m, lin.n, b, b, synth.SEED_PERM_R + li, synth.SEED_PERM_P + li,
                           "neumann" if mode == "neumann" else "exact", 3)
        inp = synth.layer_inputs(lin, li, wl.tokens, wl.dtype, O.packed_length(lin.m, b),
                                 O.packed_length(lin.n, b), t0=0, t1=tokens)
        args = [inp.W0.double().numpy(), inp.X.double().numpy(), inp.dY.double().numpy(),
                inp.genR.double().numpy(), inp.genP.double().numpy()]
        t0 = time.perf_counter()
        O.backward(spec, *args)
        total += time.perf_counter() - t0
    return total, threads


def run_reference(args, wl, b, rank):
    if rank != 0:
        return
    for _ in range(args.warmup):
        oracle_sample(wl, b, args.cpu_tokens, args.mode)
    times = []
    threads = None
    for _ in range(args.steps):
        t, threads = oracle_sample(wl, b, args.cpu_tokens, args.mode)
        times.append(t)
    tot = sum(times)
    tps = args.cpu_tokens * args.steps / tot
    sample = (f"{len(wl.linears)} linears x {args.cpu_tokens} tokens per step (of {wl.tokens}), "
              f"fwd+bwd with block build, fp64 numpy; merge not timed (the cpu_baseline sample)")
    line = {
        "impl": "reference", "metric": METRIC, "value": tps, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(wl, b, args),
        "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def graph_replay(wl, args) -> bool:
    """Whether the timed steps replay a captured CUDA graph: on request, or
    (auto) for workloads without a per-step merge, whose new permutations
    come from the host, and without an optimizer step, whose step count
    comes from the host, on one GPU (with several ranks the per-layer
    gradient sums run eagerly on their own stream)."""
    return args.graph == "on" or (args.graph == "auto" and not wl.merge_each_step
                                  and args.optimizer == "none" and args.gpus == 1)


def workload_config(wl, b, args):
    return {
        "workload": wl.key, "description": wl.description,
        "linears": [f"{l.name}:{l.n}->{l.m}" for l in wl.linears],
        "tokens": wl.tokens, "b": b, "mode": args.mode, "weight": args.weight,
        "optimizer": args.optimizer,
        "recompute": wl.recompute,
        "merge_each_step": wl.merge_each_step,
        "l2": "inputs larger than L2 (activations of all linears, several GB per step)",
        "parallelism": f"dp{args.gpus}",
        "cuda_graph": graph_replay(wl, args),
        # linears joined by "|" run on parallel streams within the step
        "linear_order": " ".join("|".join(wl.linears[i].name for i in g) for g in
                                 (concurrent_groups(wl) if use_concurrent(args, wl)
                                  else [[i] for i in range(len(wl.linears))])),
    }


# ---------------------------------------------------------------- the CUDA path

def run_builds_only(args, wl, b, px, torch, dev):
    """Isolated device time of poetx_blocks_build (both sides of a layer) per
    linear: CUDA events around K builds after W warm-up builds."""
    per = []
    for li, lin in enumerate(wl.linears):
        desc = px.make_desc(lin.m, lin.n, b, b, synth.SEED_PERM_R + li, synth.SEED_PERM_P + li,
                            dtype=wl.dtype, mode=args.mode, weight=args.weight)
        lr, lp = px.poetx_gen_length(lin.m, b), px.poetx_gen_length(lin.n, b)
        g = np.random.default_rng([synth.SEED_GEN_R + li, 0])
        genR = torch.from_numpy((g.standard_normal(lr) * synth.STD_GEN).astype(np.float32)).to(dev)
        genP = torch.from_numpy((g.standard_normal(lp) * synth.STD_GEN).astype(np.float32)).to(dev)
        params = torch.empty(px.poetx_params_size(desc), dtype=torch.uint8, device=dev)
        px.poetx_params_build(desc, genR, genP, params)
        for _ in range(args.warmup):
            px.poetx_blocks_build(desc, genR, genP, params)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record()
        for _ in range(args.steps):
            px.poetx_blocks_build(desc, genR, genP, params)
        e1.record()
        torch.cuda.synchronize(dev)
        per.append({"linear": f"{lin.name}:{lin.n}->{lin.m}", "ms": e0.elapsed_time(e1) / args.steps})
    st = px.poetx_device_status(reset=True)
    print(json.dumps({"metric": "block build time per linear (both sides, isolated)", "unit": "ms",
                      "higher_is_better": False, "steps": args.steps, "warmup": args.warmup,
                      "config": {"workload": wl.key, "b": b, "mode": args.mode, "dtype": wl.dtype},
                      "per_linear": per, "device_status": px.poetx_status_string(st)}))


def main():
    args = parse()
    wl = synth.WORKLOADS[args.workload]
    if args.tokens:
        import dataclasses
        wl = dataclasses.replace(wl, tokens=args.tokens)
    b = args.b or wl.block_sizes[0]
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, wl, b, rank)
        return

    import torch
    import orthogonal_equivalence_reparameterized_poetx_b300 as px

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    px.poetx_set_fused_gather_max_features(args.fused_gather_max)
    if args.fused_gather_max >= 0:
        global FUSED_GATHER_MAX
        FUSED_GATHER_MAX = args.fused_gather_max
    if args.builds_only:
        run_builds_only(args, wl, b, px, torch, dev)
        return
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    # the forward/backward stream runs at high priority and the per-layer
    # build/merge side streams at the default (lowest) priority, so the block
    # scheduler serves the critical path first when both have work queued
    lo, hi = torch.cuda.Stream.priority_range()
    stream = torch.cuda.Stream(dev, priority=hi)
    torch.cuda.set_stream(stream)
    dt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    T = wl.tokens

    # ---- resident state and inputs (seeded host generation, copied once)
    layers = []
    ws_bytes = 0
    for li, lin in enumerate(wl.linears):
        desc = px.make_desc(lin.m, lin.n, b, b, synth.SEED_PERM_R + li, synth.SEED_PERM_P + li,
                            dtype=wl.dtype, mode=args.mode, weight=args.weight)
        lr, lp = px.poetx_gen_length(lin.m, b), px.poetx_gen_length(lin.n, b)
        inp = synth.layer_inputs(lin, li, T, wl.dtype, lr, lp)
        st = dict(lin=lin, desc=desc, lr=lr, lp=lp)
        st["params"] = torch.empty(px.poetx_params_size(desc), dtype=torch.uint8, device=dev)
        if wl.merge_each_step:
            # the next step's blocks are built into a second buffer while the
            # merge still reads the current one
            st["params_next"] = torch.empty_like(st["params"])
        if args.weight == "int8":   # int8 codes and row scales, poetx_weight_size bytes
            st["W0p"] = torch.empty(px.poetx_weight_size(desc), dtype=torch.uint8, device=dev)
        else:
            st["W0p"] = torch.empty(lin.m, lin.n, dtype=dt, device=dev)
        st["genR"], st["genP"] = inp.genR.to(dev), inp.genP.to(dev)
        st["X"], st["dY"] = inp.X.to(dev), inp.dY.to(dev)
        st["Y"] = torch.empty(T, lin.m, dtype=dt, device=dev)
        st["dX"] = torch.empty(T, lin.n, dtype=dt, device=dev)
        # stored-activation workloads keep h and the permuted input u of the
        # forward; recompute workloads keep neither
        st["h"] = None if wl.recompute else torch.empty(T, lin.m, dtype=dt, device=dev)
        st["u"] = None if wl.recompute else torch.empty(T, lin.n, dtype=dt, device=dev)
        st["dgR"] = torch.empty(lr, dtype=torch.float32, device=dev)
        st["dgP"] = torch.empty(lp, dtype=torch.float32, device=dev)
        if args.optimizer == "adamw":   # AdamW moments of the packed generators
            st["mom"] = [torch.zeros(x, dtype=torch.float32, device=dev) for x in (lr, lr, lp, lp)]
        W0 = inp.W0.to(dev)
        px.poetx_params_build(desc, st["genR"], st["genP"], st["params"], stream)
        px.poetx_weight_premerge(desc, st["params"], W0, st["W0p"], stream)
        ws_bytes = max(ws_bytes, px.poetx_workspace_size(desc, T),
                       px.poetx_merge_workspace_size(desc))
        layers.append(st)
        del inp, W0
    workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    # linears that a transformer block runs on the same input (q, k, v; gate,
    # up) are independent: with --concurrent their passes run on parallel
    # streams, each with its own workspace
    groups = concurrent_groups(wl) if use_concurrent(args, wl) else [[i] for i in range(len(layers))]
    sched = {"groups": groups}   # the schedule step() runs
    width = max(len(g) for g in groups)
    workspaces = [workspace] + [torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
                                for _ in range(width - 1)]
    par_streams = [stream] + [torch.cuda.Stream(dev, priority=hi) for _ in range(width - 1)]
    torch.cuda.synchronize(dev)

    step_counter = [0]
    # Per-layer work that depends only on that layer (rebuilding its blocks
    # from the generators, and the merge) runs on one side stream per layer,
    # ordered by per-layer events: layer l's merge starts as soon as its own
    # backward is done and its next build follows on the same side stream,
    # while the main stream runs the other layers' forward and backward.
    # Each merge has its own scratch so concurrent merges do not share it.
    side = [torch.cuda.Stream(dev, priority=lo) for _ in layers]
    side_build = [torch.cuda.Stream(dev, priority=lo) for _ in layers]
    merge_ws = ([torch.empty(px.poetx_merge_workspace_size(st["desc"]), dtype=torch.uint8,
                             device=dev) for st in layers] if wl.merge_each_step else None)
    bwd_done = [None] * len(layers)    # event after layer l's backward in the previous step
    # data parallel: each layer's packed gradients are summed over ranks on
    # their own stream, right after that layer's backward, while the main
    # stream runs the next layer's backward; the main stream waits for a
    # layer's sum only before its optimizer update and at the end of the step
    comm = torch.cuda.Stream(dev, priority=hi) if dist is not None else None
    merged = [0]                       # merges issued so far (for fresh seeds)

    def merge_one(li, st, ss, tag):
        nR = synth.SEED_MERGE_R + 100 * (tag + 1) + li
        nP = synth.SEED_MERGE_P + 100 * (tag + 1) + li
        px.poetx_merge(st["desc"], st["params"], st["W0p"], nR, nP, merge_ws[li], ss)
        st["desc"].seed_R, st["desc"].seed_P = nR, nP

    def build_all(tag=None):
        """Issue every layer's merge and build on its side streams; returns
        per-layer events the main stream waits on before that layer's
        forward."""
        start = torch.cuda.Event()
        start.record(stream)
        ready = []
        for li, st in enumerate(layers):
            ss = side[li]
            # a merge must follow the layer's backward of the previous step;
            # without merges the build only follows the step's start
            dep = bwd_done[li] if (wl.merge_each_step and bwd_done[li] is not None) else start
            ss.wait_event(dep)
            if not wl.merge_each_step:   # same seeds: the blocks only (device work only)
                px.poetx_blocks_build(st["desc"], st["genR"], st["genP"], st["params"], ss)
                e = torch.cuda.Event()
                e.record(ss)
                ready.append([e])
                continue
            evs = []
            if bwd_done[li] is not None:
                # the merge reads this step's blocks and rewrites W0'; it sets
                # the new seeds on the host before the next build is issued
                merge_one(li, st, ss, tag if tag is not None else step_counter[0])
                e = torch.cuda.Event()
                e.record(ss)
                evs.append(e)
            # new seeds: permutations and blocks into the other parameter
            # buffer, on the layer's second side stream, beside the merge (the
            # buffer was last read by the step before the previous one, which
            # `dep` follows)
            sb = side_build[li]
            sb.wait_event(dep)
            px.poetx_params_build(st["desc"], st["genR"], st["genP"], st["params_next"], sb)
            e = torch.cuda.Event()
            e.record(sb)
            evs.append(e)
            st["params"], st["params_next"] = st["params_next"], st["params"]
            ready.append(evs)
        return ready

    def drain_merges(tag):
        """Merges of the last step (so that every timed step includes its merges)."""
        if not wl.merge_each_step:
            return
        done = []
        for li, st in enumerate(layers):
            ss = side[li]
            ss.wait_event(bwd_done[li])
            merge_one(li, st, ss, tag)
            e = torch.cuda.Event()
            e.record(ss)
            done.append(e)
        for e in done:
            stream.wait_event(e)
        for li in range(len(layers)):
            bwd_done[li] = None

    def run_groups(groups, body):
        """Runs body(li, strm, ws) for the layers of each group: a group of one
        on the main stream, a larger group forked over the parallel streams
        (member k on par_streams[k], with workspace k) and joined again."""
        for g in groups:
            if len(g) == 1:
                body(g[0], stream, workspaces[0])
                continue
            fork = torch.cuda.Event()
            fork.record(stream)
            for k, li in enumerate(g):
                if k > 0:
                    par_streams[k].wait_event(fork)
                body(li, par_streams[k], workspaces[k])
            for k in range(1, len(g)):
                e = torch.cuda.Event()
                e.record(par_streams[k])
                stream.wait_event(e)

    def step():
        s = step_counter[0]
        reduced = []
        ready = build_all(s)

        def fwd(li, strm, ws):
            st = layers[li]
            for e in ready[li]:
                strm.wait_event(e)
            px.poetx_linear_fwd(st["desc"], st["params"], st["W0p"], st["X"], T, st["Y"], st["h"],
                                st["u"], ws, strm)

        def bwd(li, strm, ws):
            st = layers[li]
            px.poetx_linear_bwd(st["desc"], st["params"], st["W0p"], st["X"], st["dY"], st["h"],
                                st["u"], T, st["dX"], st["dgR"], st["dgP"], 0, ws, strm)
            if dist is not None:
                e = torch.cuda.Event()
                e.record(strm)
                comm.wait_event(e)
                with torch.cuda.stream(comm):
                    dist.all_reduce(st["dgR"])
                    dist.all_reduce(st["dgP"])
                red = torch.cuda.Event()
                red.record(comm)
                reduced.append(red)
                if args.optimizer == "adamw":
                    strm.wait_event(red)
            if args.optimizer == "adamw":
                mR, vR, mP, vP = st["mom"]
                px.poetx_generator_adamw(st["genR"], st["dgR"], mR, vR, st["lr"], s + 1, 1e-3,
                                         0.9, 0.999, 1e-8, 0.0, strm)
                px.poetx_generator_adamw(st["genP"], st["dgP"], mP, vP, st["lp"], s + 1, 1e-3,
                                         0.9, 0.999, 1e-8, 0.0, strm)
            e = torch.cuda.Event()
            e.record(strm)
            bwd_done[li] = e

        run_groups(sched["groups"], fwd)
        run_groups([list(reversed(g)) for g in reversed(sched["groups"])], bwd)
        for red in reduced:   # the step's gradients are summed before it ends
            stream.wait_event(red)
        # the merges of this step are issued at the start of the next step (they
        # overlap its builds and forwards); the timed region ends with drain_merges
        step_counter[0] += 1

    # clock sampling starts before the warm-up, so that nvidia-smi's start-up
    # lies outside the timed region; only samples inside it are summarised
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    gpu_idx = int(vis.split(",")[local]) if vis and vis.split(",")[local].isdigit() else local
    clocks = ClockSampler(gpu_idx, args.clock_log)
    clocks.start()
    for _ in range(args.warmup):
        step()
    drain_merges(step_counter[0])
    torch.cuda.synchronize(dev)
    if px.poetx_device_status(reset=True) != px.POETX_OK:
        clocks.stop()
        raise SystemExit("device status reported a timeout during warm-up")

    # (an optimizer step takes its step count from the host, so it stays eager)
    use_graph = graph_replay(wl, args)
    if use_graph and wl.merge_each_step:
        raise SystemExit("--graph on needs a workload without a per-step merge")
    graph = None
    if use_graph:
        # one step captured once (the side-stream builds become graph branches);
        # the library's timing events stay off inside the graph
        px.poetx_profile_enable(False)
        graph = torch.cuda.CUDAGraph()
        l0 = px.poetx_launch_count()
        with torch.cuda.graph(graph, stream=stream):
            step()
        launches_per_step = px.poetx_launch_count() - l0
        for _ in range(2):
            graph.replay()
        torch.cuda.synchronize(dev)

    # ---- timed region (device-resident inputs), without the library's
    # per-launch timing events (about 1% of a d2048 step)
    px.poetx_profile_reset()
    px.poetx_profile_enable(False)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t_region0 = time.time()
    launches0 = px.poetx_launch_count()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        if graph is not None:
            graph.replay()
        else:
            step()
    drain_merges(step_counter[0])   # the last timed step's merges
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    t_region1 = time.time()
    launches = (launches_per_step * args.steps if graph is not None
                else px.poetx_launch_count() - launches0)
    clk = clocks.stop(t_region0, t_region1)
    # per-class device times (roofline) from as many steps with the library's
    # timing events, right after the timed region: replayed from a graph when
    # the timed steps are (the events become graph nodes, so the times hold
    # no host launch gaps), else eager.  The linears run one at a time here,
    # so that each kernel's events time that kernel alone on the GPU's main
    # stream rather than its overlap with a parallel linear.
    sched["groups"] = [[i] for i in range(len(layers))]
    px.poetx_profile_reset()
    px.poetx_profile_enable(True)
    if graph is not None:
        pgraph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(pgraph, stream=stream):
            for _ in range(args.steps):
                step()
        px.poetx_profile_enable(False)
        pgraph.replay()
    else:
        for _ in range(args.steps):
            step()
        drain_merges(step_counter[0])
    torch.cuda.synchronize(dev)
    px.poetx_profile_enable(False)
    elapsed_ms = ev0.elapsed_time(ev1)
    if dist is not None:
        t = torch.tensor([elapsed_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        elapsed_ms = float(t.item())
        dist.barrier()
    status = px.poetx_device_status(reset=True)

    kinds = {}
    for k, name in enumerate(px.KIND_NAMES):
        g, ms = px.poetx_profile_read(k)
        if g:
            kinds[name] = {"groups": g, "ms": ms}
    ms_per_step = elapsed_ms / args.steps
    tokens_per_s = world * T * args.steps / (elapsed_ms / 1e3)
    flops = step_flops(wl, b)
    tflops = flops / (ms_per_step / 1e3) / 1e12
    peaks = load_peaks()

    # ---- roofline of the kernel class with the largest device time
    # candidates: kernel classes issued on the main stream one launch at a time
    # (builds and merges run concurrently on side streams, so their summed
    # group times are not wall time)
    serial = {k: v for k, v in kinds.items() if k not in ("build", "merge")}
    top = max(serial, key=lambda k: serial[k]["ms"])
    roof = None
    if top in ("gemm_fwd", "gemm_dgrad"):
        per_step = kind_flops_per_step(wl, b, top)
        launches_top = kinds[top]["groups"]
        achieved = per_step * args.steps / (kinds[top]["ms"] / 1e3) / 1e12
        roof = {"kernel": top, "bound": "tensor", "achieved": achieved,
                "peak": peaks["bf16"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16"],
                "peak_source": f"{peaks['source']} bf16 burst",
                "launches": launches_top,
                "avg_launch_ms": kinds[top]["ms"] / launches_top,
                "flops_per_launch": per_step * args.steps / launches_top,
                "traffic": measured_traffic(top, wl.key, b)}
    elif top in ("gather", "blockdiag", "gradred"):
        by = kind_bytes_per_step(wl, b, top)
        achieved = by * args.steps / (kinds[top]["ms"] / 1e3) / 1e9
        launches_top = kinds[top]["groups"]
        roof = {"kernel": top, "bound": "hbm", "achieved": achieved, "peak": peaks["hbm"],
                "unit": "GB/s", "frac": achieved / peaks["hbm"],
                "peak_source": f"{peaks['source']} HBM copy", "launches": launches_top,
                "avg_launch_ms": kinds[top]["ms"] / launches_top,
                "algorithmic_bytes_per_launch": by * args.steps / launches_top,
                "traffic": measured_traffic(top, wl.key, b)}

    line = {
        "metric": METRIC, "value": tokens_per_s, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": wl.dtype, "data": "synthetic: seeded N(0,1) activations, N(0,0.02^2) W0, "
                                   "N(0,0.01^2) packed generators",
        "config": workload_config(wl, b, args),
        "tflops": tflops, "tflops_frac_of_bf16_peak": tflops / peaks["bf16"],
        "tflops_frac_of_bf16_peak_basis": f"{peaks['source']} bf16 burst ({peaks['bf16']} TFLOP/s)",
        "tflops_frac_of_bf16_burst": tflops / peaks["bf16"],
        "tflops_frac_of_bf16_sustained": tflops / peaks["bf16_sustained"],
        "step_tflop": flops / 1e12, "roofline": roof, "kernels": kinds,
        "kernels_timing": ("library CUDA events on the launching streams over as many steps "
                           "run right after the timed region, the linears one at a time, "
                           + ("replayed from a captured graph (events as graph nodes)"
                              if graph is not None else "eager")),
        "gpu_launches": launches, "clocks": clk,
        "device_status": px.poetx_status_string(status),
    }

    # ---- per-linear times and the plain-linear comparison
    if not args.no_overhead:
        line["per_linear"], line["overhead"] = overhead_and_breakdown(
            args, wl, b, layers, workspace, stream, dev, px, torch, ms_per_step)

    # ---- end to end through the C ABI from pinned host buffers
    if not args.no_e2e:
        line["e2e"] = run_e2e(args, wl, b, layers, workspace, stream, dev, px, torch, world, dist,
                              build_all, drain_merges, bwd_done)

    # ---- the oracle on this host's cores (rank 0, N = 1)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        secs, threads = oracle_sample(wl, b, args.cpu_tokens, args.mode)
        line["cpu_baseline"] = {
            "value": args.cpu_tokens / secs, "unit": "tokens/s", "cores": threads,
            "kind": "oracle",
            "sample": (f"{len(wl.linears)} linears x {args.cpu_tokens} tokens (of {T}), fwd+bwd "
                       f"with block build, fp64 numpy, {secs:.1f} s; merge not timed")}
    # ---- the other workloads, each in a child process (rank 0, N = 1)
    if rank == 0 and world == 1 and not args.no_extra:
        line["workloads"] = run_extra_workloads(args)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# The benchmark's other configurations, measured after the main line: the
# single fp32 linear, the LLaMA-60M and d = 1024 blocks, the d = 2048 block
# with 256-wide blocks, and the d = 4096 FFN pair at b = 128 and b = 512.
EXTRA_WORKLOADS = [("fp32_256", 32), ("llama60m_block", 32), ("d1024_block", 64),
                   ("d2048_block", 256), ("d4096_ffn", 128), ("d4096_ffn", 512)]


def summarise_extra(d: dict) -> dict:
    """The fields of a child benchmark line that the main line reports."""
    roof = d.get("roofline") or {}
    clk = d.get("clocks") or {}
    return {
        "workload": d["config"]["workload"], "b": d["config"]["b"], "dtype": d["dtype"],
        "tokens_per_s": d["value"], "ms_per_step": d["ms_per_step"], "steps": d["steps"],
        "step_tflop": d.get("step_tflop"), "tflops": d.get("tflops"),
        "frac_of_bf16_burst": d.get("tflops_frac_of_bf16_burst"),
        "frac_of_bf16_sustained": d.get("tflops_frac_of_bf16_sustained"),
        "cuda_graph": d["config"].get("cuda_graph"), "recompute": d["config"].get("recompute"),
        "merge_each_step": d["config"].get("merge_each_step"),
        "roofline": {k: roof.get(k) for k in ("kernel", "bound", "achieved", "peak", "unit", "frac")}
        if roof else None,
        "gpu_launches": d.get("gpu_launches"),
        "clocks": {k: clk.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons")} if clk else None,
        "device_status": d.get("device_status"),
    }


def run_extra_workloads(args):
    out = []
    for key, b in EXTRA_WORKLOADS:
        cmd = [sys.executable, os.path.abspath(__file__), "--workload", key, "--b", str(b),
               "--steps", str(args.extra_steps), "--warmup", "3", "--mode", args.mode,
               "--no-e2e", "--no-cpu-baseline", "--no-overhead", "--no-extra"]
        t0 = time.time()
        try:
            res = subprocess.run(cmd, capture_output=True, text=True, timeout=900)
            lines = [l for l in res.stdout.strip().splitlines() if l.startswith("{")]
            if res.returncode != 0 or not lines:
                out.append({"workload": key, "b": b, "error": (res.stderr or res.stdout)[-400:]})
                continue
            rec = summarise_extra(json.loads(lines[-1]))
            rec["wall_s"] = round(time.time() - t0, 1)
            out.append(rec)
        except Exception as exc:  # a failed child is reported, not fatal to the main line
            out.append({"workload": key, "b": b, "error": repr(exc)[-400:]})
    return out


def flush_l2(torch, buf):
    buf.add_(1)  # a write pass over a buffer larger than L2


def overhead_and_breakdown(args, wl, b, layers, workspace, stream, dev, px, torch, ms_per_step):
    """Per-linear POET-X fwd+bwd times, and the same layers as plain bf16
    linears (cuBLAS through torch.matmul: forward Y = X W^T, dgrad dX = dY W,
    wgrad dW = dY^T X) and as only the GEMMs POET-X itself runs (forward and
    dgrad, plus the recomputed forward in recompute mode).  Each repetition is
    timed alone with CUDA events after an L2 flush."""
    T = wl.tokens
    reps = 5
    flush = torch.empty(64 << 20, dtype=torch.float32, device=dev)  # 256 MB > L2
    # the plain linear keeps a dense weight of the layer dtype (an int8 layer's
    # weight buffer holds codes and scales)
    Ws = {id(st): (st["W0p"] if st["W0p"].dtype != torch.uint8 else
                   torch.zeros(st["lin"].m, st["lin"].n, dtype=st["X"].dtype, device=dev))
          for st in layers}
    dWs = {id(st): torch.empty_like(st["W0p"]) for st in layers}

    def timed(fn):
        tot = 0.0
        with torch.cuda.stream(stream):
            fn()   # warm-up
            for _ in range(reps):
                flush_l2(torch, flush)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                e1.synchronize()
                tot += e0.elapsed_time(e1)
        return tot / reps

    per = []
    plain_total = gemm_total = 0.0
    for st in layers:
        lin = st["lin"]

        def poetx_fb(st=st):
            px.poetx_linear_fwd(st["desc"], st["params"], st["W0p"], st["X"], T, st["Y"], st["h"],
                                st["u"], workspace, stream)
            px.poetx_linear_bwd(st["desc"], st["params"], st["W0p"], st["X"], st["dY"], st["h"],
                                st["u"], T, st["dX"], st["dgR"], st["dgP"], 0, workspace, stream)

        def plain(st=st):
            W = Ws[id(st)]
            torch.matmul(st["X"], W.t(), out=st["Y"])
            torch.matmul(st["dY"], W, out=st["dX"])
            torch.matmul(st["dY"].t(), st["X"], out=dWs[id(st)])

        def same_gemms(st=st):
            W = Ws[id(st)]
            torch.matmul(st["X"], W.t(), out=st["Y"])
            if wl.recompute:
                torch.matmul(st["X"], W.t(), out=st["Y"])
            torch.matmul(st["dY"], W, out=st["dX"])

        t_p = timed(poetx_fb)
        t_l = timed(plain)
        t_g = timed(same_gemms)
        sR, sP = block_square_sum(lin.m, b), block_square_sum(lin.n, b)
        fl = 4.0 * T * lin.m * lin.n + 6.0 * T * (sR + sP)
        if wl.recompute:
            fl += 2.0 * T * lin.m * lin.n + 2.0 * T * sP
        per.append({"linear": f"{lin.name}:{lin.n}->{lin.m}", "ms": t_p,
                    "tflops": fl / (t_p / 1e3) / 1e12, "plain_linear_ms": t_l,
                    "same_gemms_ms": t_g})
        plain_total += t_l
        gemm_total += t_g
    torch.cuda.synchronize(dev)
    sum_linears = sum(p["ms"] for p in per)
    return per, {
        "reading": ("primary: POET-X fwd+bwd vs a plain bf16 linear layer of the same shapes "
                    "(forward, dgrad and wgrad GEMMs via cuBLAS); secondary: vs only the GEMMs "
                    "POET-X runs (forward, dgrad, recomputed forward)"),
        "poetx_linears_ms": sum_linears, "poetx_step_ms": ms_per_step,
        "plain_linear_ms": plain_total, "same_gemms_ms": gemm_total,
        "vs_plain_linear": sum_linears / plain_total - 1.0,
        "vs_same_gemms": sum_linears / gemm_total - 1.0,
        "note": ("per-linear sums exclude the block builds and merges, which the step also runs; "
                 "each linear timed alone after an L2 flush"),
    }


def run_e2e(args, wl, b, layers, workspace, stream, dev, px, torch, world, dist, build_all,
            drain_merges, bwd_done):
    T = wl.tokens
    maxn = max(l.n for l in wl.linears)
    maxm = max(l.m for l in wl.linears)
    # one pinned host buffer per operand, sized for the widest linear; each
    # linear copies its own T x n (T x m) prefix every step
    Xh = torch.empty(T * maxn, dtype=layers[0]["X"].dtype, pin_memory=True)
    dYh = torch.empty(T * maxm, dtype=layers[0]["X"].dtype, pin_memory=True)
    wide_n = max(layers, key=lambda s: s["lin"].n)
    wide_m = max(layers, key=lambda s: s["lin"].m)
    Xh[: T * wide_n["lin"].n].copy_(wide_n["X"].reshape(-1).cpu())
    dYh[: T * wide_m["lin"].m].copy_(wide_m["dY"].reshape(-1).cpu())
    ghR = {id(st): torch.empty(st["lr"], dtype=torch.float32, pin_memory=True) for st in layers}
    ghP = {id(st): torch.empty(st["lp"], dtype=torch.float32, pin_memory=True) for st in layers}
    h2d = sum(T * (st["lin"].n + st["lin"].m) * Xh.element_size() for st in layers)
    d2h = sum((st["lr"] + st["lp"]) * 4 for st in layers)
    cnt = [0]

    def step():
        s = cnt[0]
        ready = build_all(1000 + s)
        for evs in ready:
            for e in evs:
                stream.wait_event(e)
        # every linear has its own device buffers, so the asynchronous host
        # step may stream later linears' inputs while earlier ones compute;
        # the step ends with one synchronisation
        for st in layers:
            px.poetx_linear_step_host_async(st["desc"], st["params"], st["W0p"], Xh, dYh, T, st["X"],
                                            st["dY"], st["Y"], st["h"], st["u"], st["dX"], st["dgR"],
                                            st["dgP"], ghR[id(st)], ghP[id(st)], workspace, stream)
        if wl.merge_each_step:
            for li in range(len(layers)):
                e = torch.cuda.Event()
                e.record(stream)
                bwd_done[li] = e
            drain_merges(1000 + s)
        torch.cuda.synchronize(dev)
        cnt[0] += 1

    for _ in range(max(1, min(args.warmup, 2))):
        step()
    if dist is not None:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    if dist is not None:
        t = torch.tensor([el], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        el = float(t.item())
    return {"value": world * T * args.steps / el, "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": 1e3 * el / args.steps,
            "scope": ("per step and linear through poetx_linear_step_host_async: X and dY copied "
                      "host -> device from pinned buffers, forward and backward (with the step's "
                      "block builds and, where the workload merges, the merges), packed generator "
                      "gradients copied device -> host; Y and dX stay on the device"),
            "timing": "host wall clock around the steps, one device synchronisation per step"}


if __name__ == "__main__":
    main()
