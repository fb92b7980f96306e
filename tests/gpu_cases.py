"""Shared helpers of the GPU parity tests: run one layer through the C ABI and
through the fp64 oracle on the same seeded inputs, and compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
import synth


def rel_fro(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))


def worst_row_rel(a, b) -> float:
    """Largest relative error of a single row, max_t ||a_t - b_t|| / ||b_t||:
    a wrong tile of tokens or a wrong short row cannot hide in the aggregate."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    if a.size == 0:
        return 0.0
    nb = np.linalg.norm(b, axis=1)
    return float((np.linalg.norm(a - b, axis=1) / np.where(nb > 0, nb, 1.0)).max())


def packed_block_slices(d: int, b: int):
    """Slices of the packed generator vector that belong to each block
    (blocks of b, then a ragged d mod b; 1 x 1 blocks have no entries)."""
    out, off = [], 0
    for s in O.block_sizes(d, b):
        n = s * (s - 1) // 2
        if n:
            out.append(slice(off, off + n))
        off += n
    return out


def worst_block_rel(a, b, d: int, bs: int) -> float:
    """Largest relative Frobenius error of one block's packed gradient."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return max((rel_fro(a[sl], b[sl]) for sl in packed_block_slices(d, bs)), default=0.0)


def parity_errors(g, o, m, n, bR, bP) -> dict:
    """Aggregate relative Frobenius errors of Y, dX, dgR, dgP, plus the worst
    row of Y and dX and the worst block of dgR and dgP."""
    errs = {k: rel_fro(g[k], o[k]) for k in ("Y", "dX", "dgR", "dgP")
            if g.get(k) is not None and o[k].size}
    if g.get("Y") is not None and o["Y"].size:
        errs["Y_worst_row"] = worst_row_rel(g["Y"], o["Y"])
    if g.get("dX") is not None and o["dX"].size:
        errs["dX_worst_row"] = worst_row_rel(g["dX"], o["dX"])
    if o["dgR"].size:
        errs["dgR_worst_block"] = worst_block_rel(g["dgR"], o["dgR"], m, bR)
    if o["dgP"].size:
        errs["dgP_worst_block"] = worst_block_rel(g["dgP"], o["dgP"], n, bP)
    return errs


def make_inputs(m, n, bR, bP, T, dtype, index=0, t0=0, t1=None, gstd=synth.STD_GEN):
    lin = synth.Linear("case", n, m)
    lr, lp = O.packed_length(m, bR), O.packed_length(n, bP)
    inp = synth.layer_inputs(lin, index, T, dtype, lr, lp, t0=t0, t1=t1)
    if gstd != synth.STD_GEN:
        inp.genR = inp.genR * (gstd / synth.STD_GEN)
        inp.genP = inp.genP * (gstd / synth.STD_GEN)
    return inp


def run_gpu(px, desc, inp, recompute: bool, want_dX=True, dev="cuda", save_u=False):
    """Forward + backward through the C ABI; returns CPU float64 numpy arrays.

    recompute: h is not saved by the forward.  save_u: the forward saves the
    permuted input u and the backward gets it instead of X (X is passed as
    NULL there, so the backward cannot read it)."""
    T = inp.X.shape[0]
    layer = px.Layer(desc, max(T, 1), device=dev)
    layer.build(inp.genR.to(dev), inp.genP.to(dev))
    W0 = inp.W0.to(dev)
    layer.premerge(W0)
    X = inp.X.to(dev)
    dY = inp.dY.to(dev)
    Y = torch.empty(T, desc.m, dtype=layer.dtype, device=dev)
    h = None if recompute else torch.empty(T, desc.m, dtype=layer.dtype, device=dev)
    u = torch.empty(T, desc.n, dtype=layer.dtype, device=dev) if save_u else None
    layer.forward(X, Y, saved_h=h, saved_u=u)
    dX = torch.empty(T, desc.n, dtype=layer.dtype, device=dev) if want_dX else None
    dgR = torch.empty(layer.len_R, dtype=torch.float32, device=dev)
    dgP = torch.empty(layer.len_P, dtype=torch.float32, device=dev)
    layer.backward(None if save_u else X, dY, dX, dgR, dgP, saved_h=h, saved_u=u)
    torch.cuda.synchronize()
    st = px.poetx_device_status(reset=True)
    assert st == px.POETX_OK, px.poetx_status_string(st)
    f = lambda t: None if t is None else t.double().cpu().numpy()
    return dict(Y=f(Y), dX=f(dX), dgR=f(dgR), dgP=f(dgP), W0p=f(layer.W0p), u=f(u), layer=layer)


def run_oracle(spec: O.LayerSpec, inp):
    W0 = inp.W0.double().numpy()
    X = inp.X.double().numpy()
    dY = inp.dY.double().numpy()
    gR = inp.genR.double().numpy()
    gP = inp.genP.double().numpy()
    dX, dgR, dgP, ex = O.backward(spec, W0, X, dY, gR, gP)
    return dict(Y=ex["Y"], dX=dX, dgR=dgR, dgP=dgP, W0p=ex["W0p"], h=ex["h"])
