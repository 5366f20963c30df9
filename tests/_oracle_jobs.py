"""Oracle sub-problems for the full-size parity tests, run in worker
processes.  The pool is started with the ``spawn`` method, so workers never
inherit the parent's CUDA context; this module imports no GPU code.

One job is one expert e and a list of its assignments in ascending order.
Every MXFP8 operand of the rows' forward, of D and of dX is blocked along a
row (or is a weight), so each row's Y / dX / d(gate) contribution is the same
in a sub-batch as in the full layer.  Only the weight gradients need the
expert's whole ascending row list (their token-axis blocks of 32 rows), which
the jobs that check them carry.
"""
from __future__ import annotations

import os

import numpy as np

from oracle import moe_oracle as O
from workloads import bf16_bits_to_f32


def _f32(a):
    return bf16_bits_to_f32(a) if a.dtype == np.uint16 else np.asarray(a, np.float32)


def expert_subbatch(job):
    """job: dict(e, t, j (the assignments' tokens and slots), X, dY (their
    rows), W13, W2 (expert e's weights), gate (per assignment), mode, dw).
    Returns (e, t, j, gate * z rows, dX rows, d(gate) per row, dW13 and dW2
    of the sub-batch or None)."""
    n = len(job["t"])
    one = np.zeros((n, 1), np.int32)
    g = np.asarray(job["gate"], np.float64)[:, None]
    args = (_f32(job["X"]), _f32(job["W13"])[None], _f32(job["W2"])[None], one, g)
    y = O.forward(*args, mode=job["mode"])
    b = O.backward(*args, _f32(job["dY"]), mode=job["mode"])
    dw = (b["dW13"][0], b["dW2"][0]) if job["dw"] else None
    return job["e"], job["t"], job["j"], y, b["dX"], b["dgate"][:, 0], dw


def run_sampled(inp, idx, gate, tokens, dw_experts, mode, workers=None):
    """Y, dX and d(gate) of ``tokens`` and dW13 / dW2 of ``dw_experts`` from
    per-expert sub-batches, computed in a spawned process pool.  Returns
    (Y, dX, dgate, {e: (dW13_e, dW2_e)}) with rows following ``tokens``."""
    import multiprocessing as mp
    k = idx.shape[1]
    pos = {int(t): i for i, t in enumerate(tokens)}
    tokset = set(pos)
    jobs = []
    for e in range(int(idx.max()) + 1):
        t_all, j_all = np.nonzero(idx == e)          # ascending assignment order
        if e in dw_experts:
            t, j = t_all, j_all
        else:
            keep = np.isin(t_all, tokens)
            t, j = t_all[keep], j_all[keep]
        if t.size == 0:
            continue
        jobs.append(dict(e=e, t=t, j=j, X=inp["X"][t], dY=inp["dY"][t], W13=inp["W13"][e],
                         W2=inp["W2"][e], gate=gate[t, j], mode=mode, dw=e in dw_experts))
    H = inp["X"].shape[1]
    Y = np.zeros((len(tokens), H))
    dX = np.zeros((len(tokens), H))
    dg = np.zeros((len(tokens), k))
    dws = {}
    n = workers or min(16, os.cpu_count() or 1)
    with mp.get_context("spawn").Pool(n) as pool:
        for e, t, j, y, dx, dgr, dw in pool.imap_unordered(expert_subbatch, jobs):
            for r, (tt, jj) in enumerate(zip(t, j)):
                if int(tt) in tokset:
                    Y[pos[int(tt)]] += y[r]
                    dX[pos[int(tt)]] += dx[r]
                    dg[pos[int(tt)], jj] = dgr[r]
            if dw is not None:
                dws[e] = dw
    return Y, dX, dg, dws
