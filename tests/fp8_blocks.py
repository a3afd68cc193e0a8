"""The float64 FP8 oracle (oracle.fp8) of a one-microbatch synth workload,
evaluated in row blocks on a pool of spawned processes: first every block's
max |a| and max |dh| (oracle.fp8.block_amaxes), then every block's forward and
backward with the whole tensors' scales.  Elementwise, the oracle is row-wise,
so each output row is the one the whole-tensor evaluation gives; the weight
gradients are the blocks' float64 partial sums added in block order.  Used by
the FP8 parity test at the wide workload's full size, where one process would
take minutes of single-threaded numpy."""

from __future__ import annotations

import multiprocessing
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

_inputs = {}


def _inp(name):
    import synth
    if name not in _inputs:
        _inputs.clear()
        _inputs[name] = synth.config_inputs(name)
    return _inputs[name]


def _block(job):
    import oracle
    from oracle import fp8
    name, i0, i1, amaxes = job
    inp = _inp(name)
    x, dy = inp.x[0][i0:i1], inp.dy[0][i0:i1]
    dy_amax = np.float32(np.max(np.abs(inp.dy[0].astype(np.float32))))
    if amaxes is None:
        return fp8.block_amaxes(x, dy, inp.gamma, inp.w1, inp.w2, inp.eps, dy_amax)
    a_amax, dh_amax = amaxes
    y, h, a_q, n_q, r = fp8.forward(x, inp.gamma, inp.w1, inp.w2, inp.eps, a_amax)
    g = oracle.new_grads(inp.d, inp.ffn)
    dx = fp8.backward(dy, x, inp.gamma, inp.w1, inp.w2, h, a_q, n_q, r, g, dy_amax, dh_amax)
    return {"y": y, "h": h, "r": r, "dx": dx}, g


def run_blocks(name, rows=2048, procs=None):
    """({"y", "h", "r", "dx"}, grads) of the workload's first microbatch."""
    import synth
    tokens = synth.CONFIGS[name]["tokens"]
    spans = [(i, min(tokens, i + rows)) for i in range(0, tokens, rows)]
    if procs is None:
        # each process holds the inputs and one block's float64 temporaries (~3 GB)
        try:
            free_gb = os.sysconf("SC_AVPHYS_PAGES") * os.sysconf("SC_PAGE_SIZE") / 2**30
        except (ValueError, OSError):
            free_gb = 24.0
        procs = max(1, min(len(spans), 8, os.cpu_count() or 1, int(free_gb // 3)))
    ctx = multiprocessing.get_context("spawn")
    with ctx.Pool(procs) as pool:
        am = pool.map(_block, [(name, i0, i1, None) for i0, i1 in spans])
        amaxes = (max(a for a, _ in am), max(h for _, h in am))
        parts = pool.map(_block, [(name, i0, i1, amaxes) for i0, i1 in spans])
    outs = {k: np.concatenate([p[0][k] for p in parts]) for k in ("y", "h", "r", "dx")}
    grads = {k: np.zeros_like(parts[0][1][k]) for k in parts[0][1]}
    for _, g in parts:
        for k in grads:
            grads[k] += g[k]
    return outs, grads
