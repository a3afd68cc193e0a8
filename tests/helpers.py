"""Shared helpers of the GPU tests: move synthetic inputs to the device, run the
CUDA path through the C ABI, and run the float64 oracle on the same inputs."""

from __future__ import annotations

import numpy as np

import oracle

TOL = {"bf16": 2e-2, "f32": 1e-5}   # max scaled error per tensor
OUT_KEYS = ("y", "h", "a", "rstd", "dx")
GRAD_KEYS = ("dgamma", "dw1", "dw2")


def to_dev(arr, dtype):
    import torch
    return torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32)).to("cuda").to(dtype)


def to_np(t):
    return t.float().cpu().numpy().astype(np.float64)


def gpu_buffers(inp):
    import mlp_block_backprop_gb300 as mb
    bb = mb.BlockBuffers(inp.tokens, inp.d, inp.ffn, dtype=inp.dtype, eps=inp.eps)
    bb.gamma.copy_(to_dev(inp.gamma, bb.dt))
    bb.w1.copy_(to_dev(inp.w1, bb.dt))
    bb.w2.copy_(to_dev(inp.w2, bb.dt))
    return bb


def run_gpu(inp, keep_outputs=True, overwrite_first=False):
    """Forward + backward of every microbatch through the C ABI; grad_scale at the end.
    overwrite_first: no zero_grads; the gradient buffers start as NaN and the first
    microbatch's backward writes them (mlpblk_backward_overwrite)."""
    import torch
    bb = gpu_buffers(inp)
    if overwrite_first:
        for k in GRAD_KEYS:
            getattr(bb, k).fill_(float("nan"))
    else:
        bb.zero_grads()
    outs = []
    for i, (x, dy) in enumerate(zip(inp.x, inp.dy)):
        bb.x.copy_(to_dev(x, bb.dt))
        bb.dy.copy_(to_dev(dy, bb.dt))
        bb.forward()
        bb.backward(overwrite=overwrite_first and i == 0)
        if keep_outputs:
            outs.append({k: to_np(getattr(bb, k)) for k in OUT_KEYS})
    if inp.grad_scale is not None:
        bb.scale_grads(inp.grad_scale)
    torch.cuda.synchronize()
    grads = {k: to_np(getattr(bb, k)) for k in GRAD_KEYS}
    return outs, grads, bb


def compare(got_outs, got_grads, ref_outs, ref_grads, tol):
    """Scaled errors of every output and gradient; returns {name: error}."""
    errs = {}
    for i, (g, r) in enumerate(zip(got_outs, ref_outs)):
        for k in OUT_KEYS:
            rk = "r" if k == "rstd" else k
            errs[f"{k}[{i}]"] = oracle.scaled_error(g[k], r[rk])
    for k in GRAD_KEYS:
        errs[k] = oracle.scaled_error(got_grads[k], ref_grads[k])
    bad = {k: v for k, v in errs.items() if not (v <= tol)}
    assert not bad, f"scaled error above {tol}: {bad} (all: {errs})"
    return errs


def sampled_reference(inp, rows, units):
    """Oracle values of a sample of a large workload, each exact for its entry.

    rows : token indices; y, h, a, r and dx of a token depend on that token's row
           only, so the oracle runs on those rows alone.
    units: hidden units f; h[:, f] and a[:, f] depend on W1[f] only, so the oracle
           restricted to those units gives dW2[:, f] and dW1[f, :] exactly.
    Returns per-microbatch row outputs and the summed sampled gradient slices.
    """
    out_rows = []
    dw2_cols = np.zeros((inp.d, len(units)))
    dw1_rows = np.zeros((len(units), inp.d))
    for x, dy in zip(inp.x, inp.dy):
        xr, dyr = x[rows].astype(np.float64), dy[rows].astype(np.float64)
        y, h, a, r = oracle.forward(xr, inp.gamma, inp.w1, inp.w2, inp.eps)
        g = oracle.new_grads(inp.d, inp.ffn)
        dx = oracle.backward(dyr, xr, inp.gamma, inp.w1, inp.w2, h, r, g)
        out_rows.append({"y": y, "h": h, "a": a, "r": r, "dx": dx})
        w1s, w2s = inp.w1[units], inp.w2[:, units]
        _, hs, _, rs = oracle.forward(x, inp.gamma, w1s, w2s, inp.eps)
        gs = oracle.new_grads(inp.d, len(units))
        oracle.backward(dy, x, inp.gamma, w1s, w2s, hs, rs, gs)
        dw2_cols += gs["dw2"]
        dw1_rows += gs["dw1"]
    if inp.grad_scale is not None:
        dw2_cols *= inp.grad_scale
        dw1_rows *= inp.grad_scale
    return out_rows, dw2_cols, dw1_rows
