"""Run by tests/test_gpu_schedules.py in a child process, so that the library's
schedule switches (read once per process from the environment) take effect:
a few ragged dense and routed-expert workloads through the C ABI against the
float64 oracle.  Exits non-zero on the first parity failure."""

import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import synth  # noqa: E402
from helpers import TOL, compare, run_gpu, to_dev, to_np  # noqa: E402
from oracle import moe as moe_oracle  # noqa: E402


def dense(T, d, F, n_mb, overwrite=False):
    inp = synth.make_inputs(tokens=T, d=d, ffn=F, dtype="bf16", seed=T + d + F, n_mb=n_mb, eps=1e-5)
    outs, grads, _ = run_gpu(inp, overwrite_first=overwrite)
    ref_outs, ref_grads = oracle.run_workload(inp)
    compare(outs, grads, ref_outs, ref_grads, TOL["bf16"])


def routed(T, d, F, E, k, overwrite=False):
    import torch
    import mlp_block_backprop_gb300 as mb
    inp = synth.make_moe_inputs(T, d, F, E, k, seed=T + d + F + E, eps=1e-5)
    bb = mb.MoeBuffers(T, d, F, E, k, eps=inp.eps)
    for name in ("gamma", "w1s", "w2s", "x", "dy"):
        getattr(bb, name).copy_(to_dev(getattr(inp, name), torch.bfloat16))
    bb.idx.copy_(torch.from_numpy(np.ascontiguousarray(inp.idx, dtype=np.int32)).to("cuda"))
    bb.p.copy_(torch.from_numpy(np.ascontiguousarray(inp.p, dtype=np.float32)).to("cuda"))
    if overwrite:
        for name in ("dgamma", "dw1s", "dw2s"):
            getattr(bb, name).fill_(float("nan"))
    else:
        bb.zero_grads()
    bb.forward()
    bb.backward(overwrite=overwrite)
    torch.cuda.synchronize()
    p = inp.p.astype(np.float64)
    y, h, o, r = moe_oracle.forward(inp.x, inp.gamma, inp.w1s, inp.w2s, inp.idx, p, inp.eps)
    g = moe_oracle.new_grads(E, d, F)
    dx, dp = moe_oracle.backward(inp.dy, inp.x, inp.gamma, inp.w1s, inp.w2s, inp.idx, p, h, o, r, g)
    ref = {"y": y, "dx": dx, "dp": dp, "dgamma": g["dgamma"], "dw1s": g["dw1"], "dw2s": g["dw2"]}
    for key, val in ref.items():
        err = oracle.scaled_error(to_np(getattr(bb, key)), val)
        assert err <= TOL["bf16"], f"routed {key}: scaled error {err}"


if __name__ == "__main__":
    import mlp_block_backprop_gb300 as mb
    dense(520, 520, 520, 2)
    dense(1024, 512, 2048, 2)
    dense(2048, 256, 2560, 1)   # a 256 x 256 dgrad-h tile for every CTA pair
    dense(1024, 512, 2048, 2, overwrite=True)   # first microbatch writes the gradients
    dense(600, 1024, 1536, 1, overwrite=True)   # (row-kernel RMSNorm backward)
    dense(131, 2048, 512, 1)    # RMSNorm backward rows that take a whole CTA (odd row count)
    dense(67, 4096, 256, 2)
    routed(600, 512, 512, 4, 2)
    routed(300, 256, 256, 4, 3)
    routed(600, 512, 512, 4, 2, overwrite=True)
    rc = mb.mlpblk_last_error()
    assert rc == mb.MLPBLK_OK, f"device error {rc}"
    print("schedule case ok")
