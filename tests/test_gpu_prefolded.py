"""W1 * gamma made once per weight update (mlpblk_fold_weights) and read by
every microbatch's forward (mlpblk_forward_prefolded), against the per-call
fold of mlpblk_forward and against the float64 oracle (GB300 only).

The contract: the same fold arithmetic either way, so y, h, a and rstd are the
per-call path's bit for bit, and so is everything the backward computes from
them; with gradient accumulation only the fp32 += weight gradients may differ,
in the order of their stream-K additions.
"""

import numpy as np
import pytest

import oracle
import synth
from helpers import GRAD_KEYS, OUT_KEYS, TOL, compare, to_dev, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mlp_block_backprop_gb300 as mb  # noqa: F401  (fails loudly if unbuilt)
    yield
    mb.mlpblk_set_rmsnorm_mode(mb.MLPBLK_RMSNORM_STATS_PASS)
    assert mb.mlpblk_last_error() == mb.MLPBLK_OK


def _run(inp, prefolded):
    import torch
    import mlp_block_backprop_gb300 as mb
    bb = mb.BlockBuffers(inp.tokens, inp.d, inp.ffn, dtype=inp.dtype, eps=inp.eps)
    bb.gamma.copy_(to_dev(inp.gamma, bb.dt))
    bb.w1.copy_(to_dev(inp.w1, bb.dt))
    bb.w2.copy_(to_dev(inp.w2, bb.dt))
    bb.zero_grads()
    if prefolded:
        bb.fold_weights()
    outs = []
    for x, dy in zip(inp.x, inp.dy):
        bb.x.copy_(to_dev(x, bb.dt))
        bb.dy.copy_(to_dev(dy, bb.dt))
        if prefolded:
            bb.forward_prefolded()
        else:
            bb.forward()
        bb.backward()
        outs.append({k: getattr(bb, k).clone() for k in OUT_KEYS})
    if inp.grad_scale is not None:
        bb.scale_grads(inp.grad_scale)
    torch.cuda.synchronize()
    grads = {k: getattr(bb, k).clone() for k in GRAD_KEYS}
    return outs, grads


CASES = [
    dict(tokens=520, d=520, ffn=520, dtype="bf16", n_mb=2),
    dict(tokens=1024, d=512, ffn=2048, dtype="bf16", n_mb=3, grad_scale=1.0 / 3.0),
    dict(tokens=300, d=1024, ffn=1536, dtype="bf16", n_mb=2),
    dict(tokens=64, d=128, ffn=512, dtype="f32", n_mb=2),
]


@pytest.mark.parametrize("mode", ["stats", "prologue"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"T{c['tokens']}_d{c['d']}_F{c['ffn']}_{c['dtype']}")
def test_prefolded_matches_per_call_fold_and_oracle(case, mode):
    import torch
    import mlp_block_backprop_gb300 as mb
    mb.mlpblk_set_rmsnorm_mode(mb.MLPBLK_RMSNORM_IN_W1_PROLOGUE if mode == "prologue"
                               else mb.MLPBLK_RMSNORM_STATS_PASS)
    c = dict(case)
    inp = synth.make_inputs(tokens=c.pop("tokens"), d=c.pop("d"), ffn=c.pop("ffn"), seed=17, **c)
    base_outs, base_grads = _run(inp, prefolded=False)
    outs, grads = _run(inp, prefolded=True)
    for i, (o, b) in enumerate(zip(outs, base_outs)):
        for k in OUT_KEYS:
            assert torch.equal(o[k], b[k]), f"{k}[{i}] differs from the per-call fold"
    if inp.n_mb == 1:
        for k in GRAD_KEYS:
            assert torch.equal(grads[k], base_grads[k]), k
    ref_outs, ref_grads = oracle.run_workload(inp)
    compare([{k: to_np(v) for k, v in o.items()} for o in outs], {k: to_np(v) for k, v in grads.items()},
            ref_outs, ref_grads, TOL[inp.dtype])


def test_fold_weights_is_the_columnwise_product():
    """w1g[f, k] = w1[f, k] * gamma[k], rounded once to the dtype."""
    import torch
    import mlp_block_backprop_gb300 as mb
    inp = synth.make_inputs(tokens=8, d=264, ffn=136, seed=5)
    w1 = to_dev(inp.w1, torch.bfloat16)
    g = to_dev(inp.gamma, torch.bfloat16)
    w1g = torch.empty_like(w1)
    mb.mlpblk_fold_weights(mb.make_desc(8, 264, 136), g, w1, w1g)
    torch.cuda.synchronize()
    want = torch.from_numpy((inp.w1.astype(np.float32) * inp.gamma.astype(np.float32)[None, :])).to(torch.bfloat16)
    assert torch.equal(w1g.cpu(), want)
