"""mlpblk_backward_overwrite / mlpblk_moe_backward_overwrite: the first microbatch
of an accumulation window sets the weight gradients instead of adding into them
(zero_grads then += is the same as = for it).  The gradient buffers start as NaN,
so any element the overwrite misses, or any read of the old contents, shows up
(GB300 only).
"""

import numpy as np
import pytest

import oracle
import synth
from helpers import GRAD_KEYS, OUT_KEYS, TOL, compare, run_gpu, to_dev, to_np
from oracle import moe as moe_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mlp_block_backprop_gb300 as mb  # noqa: F401  (fails loudly if unbuilt)
    yield
    assert mb.mlpblk_last_error() == mb.MLPBLK_OK


CASES = [
    dict(tokens=520, d=520, ffn=520, dtype="bf16", n_mb=2),
    dict(tokens=1024, d=512, ffn=2048, dtype="bf16", n_mb=3, grad_scale=1.0 / 3.0),
    dict(tokens=1000, d=768, ffn=3072, dtype="bf16", n_mb=1),   # side-warp RMSNorm backward
    dict(tokens=300, d=1024, ffn=1536, dtype="bf16", n_mb=2),   # row-kernel RMSNorm backward
    dict(tokens=2048, d=256, ffn=2560, dtype="bf16", n_mb=1),
    dict(tokens=64, d=128, ffn=512, dtype="f32", n_mb=2),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"T{c['tokens']}_d{c['d']}_F{c['ffn']}_{c['dtype']}_mb{c['n_mb']}")
def test_overwrite_first_microbatch_matches_oracle(case):
    c = dict(case)
    inp = synth.make_inputs(tokens=c.pop("tokens"), d=c.pop("d"), ffn=c.pop("ffn"), seed=23, eps=1e-5, **c)
    outs, grads, _ = run_gpu(inp, overwrite_first=True)
    for k, v in grads.items():
        assert np.isfinite(v).all(), f"{k}: an element was not written"
    ref_outs, ref_grads = oracle.run_workload(inp)
    compare(outs, grads, ref_outs, ref_grads, TOL[inp.dtype])


@pytest.mark.parametrize("shape", [(2304, 768, 3072), (8192, 1024, 4096)], ids=["d768", "d1024_operands_beyond_l2"])
def test_overwrite_is_zero_then_add(shape):
    """The dense block clears the gradients in the backward's first launch and
    adds as before: the outputs bit for bit, the gradients up to the order in
    which split tiles' parts reach them (fp32 adds of three or more parts)."""
    T, d, F = shape
    inp = synth.make_inputs(tokens=T, d=d, ffn=F, dtype="bf16", seed=5, eps=1e-5)
    outs_a, grads_a, _ = run_gpu(inp)
    outs_b, grads_b, _ = run_gpu(inp, overwrite_first=True)
    for k in OUT_KEYS:
        assert np.array_equal(outs_a[0][k], outs_b[0][k]), k
    for k in GRAD_KEYS:
        assert np.isfinite(grads_b[k]).all(), k
        err = oracle.scaled_error(grads_b[k], grads_a[k])
        assert err <= 1e-6, f"{k}: {err}"


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_overwrite_with_no_tokens_leaves_zero_gradients(dtype):
    import torch
    import mlp_block_backprop_gb300 as mb
    bb = mb.BlockBuffers(0, 256, 512, dtype=dtype)
    for k in GRAD_KEYS:
        getattr(bb, k).fill_(float("nan"))
    bb.backward(overwrite=True)
    torch.cuda.synchronize()
    for k in GRAD_KEYS:
        assert torch.count_nonzero(getattr(bb, k)).item() == 0, k


def _routed(inp, overwrite):
    import torch
    import mlp_block_backprop_gb300 as mb
    T, d, F, E, k = inp.tokens, inp.d, inp.ffn, inp.experts, inp.top_k
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
    return bb


def test_routed_overwrite_with_an_unchosen_expert():
    """Expert E-1 is chosen by no token: its gradient blocks must come out zero
    (the K-grouped GEMMs have no tile for it); the rest against the oracle."""
    inp = synth.make_moe_inputs(600, 512, 512, 4, 2, seed=31, eps=1e-5)
    idx = inp.idx.copy()
    E = inp.experts
    for t in range(idx.shape[0]):
        for j in range(idx.shape[1]):
            if idx[t, j] == E - 1:
                idx[t, j] = next(e for e in range(E - 1) if e not in idx[t])
    inp.idx = idx
    bb = _routed(inp, overwrite=True)
    p = inp.p.astype(np.float64)
    y, h, o, r = moe_oracle.forward(inp.x, inp.gamma, inp.w1s, inp.w2s, idx, p, inp.eps)
    g = moe_oracle.new_grads(E, inp.d, inp.ffn)
    dx, dp = moe_oracle.backward(inp.dy, inp.x, inp.gamma, inp.w1s, inp.w2s, idx, p, h, o, r, g)
    got = {k: to_np(getattr(bb, k)) for k in ("y", "dx", "dp", "dgamma", "dw1s", "dw2s")}
    assert not got["dw1s"][E - 1].any() and not got["dw2s"][E - 1].any()
    ref = {"y": y, "dx": dx, "dp": dp, "dgamma": g["dgamma"], "dw1s": g["dw1"], "dw2s": g["dw2"]}
    for key, val in ref.items():
        assert np.isfinite(got[key]).all(), key
        err = oracle.scaled_error(got[key], val)
        assert err <= TOL["bf16"], f"{key}: scaled error {err}"


def test_routed_overwrite_agrees_with_zero_then_add():
    """Whole K-grouped tiles: the store and the add of the same tile give the
    same bits."""
    inp = synth.make_moe_inputs(1024, 512, 1024, 8, 2, seed=37, eps=1e-5)
    a = _routed(inp, overwrite=False)
    b = _routed(inp, overwrite=True)
    import torch
    for name in ("dx", "dp", "dgamma", "dw1s", "dw2s"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
