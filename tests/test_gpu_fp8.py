"""The FP8 (E4M3) operand variant against its float64 oracle (oracle.fp8), which
quantises the same tensors with the same per-tensor scales (GB300 only).

Tolerance: scaled error 2e-2, as for the bf16 block.  The quantisation decisions
are taken on float32 values on both sides (the same codes wherever the inputs to
a quantisation agree: W1*gamma, W2, W1 and dy exactly; n', a and dh up to the
last bits of their float32 sums, which moves a few codes by one step); what
remains is float32 accumulation and the bf16 roundings of the bf16 block.
"""

import numpy as np
import pytest

import oracle
import synth
from oracle import fp8 as fp8_oracle
from helpers import to_dev, to_np

pytestmark = pytest.mark.gpu
TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mlp_block_backprop_gb300 as mb  # noqa: F401
    yield
    assert mb.mlpblk_last_error() == mb.MLPBLK_OK


def _run_fp8(inp):
    import torch
    import mlp_block_backprop_gb300 as mb
    bb = mb.BlockBuffers(inp.tokens, inp.d, inp.ffn, dtype="bf16", eps=inp.eps, fp8=True)
    bb.gamma.copy_(to_dev(inp.gamma, bb.dt))
    bb.w1.copy_(to_dev(inp.w1, bb.dt))
    bb.w2.copy_(to_dev(inp.w2, bb.dt))
    bb.zero_grads()
    outs = []
    for x, dy in zip(inp.x, inp.dy):
        bb.x.copy_(to_dev(x, bb.dt))
        bb.dy.copy_(to_dev(dy, bb.dt))
        bb.forward()
        bb.backward()
        outs.append({k: to_np(getattr(bb, k)) for k in ("y", "h", "rstd", "dx")})
    if inp.grad_scale is not None:
        bb.scale_grads(inp.grad_scale)
    torch.cuda.synchronize()
    grads = {k: to_np(getattr(bb, k)) for k in ("dgamma", "dw1", "dw2")}
    return outs, grads, bb


def _check(inp):
    outs, grads, _ = _run_fp8(inp)
    ref_outs, ref_grads = fp8_oracle.run_workload(inp)
    errs = {}
    for i, (g, r) in enumerate(zip(outs, ref_outs)):
        for k, rk in (("y", "y"), ("h", "h"), ("rstd", "r"), ("dx", "dx")):
            errs[f"{k}[{i}]"] = oracle.scaled_error(g[k], r[rk])
    for k in ("dgamma", "dw1", "dw2"):
        errs[k] = oracle.scaled_error(grads[k], ref_grads[k])
    bad = {k: v for k, v in errs.items() if not (v <= TOL)}
    assert not bad, f"scaled error above {TOL}: {bad} (all: {errs})"
    return errs


def test_fp8_small_bf16_accum4_config():
    _check(synth.config_inputs("small_bf16_accum4"))


@pytest.mark.parametrize("shape", [
    (333, 208, 336),    # ragged tokens; several tiles in every GEMM
    (1, 256, 512),      # one token
    (77, 144, 1040),    # ffn spans five 256-wide tiles with a tail
    (520, 528, 528),
])
def test_fp8_ragged(shape):
    T, d, F = shape
    _check(synth.make_inputs(tokens=T, d=d, ffn=F, dtype="bf16", seed=T + d + F, n_mb=2, eps=1e-5))


@pytest.mark.slow
def test_fp8_wide_workload_full_size():
    """The wide workload (16384 tokens, d 2048, ffn 8192: K up to 16384 in
    128-value E4M3 stages, stream-K splits and reduce-add epilogues at a benched
    size), every element of every output against the float64 FP8 oracle, which
    runs in row blocks with the whole tensors' scales (tests/fp8_blocks.py)."""
    import fp8_blocks
    inp = synth.config_inputs("wide")
    outs, grads, _ = _run_fp8(inp)
    ref, ref_grads = fp8_blocks.run_blocks("wide")
    errs = {k: oracle.scaled_error(outs[0][k], ref["r" if k == "rstd" else k]) for k in ("y", "h", "rstd", "dx")}
    errs.update({k: oracle.scaled_error(grads[k], ref_grads[k]) for k in ("dgamma", "dw1", "dw2")})
    bad = {k: v for k, v in errs.items() if not (v <= TOL)}
    assert not bad, f"scaled error above {TOL}: {bad} (all: {errs})"


def test_fp8_saved_codes_and_scale():
    """The saved a codes are E4M3 bytes whose largest magnitude is 448 (the amax
    element), and a's scale record is {amax, 448/amax, amax/448, 0}."""
    import torch
    inp = synth.make_inputs(tokens=256, d=128, ffn=512, dtype="bf16", seed=3, n_mb=1, eps=1e-6)
    _, _, bb = _run_fp8(inp)
    a8 = bb.a8.view(torch.float8_e4m3fn).float()
    assert float(a8.abs().max()) == 448.0
    assert float(a8.min()) >= 0.0           # a = relu(h)^2 >= 0
    sc = bb.scales.cpu().numpy()
    assert sc[1] == np.float32(448.0) / np.float32(sc[0])
    assert sc[2] == np.float32(sc[0]) / np.float32(448.0)
    n8 = bb.n8.view(torch.float8_e4m3fn).float().cpu().numpy()
    x = inp.x[0].astype(np.float32)
    r = fp8_oracle.rstd32(inp.x[0], inp.eps)
    ref = fp8_oracle.e4m3((x * r[:, None]).astype(np.float32))
    # the codes of n' = x * rstd: equal, except where the two float32 rstd values
    # (different summation orders) put x * rstd on either side of a rounding
    # boundary, and there one step apart
    diff = n8 != ref
    assert diff.mean() <= 1e-3
    step = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref[diff]), 2.0 ** -6))) - 3)
    assert np.all(np.abs(n8[diff] - ref[diff]) <= step * (1 + 1e-6))


def test_fp8_matches_the_bf16_block_within_fp8_error():
    inp = synth.make_inputs(tokens=384, d=256, ffn=768, dtype="bf16", seed=21, n_mb=1, eps=1e-6)
    outs, grads, _ = _run_fp8(inp)
    ref_outs, ref_grads = oracle.run_workload(inp)
    assert oracle.scaled_error(outs[0]["y"] - inp.x[0], ref_outs[0]["y"] - inp.x[0]) < 0.15
    for k in ("dw1", "dw2"):
        assert oracle.scaled_error(grads[k], ref_grads[k]) < 0.15


@pytest.mark.parametrize("shape", [(300, 128, 512), (1024, 512, 2048)])
def test_fp8_prequantised_weights_give_the_same_bits(shape):
    """Weights quantised once (mlpblk_fp8_quantize_weights) and used by every
    microbatch give bitwise the outputs and dgamma of the calls that quantise them
    each time; dW1 and dW2 agree up to the order of the fp32 reduce-adds of a
    weight-gradient tile split between workers (the one unordered sum)."""
    import torch
    import mlp_block_backprop_gb300 as mb
    T, d, F = shape
    inp = synth.make_inputs(tokens=T, d=d, ffn=F, dtype="bf16", seed=T + F, n_mb=3, eps=1e-6)
    outs, grads, bb = _run_fp8(inp)
    bb.zero_grads()
    mb.mlpblk_fp8_quantize_weights(bb.desc, bb.gamma, bb.w1, bb.w2, bb.wq, bb.ws)
    outs2 = []
    for x, dy in zip(inp.x, inp.dy):
        bb.x.copy_(to_dev(x, bb.dt))
        bb.dy.copy_(to_dev(dy, bb.dt))
        mb.mlpblk_forward_fp8_prequant(bb.desc, bb.x, bb.wq, bb.y, bb.h, bb.a8, bb.n8, bb.rstd, bb.scales, bb.ws)
        mb.mlpblk_backward_fp8_prequant(bb.desc, bb.dy, bb.x, bb.gamma, bb.wq, bb.h, bb.a8, bb.n8, bb.rstd,
                                        bb.scales, bb.dx, bb.dgamma, bb.dw1, bb.dw2, bb.ws)
        outs2.append({k: to_np(getattr(bb, k)) for k in ("y", "h", "rstd", "dx")})
    torch.cuda.synchronize()
    for a, b in zip(outs, outs2):
        for k in a:
            np.testing.assert_array_equal(a[k], b[k], err_msg=k)
    np.testing.assert_array_equal(grads["dgamma"], to_np(bb.dgamma), err_msg="dgamma")
    for k in ("dw1", "dw2"):
        got = to_np(getattr(bb, k))
        np.testing.assert_allclose(got, grads[k], rtol=1e-5, atol=1e-6 * float(np.max(np.abs(grads[k]))),
                                   err_msg=k)


def test_fp8_interleaved_writers_and_readers_in_a_graph():
    """Stream kernels writing x and dy right before the calls and reading the
    outputs right after, three microbatches captured as one CUDA graph, match the
    FP8 oracle's accumulation (the backward's GEMM pairs overlap at their launch
    boundary)."""
    import torch
    import mlp_block_backprop_gb300 as mb
    inp = synth.make_inputs(tokens=640, d=256, ffn=1040, seed=31, n_mb=3)
    bb = mb.BlockBuffers(inp.tokens, inp.d, inp.ffn, dtype="bf16", eps=inp.eps, fp8=True)
    bb.gamma.copy_(to_dev(inp.gamma, bb.dt))
    bb.w1.copy_(to_dev(inp.w1, bb.dt))
    bb.w2.copy_(to_dev(inp.w2, bb.dt))
    xs = [to_dev(x, bb.dt) for x in inp.x]
    dys = [to_dev(g, bb.dt) for g in inp.dy]
    keys = ("y", "h", "rstd", "dx")
    keep = {k: [torch.empty_like(getattr(bb, k)) for _ in inp.x] for k in keys}

    def steps():
        bb.zero_grads()
        for i in range(len(xs)):
            bb.x.copy_(xs[i])
            bb.forward()
            for k in ("y", "h", "rstd"):
                keep[k][i].copy_(getattr(bb, k))
            bb.dy.copy_(dys[i])
            bb.backward()
            keep["dx"][i].copy_(bb.dx)

    steps()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        steps()
    for k in keys:
        for t in keep[k]:
            t.fill_(5.0)
    g.replay()
    torch.cuda.synchronize()
    ref_outs, ref_grads = fp8_oracle.run_workload(inp)
    errs = {}
    for i, r in enumerate(ref_outs):
        for k, rk in (("y", "y"), ("h", "h"), ("rstd", "r"), ("dx", "dx")):
            errs[f"{k}[{i}]"] = oracle.scaled_error(to_np(keep[k][i]), r[rk])
    for k in ("dgamma", "dw1", "dw2"):
        errs[k] = oracle.scaled_error(to_np(getattr(bb, k)), ref_grads[k])
    bad = {k: v for k, v in errs.items() if not (v <= TOL)}
    assert not bad, f"scaled error above {TOL}: {bad} (all: {errs})"


@pytest.mark.parametrize("shape", [(2304, 768, 3072), (8192, 1024, 4096)], ids=["d768", "d1024_operands_beyond_l2"])
@pytest.mark.parametrize("prequant", [False, True], ids=["quantise_each_call", "prequantised"])
def test_fp8_overwrite_is_zero_then_add(shape, prequant):
    """mlpblk_backward_fp8_overwrite / _prequant_overwrite on the first of two
    microbatches: the gradient buffers start as NaN and come out as zero_grads
    followed by adding backwards would leave them, the outputs bit for bit and
    dW1, dW2, dgamma up to the order in which a split tile's parts reach it."""
    import torch
    import mlp_block_backprop_gb300 as mb
    T, d, F = shape
    inp = synth.make_inputs(tokens=T, d=d, ffn=F, dtype="bf16", seed=T + 7, n_mb=2, eps=1e-5)
    bb = mb.BlockBuffers(inp.tokens, inp.d, inp.ffn, dtype="bf16", eps=inp.eps, fp8=True)
    bb.gamma.copy_(to_dev(inp.gamma, bb.dt))
    bb.w1.copy_(to_dev(inp.w1, bb.dt))
    bb.w2.copy_(to_dev(inp.w2, bb.dt))
    if prequant:
        mb.mlpblk_fp8_quantize_weights(bb.desc, bb.gamma, bb.w1, bb.w2, bb.wq, bb.ws)
    runs = []
    for overwrite in (False, True):
        if overwrite:
            for k in ("dgamma", "dw1", "dw2"):
                getattr(bb, k).fill_(float("nan"))
        else:
            bb.zero_grads()
        outs = []
        for i, (x, dy) in enumerate(zip(inp.x, inp.dy)):
            bb.x.copy_(to_dev(x, bb.dt))
            bb.dy.copy_(to_dev(dy, bb.dt))
            first = overwrite and i == 0
            if prequant:
                mb.mlpblk_forward_fp8_prequant(bb.desc, bb.x, bb.wq, bb.y, bb.h, bb.a8, bb.n8, bb.rstd, bb.scales,
                                               bb.ws)
                mb.mlpblk_backward_fp8_prequant(bb.desc, bb.dy, bb.x, bb.gamma, bb.wq, bb.h, bb.a8, bb.n8, bb.rstd,
                                                bb.scales, bb.dx, bb.dgamma, bb.dw1, bb.dw2, bb.ws, overwrite=first)
            else:
                bb.forward()
                bb.backward(overwrite=first)
            outs.append({k: to_np(getattr(bb, k)) for k in ("y", "h", "rstd", "dx")})
        torch.cuda.synchronize()
        runs.append((outs, {k: to_np(getattr(bb, k)) for k in ("dgamma", "dw1", "dw2")}))
    (outs_a, grads_a), (outs_b, grads_b) = runs
    for a, b in zip(outs_a, outs_b):
        for k in a:
            np.testing.assert_array_equal(a[k], b[k], err_msg=k)
    for k in grads_a:
        assert np.isfinite(grads_b[k]).all(), f"{k}: an element was not written"
        err = oracle.scaled_error(grads_b[k], grads_a[k])
        assert err <= 1e-6, f"{k}: {err}"


def test_fp8_overwrite_with_no_tokens_leaves_zero_gradients():
    import torch
    import mlp_block_backprop_gb300 as mb
    bb = mb.BlockBuffers(0, 256, 512, dtype="bf16", fp8=True)
    for k in ("dgamma", "dw1", "dw2"):
        getattr(bb, k).fill_(float("nan"))
    bb.backward(overwrite=True)
    torch.cuda.synchronize()
    for k in ("dgamma", "dw1", "dw2"):
        assert torch.count_nonzero(getattr(bb, k)).item() == 0, k
