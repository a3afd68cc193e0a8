"""CUDA path vs the float64 oracle on the same seeded inputs (GB300 only).

Tolerances: max scaled error max|gpu - oracle| / max|oracle| per tensor, 2e-2 for
the bf16 workloads and 1e-5 for the fp32 one.  Cases span several tiles and
ragged tails in every GEMM dimension, plus the degenerate cases of the method.
"""

import numpy as np
import pytest

import oracle
import synth
from helpers import GRAD_KEYS, OUT_KEYS, TOL, compare, gpu_buffers, run_gpu, to_dev, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mlp_block_backprop_gb300 as mb  # noqa: F401  (fails loudly if unbuilt)
    yield
    assert mb.mlpblk_last_error() == mb.MLPBLK_OK


def _check(inp):
    outs, grads, _ = run_gpu(inp)
    ref_outs, ref_grads = oracle.run_workload(inp)
    return compare(outs, grads, ref_outs, ref_grads, TOL[inp.dtype])


def test_tiny_fp32_config():
    _check(synth.config_inputs("tiny_fp32"))


def test_small_bf16_accum4_config():
    _check(synth.config_inputs("small_bf16_accum4"))


@pytest.mark.parametrize("shape", [
    (333, 200, 328),    # ragged in every GEMM dimension, several tiles
    (129, 64, 264),     # one row past a tile; K below one stage in the W1 GEMM
    (1, 256, 512),      # a single token
    (40, 8, 8),         # the narrowest widths (one 16-byte row)
    (77, 136, 1032),    # ffn spans five 256-wide tiles with a ragged tail
    (520, 520, 520),
    (300, 4096, 520),   # the widest d_model the library takes
    (97, 4088, 264),    # the widest ragged d_model (4096 - 8)
])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_ragged_shapes(shape, dtype):
    T, d, F = shape
    _check(synth.make_inputs(tokens=T, d=d, ffn=F, dtype=dtype, seed=T + d + F, n_mb=2, eps=1e-5))


def test_block_120m_config_full():
    _check(synth.config_inputs("block_120m"))


def test_empty_microbatch_touches_nothing():
    import torch
    import mlp_block_backprop_gb300 as mb
    inp = synth.make_inputs(tokens=16, d=64, ffn=128, seed=1)
    bb = gpu_buffers(inp)
    for t in (bb.y, bb.h, bb.a, bb.dx):
        t.fill_(7.0)
    bb.rstd.fill_(7.0)
    bb.dgamma.fill_(3.0)
    desc = mb.make_desc(0, inp.d, inp.ffn, inp.eps)
    mb.mlpblk_forward(desc, bb.x, bb.gamma, bb.w1, bb.w2, bb.y, bb.h, bb.a, bb.rstd, bb.ws)
    mb.mlpblk_backward(desc, bb.dy, bb.x, bb.gamma, bb.w1, bb.w2, bb.h, bb.a, bb.rstd, bb.dx,
                       bb.dgamma, bb.dw1, bb.dw2, bb.ws)
    torch.cuda.synchronize()
    assert torch.all(bb.y == 7.0) and torch.all(bb.rstd == 7.0) and torch.all(bb.dgamma == 3.0)


def test_zero_upstream_gradient_keeps_grads_bitwise():
    import torch
    inp = synth.make_inputs(tokens=300, d=256, ffn=512, seed=5)
    bb = gpu_buffers(inp)
    bb.x.copy_(to_dev(inp.x[0], bb.dt))
    bb.dy.zero_()
    g = torch.Generator(device="cuda").manual_seed(0)
    for t in (bb.dgamma, bb.dw1, bb.dw2):
        t.copy_(torch.randn(t.shape, generator=g, device="cuda"))
    before = [t.clone() for t in (bb.dgamma, bb.dw1, bb.dw2)]
    bb.forward()
    bb.backward()
    torch.cuda.synchronize()
    assert torch.all(bb.dx == 0)
    for b, t in zip(before, (bb.dgamma, bb.dw1, bb.dw2)):
        assert torch.equal(b, t)


def test_w2_zero_gives_identity_residual():
    import torch
    inp = synth.make_inputs(tokens=200, d=128, ffn=384, seed=6)
    bb = gpu_buffers(inp)
    bb.w2.zero_()
    bb.x.copy_(to_dev(inp.x[0], bb.dt))
    bb.dy.copy_(to_dev(inp.dy[0], bb.dt))
    bb.zero_grads()
    bb.forward()
    bb.backward()
    torch.cuda.synchronize()
    assert torch.equal(bb.y, bb.x)
    assert torch.equal(bb.dx, bb.dy)
    assert not torch.any(bb.dw1) and not torch.any(bb.dgamma)


def test_two_backward_calls_accumulate():
    import torch
    inp = synth.make_inputs(tokens=384, d=256, ffn=768, seed=7)
    bb = gpu_buffers(inp)
    bb.x.copy_(to_dev(inp.x[0], bb.dt))
    bb.dy.copy_(to_dev(inp.dy[0], bb.dt))
    bb.zero_grads()
    bb.forward()
    bb.backward()
    once = [t.clone() for t in (bb.dgamma, bb.dw1, bb.dw2)]
    bb.backward()
    torch.cuda.synchronize()
    for o, t in zip(once, (bb.dgamma, bb.dw1, bb.dw2)):
        assert oracle.scaled_error(to_np(t), 2.0 * to_np(o)) <= 1e-6
    bb.scale_grads(0.5)
    torch.cuda.synchronize()
    for o, t in zip(once, (bb.dgamma, bb.dw1, bb.dw2)):
        assert oracle.scaled_error(to_np(t), to_np(o)) <= 1e-6


@pytest.mark.parametrize("graph", [False, True])
def test_interleaved_writers_and_readers(graph):
    """Stream kernels that write an input just before a call, or read an output
    just after it, see the call's reads and writes in order: three microbatches
    with x and dy copied in between the calls and every output copied out right
    after, eager and as one CUDA graph, match the oracle's accumulation."""
    import torch
    inp = synth.make_inputs(tokens=700, d=384, ffn=1032, seed=21, n_mb=3)
    bb = gpu_buffers(inp)
    xs = [to_dev(x, bb.dt) for x in inp.x]
    dys = [to_dev(g, bb.dt) for g in inp.dy]
    keep = {k: [torch.empty_like(getattr(bb, k)) for _ in inp.x] for k in OUT_KEYS}
    for k in OUT_KEYS:
        getattr(bb, k).fill_(3.0)

    def steps():
        bb.zero_grads()
        for i in range(len(xs)):
            bb.x.copy_(xs[i])
            bb.forward()
            for k in ("y", "h", "a", "rstd"):
                keep[k][i].copy_(getattr(bb, k))
            bb.dy.copy_(dys[i])
            bb.backward()
            keep["dx"][i].copy_(bb.dx)

    if graph:
        steps()  # warm-up outside the capture (tensor maps, attributes)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            steps()
        for k in OUT_KEYS:
            for t in keep[k]:
                t.fill_(5.0)
        g.replay()
    else:
        steps()
    torch.cuda.synchronize()
    outs = [{k: to_np(keep[k][i]) for k in OUT_KEYS} for i in range(len(xs))]
    grads = {k: to_np(getattr(bb, k)) for k in GRAD_KEYS}
    ref_outs, ref_grads = oracle.run_workload(inp)
    compare(outs, grads, ref_outs, ref_grads, TOL[inp.dtype])


def test_outputs_stay_inside_their_buffers():
    """Guard bands around every output: a write outside the tensor changes them."""
    import torch
    import mlp_block_backprop_gb300 as mb
    T, d, F = 201, 200, 328
    inp = synth.make_inputs(tokens=T, d=d, ffn=F, seed=8)
    G = 1024  # guard elements on each side (keeps 16-byte alignment)
    dt = torch.bfloat16

    def guarded(n, dtype, fill):
        full = torch.full((n + 2 * G,), fill, dtype=dtype, device="cuda")
        return full, full[G:G + n]

    bufs = {}
    for name, n, dtype in [("y", T * d, dt), ("h", T * F, dt), ("a", T * F, dt), ("rstd", T, torch.float32),
                           ("dx", T * d, dt), ("dgamma", d, torch.float32), ("dw1", F * d, torch.float32),
                           ("dw2", d * F, torch.float32)]:
        bufs[name] = guarded(n, dtype, 0.0 if name.startswith("d") and name != "dx" else 5.0)
    for name in ("dgamma", "dw1", "dw2"):
        bufs[name][1].zero_()
    desc = mb.make_desc(T, d, F, inp.eps)
    ws_n = mb.mlpblk_workspace_size(desc)
    ws_full, ws = guarded(ws_n, torch.uint8, 0)
    x, dy = to_dev(inp.x[0], dt), to_dev(inp.dy[0], dt)
    g, w1, w2 = to_dev(inp.gamma, dt), to_dev(inp.w1, dt), to_dev(inp.w2, dt)
    B = {k: v[1] for k, v in bufs.items()}
    mb.mlpblk_forward(desc, x, g, w1, w2, B["y"], B["h"], B["a"], B["rstd"], ws)
    mb.mlpblk_backward(desc, dy, x, g, w1, w2, B["h"], B["a"], B["rstd"], B["dx"], B["dgamma"],
                       B["dw1"], B["dw2"], ws)
    torch.cuda.synchronize()
    for name, (full, _) in bufs.items():
        want = 0.0 if name.startswith("d") and name != "dx" else 5.0
        assert torch.all(full[:G] == want) and torch.all(full[-G:] == want), name
    assert torch.all(ws_full[:G] == 0) and torch.all(ws_full[-G:] == 0)


def test_no_device_error_recorded():
    import mlp_block_backprop_gb300 as mb
    inp = synth.make_inputs(tokens=256, d=128, ffn=256, seed=9)
    run_gpu(inp, keep_outputs=False)
    assert mb.mlpblk_last_error() == mb.MLPBLK_OK
