"""The routed ReLU² expert block (grouped tcgen05 GEMMs over the experts' token
segments) against its float64 oracle (oracle.moe), GB300 only.

Tolerance: scaled error 2e-2 per tensor, as for the dense bf16 block (bf16
storage of x_perm, h, a, the experts' outputs, dh and dx; fp32 accumulation).
"""

import numpy as np
import pytest

import oracle
import synth
from oracle import moe as moe_oracle
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


def _run(inp):
    import torch
    import mlp_block_backprop_gb300 as mb
    bb = mb.MoeBuffers(inp.tokens, inp.d, inp.ffn, inp.experts, inp.top_k, eps=inp.eps)
    bb.gamma.copy_(to_dev(inp.gamma, torch.bfloat16))
    bb.w1s.copy_(to_dev(inp.w1s, torch.bfloat16))
    bb.w2s.copy_(to_dev(inp.w2s, torch.bfloat16))
    bb.x.copy_(to_dev(inp.x, torch.bfloat16))
    bb.dy.copy_(to_dev(inp.dy, torch.bfloat16))
    bb.idx.copy_(torch.from_numpy(np.ascontiguousarray(inp.idx, dtype=np.int32)).to("cuda"))
    bb.p.copy_(torch.from_numpy(np.ascontiguousarray(inp.p, dtype=np.float32)).to("cuda"))
    bb.zero_grads()
    bb.forward()
    bb.backward()
    torch.cuda.synchronize()
    return {k: to_np(getattr(bb, k)) for k in ("y", "dx", "dp", "dgamma", "dw1s", "dw2s")}, bb


def _reference(inp, valid=None):
    p = inp.p.astype(np.float64)
    idx = inp.idx.copy()
    if valid is not None:   # slots that select nothing: no contribution
        p = np.where(valid, p, 0.0)
        idx = np.where(valid, idx, 0)
    y, h, o, r = moe_oracle.forward(inp.x, inp.gamma, inp.w1s, inp.w2s, idx, p, inp.eps)
    g = moe_oracle.new_grads(inp.experts, inp.d, inp.ffn)
    dx, dp = moe_oracle.backward(inp.dy, inp.x, inp.gamma, inp.w1s, inp.w2s, idx, p, h, o, r, g)
    return {"y": y, "dx": dx, "dp": dp, "dgamma": g["dgamma"], "dw1s": g["dw1"], "dw2s": g["dw2"]}


def _check(got, ref, skip_dp=None):
    errs = {}
    for k in ref:
        a, b = got[k], ref[k]
        if k == "dp" and skip_dp is not None:
            a, b = a[skip_dp], b[skip_dp]
        errs[k] = oracle.scaled_error(a, b)
    bad = {k: v for k, v in errs.items() if not (v <= TOL)}
    assert not bad, f"scaled error above {TOL}: {bad} (all: {errs})"
    return errs


@pytest.mark.parametrize("shape", [
    (200, 128, 256, 4, 2),     # several segments, each padded
    (333, 200, 328, 3, 2),     # ragged in every dimension
    (64, 64, 128, 8, 1),       # top-1, some experts get no token
    (1, 256, 512, 2, 2),       # a single token in two experts
    (520, 520, 520, 5, 3),     # top-3
    (33000, 64, 128, 4, 2),    # 66000 (token, slot) entries: 65 routing chunks
    # d a multiple of 256: the RMSNorm backward gathers the slot rows by bulk copies
    (300, 256, 256, 4, 3),
    (257, 512, 256, 6, 4),
    (1000, 768, 256, 3, 1),
    (130, 2048, 256, 4, 2),
    (70, 4096, 256, 3, 2),     # 512-thread CTAs
    (45, 4096, 256, 4, 3),
])
def test_moe_against_the_oracle(shape):
    T, d, F, E, k = shape
    inp = synth.make_moe_inputs(T, d, F, E, k, seed=T + d + F + E, eps=1e-5)
    got, _ = _run(inp)
    _check(got, _reference(inp))


def test_moe_expert_without_tokens_and_invalid_ids():
    inp = synth.make_moe_inputs(96, 64, 192, 4, 2, seed=31, eps=1e-6)
    inp.idx = np.where(inp.idx == 2, 3, inp.idx).astype(np.int32)   # expert 2 unused
    inp.idx[inp.idx[:, 0] == inp.idx[:, 1], 1] = 0                   # keep a token's experts distinct
    inp.idx[inp.idx[:, 0] == inp.idx[:, 1], 1] = 1
    valid = np.ones_like(inp.idx, dtype=bool)
    inp.idx[5, 1], inp.idx[17, 0] = -1, 9                            # ids that select nothing
    valid[5, 1] = valid[17, 0] = False
    got, _ = _run(inp)
    _check(got, _reference(inp, valid), skip_dp=valid)
    assert got["dp"][5, 1] == 0.0 and got["dp"][17, 0] == 0.0
    assert not np.any(got["dw1s"][2]) and not np.any(got["dw2s"][2])


@pytest.mark.parametrize("d", [64, 256])
def test_moe_invalid_ids_every_norm_path(d):
    """Slots that select nothing (ids -1 and E) at both RMSNorm-backward paths
    (register rows for d = 64, bulk-copied slot rows for d = 256)."""
    inp = synth.make_moe_inputs(160, d, 256, 4, 3, seed=40 + d, eps=1e-6)
    valid = np.ones_like(inp.idx, dtype=bool)
    for t, j, e in ((3, 0, -1), (3, 2, 4), (50, 1, -7), (159, 2, 4)):
        inp.idx[t, j] = e
        valid[t, j] = False
    inp.idx[7, :] = -1                                               # a token with no expert at all
    valid[7, :] = False
    got, _ = _run(inp)
    _check(got, _reference(inp, valid), skip_dp=valid)
    assert np.all(got["dp"][~valid] == 0.0)
    # a token without experts: y = x and dx = dy exactly (bf16 round trip)
    np.testing.assert_array_equal(got["y"][7], inp.x[7].astype(np.float64))
    np.testing.assert_array_equal(got["dx"][7], inp.dy[7].astype(np.float64))


def test_moe_outputs_are_deterministic():
    inp = synth.make_moe_inputs(300, 128, 384, 4, 2, seed=5)
    a, _ = _run(inp)
    b, _ = _run(inp)
    for k in ("y", "dx", "dp", "dgamma"):
        np.testing.assert_array_equal(a[k], b[k])


def test_moe_one_expert_is_the_dense_block():
    """E = 1, k = 1, p = 1: the same outputs as the dense block's kernels."""
    import mlp_block_backprop_gb300 as mb  # noqa: F401
    from helpers import run_gpu
    dense = synth.make_inputs(tokens=256, d=128, ffn=512, dtype="bf16", seed=8, n_mb=1, eps=1e-6)
    inp = synth.MoeInputs(name="one", tokens=256, d=128, ffn=512, experts=1, top_k=1, eps=1e-6,
                          gamma=dense.gamma, w1s=dense.w1[None], w2s=dense.w2[None], x=dense.x[0],
                          dy=dense.dy[0], idx=np.zeros((256, 1), np.int32), p=np.ones((256, 1), np.float32))
    got, _ = _run(inp)
    outs, grads, _ = run_gpu(dense)
    assert oracle.scaled_error(got["y"], outs[0]["y"]) <= 1e-2
    assert oracle.scaled_error(got["dx"], outs[0]["dx"]) <= 1e-2
    assert oracle.scaled_error(got["dw1s"][0], grads["dw1"]) <= 1e-2
    assert oracle.scaled_error(got["dw2s"][0], grads["dw2"]) <= 1e-2


@pytest.mark.slow
def test_moe_full_size_sampled():
    """The 8-expert top-2 workload at its full size (8192 tokens, d 2048, ffn 1024
    per expert), in the calls bench.py times, on sampled outputs the oracle
    computes alone: y, dx and d_routing_weights of 48 tokens (a token's outputs
    depend on its own row only), and whole rows of every expert's dW1 and whole
    columns of dW2 at 12 ffn indices (the ReLU^2 expert is separable over ffn, so
    the oracle over all tokens with W1 cut to those rows and W2 to those columns
    gives exactly those gradients).  dgamma needs every token's full dn and is
    left to the smaller cases."""
    inp = synth.moe_config_inputs("moe_e8k2")
    got, _ = _run(inp)
    rng = np.random.default_rng(2024)
    toks = np.sort(rng.choice(inp.tokens, size=48, replace=False))
    fs = np.sort(rng.choice(inp.ffn, size=12, replace=False))
    p = inp.p.astype(np.float64)

    y, h, o, r = moe_oracle.forward(inp.x[toks], inp.gamma, inp.w1s, inp.w2s, inp.idx[toks], p[toks], inp.eps)
    g = moe_oracle.new_grads(inp.experts, inp.d, inp.ffn)
    dx, dp = moe_oracle.backward(inp.dy[toks], inp.x[toks], inp.gamma, inp.w1s, inp.w2s, inp.idx[toks], p[toks],
                                 h, o, r, g)
    errs = {"y": oracle.scaled_error(got["y"][toks], y), "dx": oracle.scaled_error(got["dx"][toks], dx),
            "dp": oracle.scaled_error(got["dp"][toks], dp)}

    w1c, w2c = inp.w1s[:, fs, :], inp.w2s[:, :, fs]
    y2, h2, o2, r2 = moe_oracle.forward(inp.x, inp.gamma, w1c, w2c, inp.idx, p, inp.eps)
    g2 = moe_oracle.new_grads(inp.experts, inp.d, len(fs))
    moe_oracle.backward(inp.dy, inp.x, inp.gamma, w1c, w2c, inp.idx, p, h2, o2, r2, g2)
    errs["dw1"] = oracle.scaled_error(got["dw1s"][:, fs, :], g2["dw1"])
    errs["dw2"] = oracle.scaled_error(got["dw2s"][:, :, fs], g2["dw2"])
    bad = {k: v for k, v in errs.items() if not (v <= TOL)}
    assert not bad, f"scaled error above {TOL}: {bad} (all: {errs})"


def test_moe_interleaved_writers_and_readers_in_a_graph():
    """Stream kernels writing x and dy right before the calls and reading every
    output right after, one step captured as a CUDA graph and replayed twice
    with zeroed gradients in between: the same results as the oracle (the
    backward's grouped GEMM pairs overlap at their launch boundary)."""
    import torch
    import mlp_block_backprop_gb300 as mb
    inp = synth.make_moe_inputs(600, 256, 512, 4, 2, seed=41, eps=1e-5)
    bb = mb.MoeBuffers(inp.tokens, inp.d, inp.ffn, inp.experts, inp.top_k, eps=inp.eps)
    bf = torch.bfloat16
    bb.gamma.copy_(to_dev(inp.gamma, bf))
    bb.w1s.copy_(to_dev(inp.w1s, bf))
    bb.w2s.copy_(to_dev(inp.w2s, bf))
    bb.idx.copy_(torch.from_numpy(np.ascontiguousarray(inp.idx, dtype=np.int32)).to("cuda"))
    bb.p.copy_(torch.from_numpy(np.ascontiguousarray(inp.p, dtype=np.float32)).to("cuda"))
    xd, dyd = to_dev(inp.x, bf), to_dev(inp.dy, bf)
    keep = {k: torch.empty_like(getattr(bb, k)) for k in ("y", "dx", "dp")}

    def step():
        bb.zero_grads()
        bb.x.copy_(xd)
        bb.forward()
        keep["y"].copy_(bb.y)
        bb.dy.copy_(dyd)
        bb.backward()
        keep["dx"].copy_(bb.dx)
        keep["dp"].copy_(bb.dp)

    step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    ref = _reference(inp)
    for _ in range(2):
        for t in keep.values():
            t.fill_(5.0)
        bb.x.fill_(3.0)
        bb.dy.fill_(3.0)
        g.replay()
        torch.cuda.synchronize()
        got = {k: to_np(v) for k, v in keep.items()}
        got.update({k: to_np(getattr(bb, k)) for k in ("dgamma", "dw1s", "dw2s")})
        _check(got, ref)
