"""The recompute variant (save x and rstd only; rebuild h and a in the backward)
against the float64 oracle and against the saving path (GB300 only).

The variant's contract: the forward's y and rstd are exactly the saving path's
(same kernels and schedule), and the backward's dx and dgamma are too, because
the recomputed h and a are the forward's bits; the fp32 `+=` weight gradients may
differ in the order of their stream-K additions only.
"""

import numpy as np
import pytest

import oracle
import synth
from helpers import TOL, to_dev, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mlp_block_backprop_gb300 as mb  # noqa: F401  (fails loudly if unbuilt)
    yield
    assert mb.mlpblk_last_error() == mb.MLPBLK_OK


def _run(inp, recompute):
    """Forward + backward of every microbatch; per-microbatch y, rstd, dx and the grads."""
    import torch
    import mlp_block_backprop_gb300 as mb
    bb = mb.BlockBuffers(inp.tokens, inp.d, inp.ffn, dtype=inp.dtype, eps=inp.eps, recompute=recompute)
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
        outs.append({k: getattr(bb, k).clone() for k in ("y", "rstd", "dx")})
    if inp.grad_scale is not None:
        bb.scale_grads(inp.grad_scale)
    torch.cuda.synchronize()
    grads = {k: getattr(bb, k).clone() for k in ("dgamma", "dw1", "dw2")}
    return outs, grads


def _against_oracle(inp, outs, grads):
    ref_outs, ref_grads = oracle.run_workload(inp)
    tol = TOL[inp.dtype]
    errs = {}
    for i, (g, r) in enumerate(zip(outs, ref_outs)):
        for k, rk in (("y", "y"), ("rstd", "r"), ("dx", "dx")):
            errs[f"{k}[{i}]"] = oracle.scaled_error(to_np(g[k]), r[rk])
    for k in ("dgamma", "dw1", "dw2"):
        errs[k] = oracle.scaled_error(to_np(grads[k]), ref_grads[k])
    bad = {k: v for k, v in errs.items() if not (v <= tol)}
    assert not bad, f"scaled error above {tol}: {bad}"


def _against_saving_path(inp, outs, grads):
    import torch
    ref_outs, ref_grads = _run(inp, recompute=False)
    for i, (g, r) in enumerate(zip(outs, ref_outs)):
        for k in ("y", "rstd", "dx"):
            assert torch.equal(g[k], r[k]), f"{k}[{i}] differs from the saving path"
    assert torch.equal(grads["dgamma"], ref_grads["dgamma"])
    for k in ("dw1", "dw2"):
        err = oracle.scaled_error(to_np(grads[k]), to_np(ref_grads[k]))
        assert err <= 1e-6, f"{k}: {err}"


@pytest.mark.parametrize("case", ["tiny_fp32", "small_bf16_accum4"])
def test_recompute_configs(case):
    inp = synth.config_inputs(case)
    outs, grads = _run(inp, recompute=True)
    _against_oracle(inp, outs, grads)
    _against_saving_path(inp, outs, grads)


@pytest.mark.parametrize("shape", [(333, 200, 328), (1, 256, 512), (77, 136, 1032)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_recompute_ragged(shape, dtype):
    T, d, F = shape
    inp = synth.make_inputs(tokens=T, d=d, ffn=F, dtype=dtype, seed=T + d + F, n_mb=2, eps=1e-5)
    outs, grads = _run(inp, recompute=True)
    _against_oracle(inp, outs, grads)
    _against_saving_path(inp, outs, grads)


def test_recompute_block_120m_matches_saving_path():
    inp = synth.config_inputs("block_120m")
    outs, grads = _run(inp, recompute=True)
    _against_saving_path(inp, outs, grads)
    # and the oracle on a sample of rows and units (the full oracle is slow here)
    from helpers import sampled_reference
    rows = np.array([0, 1, 777, 4096, 8191])
    units = np.array([0, 5, 1500, 3071])
    ref_rows, dw2_cols, dw1_rows = sampled_reference(inp, rows, units)
    tol = TOL[inp.dtype]
    for k, rk in (("y", "y"), ("rstd", "r"), ("dx", "dx")):
        got = to_np(outs[0][k])[rows]
        assert oracle.scaled_error(got, ref_rows[0][rk]) <= tol, k
    assert oracle.scaled_error(to_np(grads["dw2"])[:, units], dw2_cols) <= tol
    assert oracle.scaled_error(to_np(grads["dw1"])[units], dw1_rows) <= tol


def test_recompute_workspace_contract():
    import torch
    import mlp_block_backprop_gb300 as mb
    d = mb.make_desc(256, 128, 512)
    small, big = mb.mlpblk_workspace_size(d), mb.mlpblk_workspace_size_recompute(d)
    assert big >= small + 2 * 256 * 512 * 2
    bb = mb.BlockBuffers(256, 128, 512, recompute=True)
    short = torch.empty(small, dtype=torch.uint8, device="cuda")
    with pytest.raises(mb.MlpBlkError) as e:
        mb.mlpblk_forward_recompute(bb.desc, bb.x, bb.gamma, bb.w1, bb.w2, bb.y, bb.rstd, short)
    assert e.value.code == mb.MLPBLK_EWORKSPACE
    with pytest.raises(mb.MlpBlkError) as e:
        mb.mlpblk_backward_recompute(bb.desc, bb.dy, bb.x, bb.gamma, bb.w1, bb.w2, bb.rstd, bb.dx,
                                     bb.dgamma, bb.dw1, bb.dw2, short)
    assert e.value.code == mb.MLPBLK_EWORKSPACE
