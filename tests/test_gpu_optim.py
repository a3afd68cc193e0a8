"""Optimizer-side kernels (gradient norm, clip, AdamW) against the float64
oracle (GB300 only).

Tolerances: the norm is a float32-compensated, float64-combined sum: relative
1e-6.  AdamW runs in float32 on float32 state: per step a few float32 roundings
of w, m, v and the update, so after k steps the scaled error stays below
k * 2^-22; 1e-6 is used for up to 5 steps.  The bf16 working copy is checked
exactly against the round-to-nearest-even of the GPU's own master weights (the
rounding decision is taken on the GPU's float32 value on both sides).
"""

import numpy as np
import pytest

import oracle
import synth
from oracle import optim
from helpers import to_dev, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mlp_block_backprop_gb300 as mb  # noqa: F401
    yield
    assert mb.mlpblk_last_error() == mb.MLPBLK_OK


def _f32(shape, seed, scale=1.0):
    return (np.random.default_rng(seed).standard_normal(shape) * scale).astype(np.float32)


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda")


@pytest.mark.parametrize("d, F", [(256, 1024), (768, 3072), (8, 8)])
def test_grad_norm_and_clip(d, F):
    import torch
    import mlp_block_backprop_gb300 as mb
    desc = mb.make_desc(1, d, F)
    gs = [_f32(d, 1, 3.0), _f32((F, d), 2, 1e-2), _f32((d, F), 3, 0.5)]
    dg = [_dev(g) for g in gs]
    ws = torch.empty(mb.mlpblk_workspace_size(desc), dtype=torch.uint8, device="cuda")
    out = torch.zeros(2, dtype=torch.float32, device="cuda")
    ref = optim.grad_norm(gs)
    max_norm = ref / 3.0
    mb.mlpblk_grad_norm(desc, *dg, max_norm, out[0:1], out[1:2], ws)
    torch.cuda.synchronize()
    norm, c = float(out[0]), float(out[1])
    assert abs(norm - ref) <= 1e-6 * ref
    assert abs(c - optim.clip_coefficient(ref, max_norm)) <= 2e-6 * c
    # fixed partition and order: a second call gives the same bits
    again = torch.zeros(2, dtype=torch.float32, device="cuda")
    mb.mlpblk_grad_norm(desc, *dg, max_norm, again[0:1], again[1:2], ws)
    torch.cuda.synchronize()
    assert torch.equal(out, again)
    # a norm below the bound leaves the scale at exactly 1
    mb.mlpblk_grad_norm(desc, *dg, ref * 2.0, None, again[1:2], ws)
    torch.cuda.synchronize()
    assert float(again[1]) == 1.0
    # clip: every element times the device scalar, as float32 products
    mb.mlpblk_clip_grads(desc, *dg, out[1:2])
    torch.cuda.synchronize()
    for g, t in zip(gs, dg):
        np.testing.assert_array_equal(t.cpu().numpy(), g * np.float32(c))


def _adam_case(n_list, seed):
    rng = np.random.default_rng(seed)
    return [dict(w=rng.standard_normal(n).astype(np.float32), decay=(i != 0)) for i, n in enumerate(n_list)]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_adamw_steps_match_the_oracle(dtype):
    import torch
    import mlp_block_backprop_gb300 as mb
    hp = dict(lr=3e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
    tensors = _adam_case([256, 4096, 1000], 11)
    wt = torch.bfloat16 if dtype == "bf16" else torch.float32
    dev = []
    for t in tensors:
        n = t["w"].size
        dev.append(dict(master=_dev(t["w"]), weight=torch.empty(n, dtype=wt, device="cuda"),
                        m=torch.zeros(n, dtype=torch.float32, device="cuda"),
                        v=torch.zeros(n, dtype=torch.float32, device="cuda"),
                        grad=torch.empty(n, dtype=torch.float32, device="cuda")))
        t.update(w64=t["w"].astype(np.float64), m64=np.zeros(n), v64=np.zeros(n))
    gsc = torch.tensor([0.5], dtype=torch.float32, device="cuda")
    for step in range(1, 6):
        use_scale = step % 2 == 0
        for i, (t, g) in enumerate(zip(tensors, dev)):
            gnp = _f32(t["w"].size, 100 * step + i, 10.0 ** (-i))
            g["grad"].copy_(_dev(gnp))
            gq = gnp.astype(np.float64) * (np.float32(0.5) if use_scale else 1.0)
            optim.adamw_step(t["w64"], gq, t["m64"], t["v64"], step, hp["lr"], hp["beta1"], hp["beta2"],
                             hp["eps"], hp["weight_decay"] if t["decay"] else 0.0)
        mb.mlpblk_adamw_step([(g["master"], g["weight"], g["grad"], g["m"], g["v"], t["decay"])
                              for t, g in zip(tensors, dev)],
                             mb.AdamW(**hp), step, mb.MLPBLK_BF16 if dtype == "bf16" else mb.MLPBLK_FP32,
                             grad_scale=gsc if use_scale else None)
    torch.cuda.synchronize()
    for t, g in zip(tensors, dev):
        master = g["master"].cpu().numpy()
        assert oracle.scaled_error(master.astype(np.float64), t["w64"]) <= 1e-6
        assert oracle.scaled_error(g["m"].cpu().numpy().astype(np.float64), t["m64"]) <= 1e-6
        assert oracle.scaled_error(g["v"].cpu().numpy().astype(np.float64), t["v64"]) <= 1e-6
        work = g["weight"].float().cpu().numpy().astype(np.float64)
        if dtype == "bf16":
            np.testing.assert_array_equal(work, optim.round_to_bf16(master))
        else:
            np.testing.assert_array_equal(work, master.astype(np.float64))


def test_training_step_after_the_block():
    """zero -> forward/backward of 4 microbatches -> x0.25 -> norm -> AdamW with
    the clip scale folded in.  The block's gradients are checked against the
    oracle's; the norm and the update against the oracle applied to the
    gradients the GPU produced (the first Adam step is sign-like, so feeding it
    the oracle's own gradients would test the block's rounding, not the update)."""
    import torch
    import mlp_block_backprop_gb300 as mb
    from helpers import TOL, run_gpu
    inp = synth.config_inputs("small_bf16_accum4")
    _, grads, bb = run_gpu(inp, keep_outputs=False)
    _, ref_grads = oracle.run_workload(inp)
    names = ("dgamma", "dw1", "dw2")
    for k in names:
        assert oracle.scaled_error(grads[k], ref_grads[k]) <= TOL["bf16"], k
    gpu_norm = optim.grad_norm([grads[k] for k in names])
    assert abs(gpu_norm - optim.grad_norm([ref_grads[k] for k in names])) <= TOL["bf16"] * gpu_norm
    max_norm = 0.5 * gpu_norm
    scale = torch.zeros(2, dtype=torch.float32, device="cuda")
    mb.mlpblk_grad_norm(bb.desc, bb.dgamma, bb.dw1, bb.dw2, max_norm, scale[0:1], scale[1:2], bb.ws)
    params = {"dgamma": bb.gamma, "dw1": bb.w1, "dw2": bb.w2}
    src = {"dgamma": inp.gamma, "dw1": inp.w1, "dw2": inp.w2}
    masters = {k: _dev(src[k].astype(np.float32)) for k in names}
    mom = {k: (torch.zeros_like(masters[k]), torch.zeros_like(masters[k])) for k in names}
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    mb.mlpblk_adamw_step([(masters[k], params[k], getattr(bb, k), mom[k][0], mom[k][1], k != "dgamma")
                          for k in names], mb.AdamW(**hp), 1, mb.MLPBLK_BF16, grad_scale=scale[1:2])
    torch.cuda.synchronize()
    assert abs(float(scale[0]) - gpu_norm) <= 1e-6 * gpu_norm
    c = float(scale[1])
    assert abs(c - optim.clip_coefficient(gpu_norm, max_norm)) <= 2e-6 * c
    for k in names:
        w = src[k].astype(np.float64).copy()
        m, v = np.zeros_like(w), np.zeros_like(w)
        g = (grads[k].astype(np.float32) * np.float32(c)).astype(np.float64)
        optim.adamw_step(w, g, m, v, 1, hp["lr"], hp["beta1"], hp["beta2"], hp["eps"],
                         hp["weight_decay"] if k != "dgamma" else 0.0)
        got = masters[k].cpu().numpy().astype(np.float64)
        assert oracle.scaled_error(got, w) <= 1e-6, k
        np.testing.assert_array_equal(to_np(params[k]).reshape(got.shape), optim.round_to_bf16(got))
