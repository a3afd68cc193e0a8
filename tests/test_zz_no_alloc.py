"""mlpblk_rmsnorm_backward_noalloc -- the RMSNorm backward for callers that
cannot allocate device scratch (engines that plan all device memory at start-up
and give extensions no allocator; threads that must not stall on cudaMalloc's
implicit synchronisation).

Checked two ways: against the workspace path of mlpblk_backward, which runs the
same row kernel on the same quantities, on two calls in a row; and against the
float64 oracle's RMSNorm backward on the same dn, element by element, with the
dgamma buffer starting from non-zero values so that the += contract is checked
too, up to the widest row the fixed array holds (d_model 4096, where 256 partial
rows each sum 32 of 8192 tokens).

Kept in a file of its own that pytest collects last, so a run stopping at the
first failure has run every other test before this one.
"""

import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mb():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import mlp_block_backprop_gb300
    return mlp_block_backprop_gb300


def _reference_and_dn(mb, inp):
    """dx and dgamma from mlpblk_backward, and the gradient dn of the normalised
    output built in fp32 from the same saved h (the input of the new call)."""
    import torch
    dt = torch.bfloat16
    dev = lambda a: torch.from_numpy(a).to("cuda").to(dt)
    bb = mb.BlockBuffers(inp.tokens, inp.d, inp.ffn, eps=inp.eps)
    bb.gamma.copy_(dev(inp.gamma))
    bb.w1.copy_(dev(inp.w1))
    bb.w2.copy_(dev(inp.w2))
    bb.x.copy_(dev(inp.x[0]))
    bb.dy.copy_(dev(inp.dy[0]))
    bb.zero_grads()
    bb.forward()
    bb.backward()
    h = bb.h.float()
    dn = ((bb.dy.float() @ bb.w2.float()) * 2.0 * torch.relu(h)) @ bb.w1.float()
    torch.cuda.synchronize()
    return bb, dn.contiguous()


@pytest.mark.parametrize("T", [300])
def test_noalloc_norm_backward_matches_workspace_path(mb, T):
    import torch
    tol = 2e-2
    # two calls in a row with different shapes: the second one must not see
    # anything the first one left in the shared array
    for call, (tokens, seed) in enumerate([(T, 11), (77, 12)]):
        inp = synth.make_inputs(tokens=tokens, d=256, ffn=512, seed=seed)
        bb, dn = _reference_and_dn(mb, inp)
        dx = torch.empty_like(bb.dx)
        dgamma = torch.zeros_like(bb.dgamma)
        desc = mb.make_desc(tokens, inp.d, inp.ffn, inp.eps)
        mb.mlpblk_rmsnorm_backward_noalloc(desc, bb.x, dn, bb.dy, bb.gamma, bb.rstd, dx, dgamma)
        torch.cuda.synchronize()
        assert mb.mlpblk_last_error() == mb.MLPBLK_OK
        got_dx = dx.float().cpu().numpy().astype(np.float64)
        ref_dx = bb.dx.float().cpu().numpy().astype(np.float64)
        got_dg = dgamma.cpu().numpy().astype(np.float64)
        ref_dg = bb.dgamma.cpu().numpy().astype(np.float64)
        assert oracle.scaled_error(got_dx, ref_dx) <= tol, call
        assert oracle.scaled_error(got_dg, ref_dg) <= tol, call


def _oracle_case(mb, tokens, d, dtype, seed):
    """One call on seeded inputs (dn drawn directly, rstd of the drawn x, dgamma
    prefilled with seeded values) and the float64 oracle on the same inputs.
    Returns the scaled errors of dx and of the dgamma increment."""
    import torch
    inp = synth.make_inputs(tokens=tokens, d=d, ffn=8, dtype=dtype, seed=seed)
    rng = np.random.default_rng(seed + 1000)
    x = inp.x[0].astype(np.float64)
    dy = inp.dy[0].astype(np.float64)
    gamma = inp.gamma.astype(np.float64)
    dn = rng.standard_normal((tokens, d)).astype(np.float32)
    rstd = (1.0 / np.sqrt(np.mean(x * x, axis=1) + inp.eps)).astype(np.float32)
    prefill = rng.standard_normal(d).astype(np.float32)

    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    on_dev = lambda a, t=dt: torch.from_numpy(np.ascontiguousarray(a)).to("cuda").to(t)
    x_d, dy_d, g_d = on_dev(inp.x[0]), on_dev(inp.dy[0]), on_dev(inp.gamma)
    dn_d, r_d = on_dev(dn, torch.float32), on_dev(rstd, torch.float32)
    dx_d = torch.empty_like(x_d)
    dg_d = on_dev(prefill, torch.float32)
    code = mb.MLPBLK_BF16 if dtype == "bf16" else mb.MLPBLK_FP32
    desc = mb.make_desc(tokens, d, 8, inp.eps, code)
    mb.mlpblk_rmsnorm_backward_noalloc(desc, x_d, dn_d, dy_d, g_d, r_d, dx_d, dg_d)
    torch.cuda.synchronize()
    assert mb.mlpblk_last_error() == mb.MLPBLK_OK

    dx_norm, dg = oracle.rmsnorm_backward(dn, x, gamma, rstd.astype(np.float64))
    ref_dx = dy + dx_norm
    got_dx = dx_d.float().cpu().numpy().astype(np.float64)
    # the increment this call added on top of the prefilled values
    got_inc = dg_d.cpu().numpy().astype(np.float64) - prefill.astype(np.float64)
    return oracle.scaled_error(got_dx, ref_dx), oracle.scaled_error(got_inc, dg)


@pytest.mark.parametrize("tokens,d,dtype,tol", [
    (300, 256, "bf16", 2e-2),
    (8192, 4096, "bf16", 2e-2),   # the widest row the array holds: 256 partial rows
    (1000, 200, "bf16", 2e-2),    # a width that is not a multiple of 64
    (77, 136, "f32", 1e-5),
    (4096, 4096, "f32", 1e-5),
])
def test_noalloc_norm_backward_matches_oracle(mb, tokens, d, dtype, tol):
    e_dx, e_dg = _oracle_case(mb, tokens, d, dtype, seed=tokens + d)
    assert e_dx <= tol, e_dx
    assert e_dg <= tol, e_dg


def test_noalloc_rejects_what_it_cannot_hold(mb):
    import ctypes
    p = [0x10000 * (i + 1) for i in range(7)]
    too_wide = mb.make_desc(64, 8192, 8)
    assert mb.lib.mlpblk_rmsnorm_backward_noalloc(ctypes.byref(too_wide), *p, None) == mb.MLPBLK_ENOTSUP
    ragged = mb.make_desc(64, 260, 8)
    assert mb.lib.mlpblk_rmsnorm_backward_noalloc(ctypes.byref(ragged), *p, None) == mb.MLPBLK_ENOTSUP
    ok_shape = mb.make_desc(64, 256, 8)
    bad = list(p)
    bad[1] = None
    assert mb.lib.mlpblk_rmsnorm_backward_noalloc(ctypes.byref(ok_shape), *bad, None) == mb.MLPBLK_EINVAL
