"""Float64 oracle for the pre-norm residual ReLU² MLP block, forward and backward.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The CUDA
library never calls it and shares no code with it; both sides receive their
inputs from ``synth`` and nothing else.

What it computes is the block's plain definition, written step by step in the
order the pages give it, in float64, with numpy's matrix product as the only
library step (and numpy's sums for the row and column reductions).  There is no
blocking, fusion or algebraic rewriting here: the CUDA path's rewrites (gamma
folded into W1, rstd folded into dh) are checked *against* this file.

Sources (page title -- section):

* "Nemotron Kernels From Inference To Backpropagation" -- "Branches Copy Forward
  And Add Backward" and "Setup: The Shared Transformer Shell": the block is
  y = x + Body(RMSNorm(x)); backward sends g_y straight to x and also through the
  body; RMSNorm backward needs the input, the learned scale and the inverse RMS.
* same page -- "Kernel 3: Dense ReLU2 Inference And Backpropagation": project,
  square of ReLU, project; the input to ReLU² is kept for backward and the
  derivative convention at u = 0 has to be fixed.
* "Reverse-mode automatic differentiation" -- §5 Operators: ``Add`` (g to each
  input), ``Relu`` (g where the output is positive), ``MatMul`` (g·Bᵀ and Aᵀ·g)
  and ``LayerNorm`` (dx = (ĝ − mean(ĝ) − x̂·mean(ĝ·x̂))/σ, dγ = Σ g·x̂).
* "grow_a_language_model_backprop" -- accumulation across microbatches: backward
  adds into the gradient buffers (+=), scale_grads(1/n) after the microbatches,
  zero_grads() before the next step.

Readings where the pages are silent (the display equations of the first page
were lost in extraction):

* block formula: y = x + W2·relu(W1·n)² with n = RMSNorm(x), the square taken on
  the ReLU output; weights stored as W1[ffn, d] and W2[d, ffn] (row = output unit);
* RMSNorm: n = x·r·γ with r = 1/sqrt(mean_k x² + eps), eps inside the root, mean
  over the model dimension ("inverse RMS" = root *mean* square);
* RMSNorm backward: the ``LayerNorm`` rule of the autograd page with the mean
  subtraction removed (no centring, no bias): with x̂ = x·r and ĝ = dn·γ,
  dx_norm = r·(ĝ − x̂·mean_k(ĝ·x̂)), dγ = Σ_t dn·x̂;
* d/dh relu(h)² = 2·relu(h); both one-sided derivatives are 0 at h = 0, so the
  convention at zero is simply 0 (the strict h > 0 test of ``Relu``);
* dx is written (=), the parameter gradients are accumulated (+=).

Every function below is pinned in ``tests/test_oracle.py`` by central finite
differences, a hand-derived worked example, closed forms and invariants.
"""

from __future__ import annotations

import numpy as np


def _f64(v):
    return np.asarray(v, dtype=np.float64)


def relu(h):
    """max(h, 0) with the strict h > 0 test of the autograd page's ``Relu``."""
    h = _f64(h)
    return np.where(h > 0.0, h, 0.0)


def relu_squared(h):
    """The ReLU² activation: relu(h) squared."""
    r = relu(h)
    return r * r


def relu_squared_grad(h):
    """d/dh relu(h)² = 2·relu(h) (0 at h = 0 from both sides)."""
    return 2.0 * relu(h)


def rmsnorm_forward(x, gamma, eps):
    """n = x·r·γ with r[t] = 1/sqrt(mean_k x[t,k]² + eps).  Returns (n, r)."""
    x = _f64(x)
    gamma = _f64(gamma)
    d = x.shape[1]
    mean_sq = np.sum(x * x, axis=1) / d
    r = 1.0 / np.sqrt(mean_sq + eps)
    n = x * r[:, None] * gamma[None, :]
    return n, r


def forward(x, gamma, w1, w2, eps):
    """Block forward on one microbatch.

    x[T,d], gamma[d], w1[ffn,d], w2[d,ffn] -> (y[T,d], h[T,ffn], a[T,ffn], r[T]).
    h is the saved pre-activation, r the saved per-row inverse RMS.
    """
    x = _f64(x)
    n, r = rmsnorm_forward(x, gamma, eps)
    h = n @ _f64(w1).T                 # project
    a = relu_squared(h)                # activate
    y = x + a @ _f64(w2).T             # project, then the identity branch adds x
    return y, h, a, r


def rmsnorm_backward(dn, x, gamma, r):
    """Gradient of n = x·r·γ.  Returns (dx_norm[T,d], dgamma contribution[d])."""
    dn = _f64(dn)
    x = _f64(x)
    gamma = _f64(gamma)
    d = x.shape[1]
    xhat = x * r[:, None]
    g = dn * gamma[None, :]
    mean_gx = np.sum(g * xhat, axis=1) / d
    dx_norm = r[:, None] * (g - xhat * mean_gx[:, None])
    dgamma = np.sum(dn * xhat, axis=0)
    return dx_norm, dgamma


def new_grads(d, ffn):
    """Zeroed float64 gradient buffers {dgamma[d], dw1[ffn,d], dw2[d,ffn]}."""
    return {"dgamma": np.zeros(d), "dw1": np.zeros((ffn, d)), "dw2": np.zeros((d, ffn))}


def backward(dy, x, gamma, w1, w2, h, r, grads):
    """Block backward on one microbatch.

    Adds the microbatch's parameter gradients into ``grads`` (+=) and returns dx,
    which is written, not accumulated.  Uses the saved h and r.
    """
    dy = _f64(dy)
    x = _f64(x)
    w1 = _f64(w1)
    w2 = _f64(w2)
    h = _f64(h)
    a = relu_squared(h)
    da = dy @ w2                                  # g·W2 through y = a·W2ᵀ
    grads["dw2"] += dy.T @ a                      # gᵀ·a
    dh = da * relu_squared_grad(h)                # ReLU² gate
    n = x * r[:, None] * _f64(gamma)[None, :]     # normalised input from the saved r
    dn = dh @ w1                                  # g·W1 through h = n·W1ᵀ
    grads["dw1"] += dh.T @ n                      # gᵀ·n
    dx_norm, dgamma = rmsnorm_backward(dn, x, gamma, r)
    grads["dgamma"] += dgamma
    return dy + dx_norm                           # identity branch adds dy


def scale_grads(grads, s):
    """grads ×= s (the 1/n_microbatches average)."""
    for k in grads:
        grads[k] *= s


def zero_grads(grads):
    """grads = 0."""
    for k in grads:
        grads[k][...] = 0.0


def run_workload(inp, grads=None):
    """Forward + backward over every microbatch of a ``synth.BlockInputs``.

    Returns (per-microbatch list of dicts with y, h, a, r, dx; grads).  Applies
    the workload's grad_scale after the last microbatch when it has one.
    """
    if grads is None:
        grads = new_grads(inp.d, inp.ffn)
    outs = []
    for x, dy in zip(inp.x, inp.dy):
        y, h, a, r = forward(x, inp.gamma, inp.w1, inp.w2, inp.eps)
        dx = backward(dy, x, inp.gamma, inp.w1, inp.w2, h, r, grads)
        outs.append({"y": y, "h": h, "a": a, "r": r, "dx": dx})
    if inp.grad_scale is not None:
        scale_grads(grads, inp.grad_scale)
    return outs, grads


def scaled_error(got, ref):
    """max|got − ref| / max|ref|: the per-tensor error measure of the autograd
    page's oracle tests.  When ref is identically zero, returns max|got|."""
    got = _f64(got)
    ref = _f64(ref)
    if got.shape != ref.shape:
        raise ValueError(f"shape mismatch {got.shape} vs {ref.shape}")
    if got.size == 0:
        return 0.0
    den = np.max(np.abs(ref))
    num = np.max(np.abs(got - ref))
    return float(num if den == 0.0 else num / den)
