"""Float64 oracle of the routed ReLU² expert block: the pre-norm residual shell
around a mixture of ReLU² experts with a fixed (given) top-k dispatch.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle``: only ``tests/``,
``__graft_entry__.smoke()`` and the CPU legs of ``bench.py`` may import it; the
CUDA library never calls it and shares no code with it.

Sources (page title -- section):

* "Nemotron Kernels From Inference To Backpropagation" -- "Kernel 4: Routed ReLU2
  MoE Inference And Backpropagation": for the selected expert set of a token the
  output is the weighted sum of the selected experts' outputs; the product rule
  gives a gradient for each mixture weight and each expert output, and the sum
  rule adds the expert input gradients where they meet; each active expert runs
  the dense ReLU² reverse equations; the routed backward returns d_hidden,
  d_routing_weights, d_expert_up and d_expert_down.
* same page -- "Backpropagation Boundary: Hard Top-K Has No Ordinary
  Derivative": the dispatch (the integer expert ids) is held fixed and only the
  selected mixture weights are differentiated.
* the dense block (``oracle``): RMSNorm shell, ReLU² expert, += gradients.

Readings: the block is y = x + sum_j p[t,j] * E_{idx[t,j]}(n_t) with n = RMSNorm(x)
and E_e(n) = W2_e relu(W1_e n)^2, experts stored W1[e] [ffn, d], W2[e] [d, ffn];
idx [T, k] int expert ids (a token may select an expert at most once), p [T, k]
the mixture weights as given (no renormalisation here); no shared experts.
"""

from __future__ import annotations

import numpy as np

import oracle as _plain


def forward(x, gamma, w1s, w2s, idx, p, eps):
    """Returns (y[T,d], h[T,k,ffn], o[T,k,d], r[T]): h the kept pre-activations and
    o the selected experts' outputs (both per token and slot)."""
    x = np.asarray(x, dtype=np.float64)
    w1s = np.asarray(w1s, dtype=np.float64)
    w2s = np.asarray(w2s, dtype=np.float64)
    p = np.asarray(p, dtype=np.float64)
    n, r = _plain.rmsnorm_forward(x, gamma, eps)
    T, k = idx.shape
    ffn, d = w1s.shape[1], w1s.shape[2]
    h = np.zeros((T, k, ffn))
    o = np.zeros((T, k, d))
    for t in range(T):
        for j in range(k):
            e = int(idx[t, j])
            h[t, j] = w1s[e] @ n[t]                            # project up
            o[t, j] = w2s[e] @ _plain.relu_squared(h[t, j])    # activate, project down
    y = x + np.einsum("tj,tjd->td", p, o)                      # weight, combine, residual
    return y, h, o, r


def new_grads(num_experts, d, ffn):
    return {"dgamma": np.zeros(d), "dw1": np.zeros((num_experts, ffn, d)),
            "dw2": np.zeros((num_experts, d, ffn))}


def backward(dy, x, gamma, w1s, w2s, idx, p, h, o, r, grads):
    """Adds d_expert_up (dw1), d_expert_down (dw2) and dgamma into grads; returns
    (d_hidden dx[T,d], d_routing_weights dp[T,k])."""
    dy = np.asarray(dy, dtype=np.float64)
    x = np.asarray(x, dtype=np.float64)
    w1s = np.asarray(w1s, dtype=np.float64)
    w2s = np.asarray(w2s, dtype=np.float64)
    p = np.asarray(p, dtype=np.float64)
    T, k = idx.shape
    d = x.shape[1]
    n = x * r[:, None] * np.asarray(gamma, dtype=np.float64)[None, :]
    dp = np.einsum("td,tjd->tj", dy, o)            # product rule: the weight's gradient
    dn = np.zeros((T, d))
    for t in range(T):
        for j in range(k):
            e = int(idx[t, j])
            do = p[t, j] * dy[t]                   # product rule: the expert output's gradient
            a = _plain.relu_squared(h[t, j])
            grads["dw2"][e] += np.outer(do, a)
            dh = (do @ w2s[e]) * _plain.relu_squared_grad(h[t, j])
            grads["dw1"][e] += np.outer(dh, n[t])
            dn[t] += dh @ w1s[e]                   # sum rule: the experts meet at n
    dx_norm, dgamma = _plain.rmsnorm_backward(dn, x, gamma, r)
    grads["dgamma"] += dgamma
    return dy + dx_norm, dp
