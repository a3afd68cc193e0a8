"""Float64 oracle for the optimizer-side steps next to the block: the global
gradient norm, the clipping coefficient, gradient scaling and AdamW.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle``: only ``tests/``,
``__graft_entry__.smoke()`` and the CPU legs of ``bench.py`` may import it; the
CUDA library never calls it and shares no code with it.

Sources (page title -- section):

* "grow_a_language_model_backprop" -- the utility kernels next to the forward /
  backward pairs: a two-stage global gradient-norm reduction and a gradient
  scale, used for gradient clipping; and "optimizer state": AdamW keeps two
  extra buffers per weight, the first moment m and the second moment v; the
  accumulation loop runs scale_grads(1/n), optimizer_step(), zero_grads().
* "Losing small gradient contributions in BF16" (Nemotron 3 Ultra page): small
  contributions vanish next to a large bf16 value, so the state the update
  accumulates into stays float32 (master weights, m, v); the block reads a bf16
  working copy of the weights.

Readings where the pages give no formula (they name the kernels only):

* gradient norm: the L2 norm over every element of every gradient tensor,
  sqrt(sum g^2);
* clipping coefficient: min(1, max_norm / (norm + 1e-6)), applied by scaling
  every gradient element (the common clip-by-global-norm form);
* AdamW: Adam with decoupled weight decay (Loshchilov & Hutter, "Decoupled
  Weight Decay Regularization", Algorithm 2), in the usual implementation order:
  w <- w * (1 - lr*wd); m <- b1*m + (1-b1)*g; v <- b2*v + (1-b2)*g^2;
  w <- w - (lr / (1 - b1^t)) * m / (sqrt(v) / sqrt(1 - b2^t) + eps), t >= 1;
* working copy: the float32 master rounded to bfloat16, to nearest, ties to
  even.
"""

from __future__ import annotations

import numpy as np

CLIP_EPS = 1e-6


def grad_norm(grads):
    """sqrt of the sum of squares of every element of every tensor in `grads`."""
    total = 0.0
    for g in grads:
        g = np.asarray(g, dtype=np.float64)
        total += float(np.sum(g * g))
    return float(np.sqrt(total))


def clip_coefficient(norm, max_norm):
    """Scale that brings a gradient of global norm `norm` to at most `max_norm`."""
    return min(1.0, float(max_norm) / (float(norm) + CLIP_EPS))


def scale(grads, s):
    """Every gradient element times s (in place)."""
    for g in grads:
        g *= s


def adamw_step(w, g, m, v, step, lr, beta1, beta2, eps, weight_decay):
    """One AdamW update of float64 arrays w, m, v from gradient g (in place).
    `step` counts updates from 1."""
    w *= 1.0 - lr * weight_decay
    m *= beta1
    m += (1.0 - beta1) * g
    v *= beta2
    v += (1.0 - beta2) * (g * g)
    bias1 = 1.0 - beta1 ** step
    bias2 = 1.0 - beta2 ** step
    denom = np.sqrt(v) / np.sqrt(bias2) + eps
    w -= (lr / bias1) * (m / denom)


def round_to_bf16(a):
    """Float32 values (given in any float dtype) rounded to bfloat16, to nearest,
    ties to even; returned as float64.  Bit-level: keep the upper 16 bits of the
    float32 pattern after adding 0x7FFF plus the lowest kept bit."""
    bits = np.asarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    keep = (bits >> 16) & 1
    rounded = ((bits + 0x7FFF + keep) >> 16) << 16
    return rounded.astype(np.uint32).view(np.float32).astype(np.float64)
