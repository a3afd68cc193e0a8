"""Float64 oracle of the FP8 (E4M3) operand variant of the block: the same forward
and backward as ``oracle``, with every GEMM operand quantised to E4M3 with a
per-tensor scale at the points listed below, and the products taken exactly
(float64) on the quantised values.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle``: only ``tests/``,
``__graft_entry__.smoke()`` and the CPU legs of ``bench.py`` may import it; the
CUDA library never calls it and shares no code with it.

Sources (page title -- section):

* "Nemotron Kernels From Inference To Backpropagation" -- "Where Quantization
  Fits": quantisation is a storage and arithmetic policy for particular tensor
  edges, the large projection matrices first; training keeps higher-precision
  accumulators and states what is quantised where.
* "grow_a_language_model_backprop" -- the FP8 E4M3 tensor-core experiments next
  to the FP16 GEMM path; precise control of which tensor lives in which
  precision.
* the block itself as in ``oracle`` (forward, the backward rules, += grads).

Readings (the pages name E4M3 but give no recipe):

* format: E4M3 as in the OCP FP8 specification (4 exponent bits, bias 7, 3
  mantissa bits, largest finite value 448, subnormals down to 2^-9, no
  infinities); rounding to nearest, ties to even; values beyond +-448 saturate;
* per-tensor scale: s = amax / 448 with amax = max |v| over the tensor, codes
  q = E4M3(v * (448 / amax)), dequantised value q * s; the two float32
  divisions 448 / amax and amax / 448 are taken in float32 (so both sides make
  the same rounding decisions on the same values);
* the normalised input n' = x * rstd (float32 product) has |n'| <= sqrt(d) <= 64
  for every row, so it is quantised with scale 1 (no amax pass); gamma is folded
  into W1 (W1 * gamma, exact in float32) before W1 is quantised;
* quantisation points: forward n', W1*gamma, a (after its bf16 rounding, the
  saved activation), W2; backward dy, dh (bf16), W2, W1; the wgrads read the
  same quantised a, dy, dh and n';
* everything else (h, the gate, the RMSNorm statistic and backward, the residual
  paths, the += gradients) is as in the bf16 block: h and dh are rounded to bf16
  where the bf16 path rounds them, and the gate reads the kept (bf16) h ("Kernel
  3: Dense ReLU2 ...": the reverse kernel applies the branch to the preserved
  input of ReLU^2) -- here, unlike in the bf16 block, that matters: dh is
  quantised next, and a difference of one bf16 step in dh moves an E4M3 code in
  about one element in sixteen; the accumulators are float32 on the GPU and
  float64 here.
"""

from __future__ import annotations

import numpy as np

import oracle as _plain

E4M3_MAX = 448.0
_MIN_NORMAL_EXP = -6   # smallest normal 2^-6
_MANT_BITS = 3


def e4m3(u):
    """Round float values to the E4M3 grid (nearest, ties to even; saturating)."""
    u = np.asarray(u, dtype=np.float64)
    a = np.abs(u)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))          # a = m * 2^ex, m in [0.5, 1)
    e = np.maximum(ex - 1, _MIN_NORMAL_EXP)             # binade; subnormals share 2^-6's spacing
    spacing = np.exp2(e - _MANT_BITS)
    q = np.rint(a / spacing) * spacing                 # exact: a / spacing is a power-of-two scaling
    q = np.minimum(q, E4M3_MAX)
    return np.copysign(q, u)


def round_to_bf16(a):
    """Float32 values rounded to bfloat16, nearest-even; returned as float64."""
    bits = np.asarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    keep = (bits >> 16) & 1
    rounded = ((bits + 0x7FFF + keep) >> 16) << 16
    return rounded.astype(np.uint32).view(np.float32).astype(np.float64)


def quantize(v, amax=None):
    """Per-tensor E4M3 quantisation of float32 values v: (dequantised values, scale).
    `amax`, when given, is the max |v| of the whole tensor that v is a row block
    of (the scale is the whole tensor's); by default v is the whole tensor."""
    v32 = np.asarray(v, dtype=np.float32)
    if amax is None:
        amax = np.float32(np.max(np.abs(v32))) if v32.size else np.float32(0)
    amax = np.float32(amax)
    if amax == 0:
        return np.zeros(v32.shape), np.float32(1.0)
    inv = np.float32(E4M3_MAX) / amax
    s = amax / np.float32(E4M3_MAX)
    q = e4m3((v32 * inv).astype(np.float32))
    return q * np.float64(s), s


def rstd32(x, eps):
    """The RMSNorm statistic rounded to float32 (the precision the kernels keep)."""
    x = np.asarray(x, dtype=np.float64)
    return (1.0 / np.sqrt(np.mean(x * x, axis=1) + eps)).astype(np.float32)


def _pre_a(x, gamma, w1, eps):
    """The forward up to a (bf16-rounded, before its quantisation): (h, a, n_q, r)."""
    x32 = np.asarray(x, dtype=np.float32)
    r = rstd32(x, eps)
    n_prime = (x32 * r[:, None]).astype(np.float32)          # n' = x * rstd, float32
    n_q = e4m3(n_prime)                                       # scale 1: |n'| <= sqrt(d)
    w1g = (np.asarray(w1, dtype=np.float32) * np.asarray(gamma, dtype=np.float32)[None, :]).astype(np.float32)
    w1g_q, _ = quantize(w1g)
    h = n_q @ w1g_q.T
    a = np.where(h > 0, h, 0.0) ** 2
    return h, round_to_bf16(a.astype(np.float32)), n_q, r


def _pre_dh(dy, h, w2, dy_amax=None):
    """The backward up to dh (bf16-rounded, before its quantisation): (dh, dy_q)."""
    dy_q, _ = quantize(dy, dy_amax)
    w2_q, _ = quantize(w2)
    da = dy_q @ w2_q                                          # [T, F]
    # the gate reads h as the forward keeps it (bf16): the reverse kernel applies
    # the branch to the preserved input of ReLU^2
    hk = round_to_bf16(np.asarray(h, dtype=np.float32))
    dh = da * 2.0 * np.where(hk > 0, hk, 0.0)                 # d relu(h)^2 / dh
    return round_to_bf16(dh.astype(np.float32)), dy_q


def forward(x, gamma, w1, w2, eps, a_amax=None):
    """FP8-operand forward.  Returns (y, h, a_q, n_q, r) with h the float64
    pre-activation (the kernels keep it in bf16), a_q and n_q the dequantised
    GEMM operands the backward reuses.  a_amax: see block_amaxes."""
    h, a, n_q, r = _pre_a(x, gamma, w1, eps)
    a_q, _ = quantize(a, a_amax)
    w2_q, _ = quantize(w2)
    y = np.asarray(x, dtype=np.float64) + a_q @ w2_q.T
    return y, h, a_q, n_q, r.astype(np.float64)


def block_amaxes(x, dy, gamma, w1, w2, eps, dy_amax=None):
    """max |a| and max |dh| (their bf16 values) over a row block of a microbatch,
    dy_amax being the whole dy's max |dy| (dy is an input).  The maxima over all
    blocks are the whole tensors' (a and dh are row-wise given the weights and
    dy's scale), so a large microbatch can be evaluated block by block:
    forward(..., a_amax=) and backward(..., dy_amax=, dh_amax=) then quantise
    each block with the whole tensor's scale."""
    h, a, _, _ = _pre_a(x, gamma, w1, eps)
    dh, _ = _pre_dh(dy, h, w2, dy_amax)
    return np.float32(np.max(np.abs(a))), np.float32(np.max(np.abs(dh)))


def backward(dy, x, gamma, w1, w2, h, a_q, n_q, r, grads, dy_amax=None, dh_amax=None):
    """FP8-operand backward; adds into grads (dgamma, dw1, dw2) and returns dx.
    dy_amax, dh_amax: see block_amaxes."""
    x = np.asarray(x, dtype=np.float64)
    gamma = np.asarray(gamma, dtype=np.float64)
    dh, dy_q = _pre_dh(dy, h, w2, dy_amax)
    dh_q, _ = quantize(dh, dh_amax)
    grads["dw2"] += dy_q.T @ a_q
    w1_q, _ = quantize(w1)
    dn = dh_q @ w1_q                                          # [T, d]
    grads["dw1"] += (dh_q.T @ n_q) * gamma[None, :]           # dW1 = (dh^T n') * gamma
    dx_norm, dgamma = _plain.rmsnorm_backward(dn, x, gamma, r)
    grads["dgamma"] += dgamma
    return np.asarray(dy, dtype=np.float64) + dx_norm


def run_workload(inp, grads=None):
    """FP8-operand forward + backward over every microbatch of a ``synth``
    workload (as ``oracle.run_workload``).  Per microbatch: y, h, r, dx."""
    if grads is None:
        grads = _plain.new_grads(inp.d, inp.ffn)
    outs = []
    for x, dy in zip(inp.x, inp.dy):
        y, h, a_q, n_q, r = forward(x, inp.gamma, inp.w1, inp.w2, inp.eps)
        dx = backward(dy, x, inp.gamma, inp.w1, inp.w2, h, a_q, n_q, r, grads)
        outs.append({"y": y, "h": h, "r": r, "dx": dx})
    if inp.grad_scale is not None:
        _plain.scale_grads(grads, inp.grad_scale)
    return outs, grads
