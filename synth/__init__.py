"""Seeded synthetic inputs for the pre-norm residual ReLU² MLP block.

This module is the one piece shared by the float64 oracle (``oracle/``) and the
CUDA path (``mlp_block_backprop_gb300``).  It draws numbers and rounds them to the
storage type; it holds none of the block's arithmetic (no normalisation, no
products, no activation), so neither side can borrow the other's maths from it.

Workloads
---------
``CONFIGS`` lists the five block workloads the work is measured and checked on.
The pages print no numeric fixtures for this block, so every input is synthetic:

* ``tiny_fp32``          64 tokens (batch 2 x seq 32), d=128, ffn=512, all fp32
* ``small_bf16_accum4``  4 microbatches x 1024 tokens (batch 4 x seq 256), d=512,
                         ffn=2048, bf16, fp32 grads accumulated then scaled by 1/4
* ``block_120m``         8192 tokens (batch 8 x seq 1024), d=768, ffn=3072, bf16
* ``wide``               16384 tokens (batch 4 x seq 4096), d=2048, ffn=8192, bf16
* ``large_accum2``       2 microbatches x 8192 tokens, d=4096, ffn=16384, bf16

Distributions (the second parameter of N(.,.) is read as a standard deviation,
which is how the weight recipe N(0, 1/sqrt(fan_in)) has to be read):
gamma ~ 1 + N(0, 0.02); W1 ~ N(0, 1/sqrt(d)); W2 ~ N(0, 1/sqrt(ffn));
x ~ N(0, 1); dy ~ N(0, dy_std) with dy_std per workload.

Generator: numpy ``default_rng(seed)`` (PCG64), float32 standard normals, scaled
in float32 (separate multiply and add), then rounded to bfloat16 with
round-to-nearest-even for the bf16 workloads.  Draw order: gamma, W1, W2, then
for each microbatch in order x_mb followed by dy_mb.  Arrays are returned as
float32 holding the exact storage values (bf16-representable for bf16 workloads).
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

EPS = 1e-6

CONFIGS = {
    "tiny_fp32": dict(tokens=64, n_mb=1, d=128, ffn=512, dtype="f32", seed=0,
                      dy_std=1.0, grad_scale=None, shape="batch 2 x seq 32"),
    "small_bf16_accum4": dict(tokens=1024, n_mb=4, d=512, ffn=2048, dtype="bf16", seed=3,
                              dy_std=1.0, grad_scale=0.25, shape="4 microbatches of batch 4 x seq 256"),
    "block_120m": dict(tokens=8192, n_mb=1, d=768, ffn=3072, dtype="bf16", seed=1,
                       dy_std=1e-2, grad_scale=None, shape="batch 8 x seq 1024"),
    "wide": dict(tokens=16384, n_mb=1, d=2048, ffn=8192, dtype="bf16", seed=4,
                 dy_std=1.0, grad_scale=None, shape="batch 4 x seq 4096"),
    "large_accum2": dict(tokens=8192, n_mb=2, d=4096, ffn=16384, dtype="bf16", seed=2,
                         dy_std=1e-3, grad_scale=None, shape="2 microbatches of batch 1 x seq 8192"),
}


def round_to_bf16(v: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); return float32.

    Non-finite inputs are not expected from the generator and are not handled.
    """
    v = np.ascontiguousarray(v, dtype=np.float32)
    u = v.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    u = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return (u.astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_bits(v: np.ndarray) -> np.ndarray:
    """Upper 16 bits of float32 values that are exactly bf16-representable."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    return (v.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


@dataclass
class BlockInputs:
    """One workload's parameters and per-microbatch activations (storage values)."""
    name: str
    tokens: int
    n_mb: int
    d: int
    ffn: int
    dtype: str
    eps: float
    grad_scale: float | None
    gamma: np.ndarray
    w1: np.ndarray
    w2: np.ndarray
    x: list = field(default_factory=list)
    dy: list = field(default_factory=list)


def _draw(rng, shape, mean, std, dtype):
    z = rng.standard_normal(shape, dtype=np.float32)
    v = np.multiply(z, np.float32(std), dtype=np.float32)
    if mean != 0.0:
        v = np.add(v, np.float32(mean), dtype=np.float32)
    return round_to_bf16(v) if dtype == "bf16" else v


def make_inputs(tokens: int, d: int, ffn: int, dtype: str = "bf16", seed: int = 0,
                n_mb: int = 1, dy_std: float = 1.0, x_std: float = 1.0,
                gamma_std: float = 0.02, grad_scale: float | None = None,
                eps: float = EPS, name: str = "custom") -> BlockInputs:
    """Draw a block workload of any size with the recipe described above."""
    if dtype not in ("bf16", "f32"):
        raise ValueError(f"unknown dtype {dtype!r}")
    rng = np.random.default_rng(seed)
    gamma = _draw(rng, (d,), 1.0, gamma_std, dtype)
    w1 = _draw(rng, (ffn, d), 0.0, 1.0 / np.sqrt(d), dtype)
    w2 = _draw(rng, (d, ffn), 0.0, 1.0 / np.sqrt(ffn), dtype)
    xs, dys = [], []
    for _ in range(n_mb):
        xs.append(_draw(rng, (tokens, d), 0.0, x_std, dtype))
        dys.append(_draw(rng, (tokens, d), 0.0, dy_std, dtype))
    return BlockInputs(name=name, tokens=tokens, n_mb=n_mb, d=d, ffn=ffn, dtype=dtype,
                       eps=eps, grad_scale=grad_scale, gamma=gamma, w1=w1, w2=w2,
                       x=xs, dy=dys)


def config_inputs(name: str) -> BlockInputs:
    """Inputs of one named workload from ``CONFIGS``."""
    c = CONFIGS[name]
    return make_inputs(tokens=c["tokens"], d=c["d"], ffn=c["ffn"], dtype=c["dtype"],
                       seed=c["seed"], n_mb=c["n_mb"], dy_std=c["dy_std"],
                       grad_scale=c["grad_scale"], name=name)


def block_flops(tokens: int, d: int, ffn: int, n_mb: int = 1) -> int:
    """Algorithmic tensor work of one forward+backward: six GEMMs of 2*T*d*ffn each."""
    return 12 * tokens * d * ffn * n_mb


# ----------------------------------------------------------- routed experts

MOE_CONFIGS = {
    # 8 experts of ffn 1024, top-2, on 8192 tokens of width 2048
    "moe_e8k2": dict(tokens=8192, d=2048, ffn=1024, experts=8, top_k=2, seed=7, dy_std=1e-2),
}


@dataclass
class MoeInputs:
    """A routed-expert workload (bf16 storage values; routing weights float32)."""
    name: str
    tokens: int
    d: int
    ffn: int
    experts: int
    top_k: int
    eps: float
    gamma: np.ndarray
    w1s: np.ndarray      # [E, ffn, d]
    w2s: np.ndarray      # [E, d, ffn]
    x: np.ndarray
    dy: np.ndarray
    idx: np.ndarray      # [T, k] int32, k distinct experts per token
    p: np.ndarray        # [T, k] float32 in [0.1, 1)


def make_moe_inputs(tokens: int, d: int, ffn: int, experts: int, top_k: int, seed: int = 0,
                    dy_std: float = 1.0, eps: float = EPS, name: str = "custom_moe") -> MoeInputs:
    """Draw order: gamma, W1 of every expert, W2 of every expert, x, dy, the
    routing (k distinct experts per token: the first k of a uniformly random
    ordering), then the weights p ~ U(0.1, 1)."""
    rng = np.random.default_rng(seed)
    gamma = _draw(rng, (d,), 1.0, 0.02, "bf16")
    w1s = _draw(rng, (experts, ffn, d), 0.0, 1.0 / np.sqrt(d), "bf16")
    w2s = _draw(rng, (experts, d, ffn), 0.0, 1.0 / np.sqrt(ffn), "bf16")
    x = _draw(rng, (tokens, d), 0.0, 1.0, "bf16")
    dy = _draw(rng, (tokens, d), 0.0, dy_std, "bf16")
    idx = np.argsort(rng.random((tokens, experts)), axis=1)[:, :top_k].astype(np.int32)
    p = rng.uniform(0.1, 1.0, size=(tokens, top_k)).astype(np.float32)
    return MoeInputs(name=name, tokens=tokens, d=d, ffn=ffn, experts=experts, top_k=top_k, eps=eps,
                     gamma=gamma, w1s=w1s, w2s=w2s, x=x, dy=dy, idx=idx, p=p)


def moe_config_inputs(name: str) -> MoeInputs:
    c = MOE_CONFIGS[name]
    return make_moe_inputs(tokens=c["tokens"], d=c["d"], ffn=c["ffn"], experts=c["experts"],
                           top_k=c["top_k"], seed=c["seed"], dy_std=c["dy_std"], name=name)


def moe_flops(tokens: int, d: int, ffn: int, top_k: int) -> int:
    """Algorithmic tensor work of one forward+backward: six GEMMs per assignment."""
    return 12 * tokens * top_k * d * ffn
