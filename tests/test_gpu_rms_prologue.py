"""The forward with the RMSNorm statistic computed inside the W1 GEMM's prologue
(mlpblk_set_rmsnorm_mode(MLPBLK_RMSNORM_IN_W1_PROLOGUE)) against the float64
oracle, and against the default statistics-pass forward (GB300 only)."""

import numpy as np
import pytest

import oracle
import synth
from helpers import TOL, compare, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _prologue_mode():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mlp_block_backprop_gb300 as mb
    mb.mlpblk_set_rmsnorm_mode(mb.MLPBLK_RMSNORM_IN_W1_PROLOGUE)
    try:
        yield mb
    finally:
        mb.mlpblk_set_rmsnorm_mode(mb.MLPBLK_RMSNORM_STATS_PASS)
    assert mb.mlpblk_last_error() == mb.MLPBLK_OK


@pytest.mark.parametrize("case", ["small_bf16_accum4", "block_120m"])
def test_prologue_configs(case):
    inp = synth.config_inputs(case)
    outs, grads, _ = run_gpu(inp)
    ref_outs, ref_grads = oracle.run_workload(inp)
    compare(outs, grads, ref_outs, ref_grads, TOL[inp.dtype])


@pytest.mark.parametrize("shape", [(333, 200, 328), (1, 256, 512), (40, 8, 8), (77, 136, 1032)])
def test_prologue_ragged(shape):
    T, d, F = shape
    inp = synth.make_inputs(tokens=T, d=d, ffn=F, dtype="bf16", seed=T + d + F, n_mb=2, eps=1e-5)
    outs, grads, _ = run_gpu(inp)
    ref_outs, ref_grads = oracle.run_workload(inp)
    compare(outs, grads, ref_outs, ref_grads, TOL["bf16"])


def test_prologue_matches_statistics_pass(_prologue_mode):
    mb = _prologue_mode
    inp = synth.make_inputs(tokens=520, d=520, ffn=520, dtype="bf16", seed=9, n_mb=1, eps=1e-6)
    outs_p, _, _ = run_gpu(inp)
    mb.mlpblk_set_rmsnorm_mode(mb.MLPBLK_RMSNORM_STATS_PASS)
    outs_s, _, _ = run_gpu(inp)
    mb.mlpblk_set_rmsnorm_mode(mb.MLPBLK_RMSNORM_IN_W1_PROLOGUE)
    # rstd: the same float32 statistic up to summation order
    r_p, r_s = outs_p[0]["rstd"], outs_s[0]["rstd"]
    assert np.max(np.abs(r_p - r_s) / np.abs(r_s)) <= 1e-6
    for k in ("y", "h", "a", "dx"):
        assert oracle.scaled_error(outs_p[0][k], outs_s[0][k]) <= 1e-2, k
