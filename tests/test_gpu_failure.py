"""Failure detection on the GPU without faulting it: a host-set test fault makes
the W1 GEMM issue no operand loads, its bounded pipeline waits run out (about
2 s), the kernel unwinds and reports MLPBLK_ETIMEOUT, and the same context then
computes a correct block again."""

import pytest

import oracle
import synth
from helpers import TOL, compare, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mb():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mlp_block_backprop_gb300
    return mlp_block_backprop_gb300


def test_bounded_wait_reports_timeout_and_context_survives(mb):
    import time

    import torch
    inp = synth.make_inputs(tokens=256, d=128, ffn=256, seed=21)
    assert mb.mlpblk_last_error() == mb.MLPBLK_OK
    mb.mlpblk_set_test_fault(mb.MLPBLK_TEST_FAULT_SKIP_LOADS)
    t0 = time.perf_counter()
    run_gpu(inp, keep_outputs=False)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert mb.mlpblk_last_error() == mb.MLPBLK_ETIMEOUT
    assert 1.0 < waited < 30.0, waited
    assert mb.mlpblk_last_error() == mb.MLPBLK_OK  # cleared once read
    outs, grads, _ = run_gpu(inp)
    ref_outs, ref_grads = oracle.run_workload(inp)
    compare(outs, grads, ref_outs, ref_grads, TOL["bf16"])
    assert mb.mlpblk_last_error() == mb.MLPBLK_OK


def test_unknown_fault_is_rejected(mb):
    with pytest.raises(mb.MlpBlkError):
        mb.mlpblk_set_test_fault(7)
