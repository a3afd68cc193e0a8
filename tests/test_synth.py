"""The seeded input generator: determinism, bf16 rounding and the workload recipe."""

import numpy as np
import pytest

import synth


def test_round_to_bf16_ties_to_even_and_exactness():
    cases = np.array([1.0, 1.00390625, 1.01171875, 1.005859375, -2.5, 3.0e38, 1e-40, 0.0],
                     dtype=np.float32)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: even mantissa (1.0) wins;
    # 1 + 3*2^-8 is a tie between 1+2^-7 and 1+2^-6: even (1+2^-6) wins.
    want = np.array([1.0, 1.0, 1.015625, 1.0078125, -2.5, 2.9999998e38, 1e-40, 0.0],
                    dtype=np.float32)
    got = synth.round_to_bf16(cases)
    assert np.array_equal(got[[0, 1, 2, 3, 4, 7]], want[[0, 1, 2, 3, 4, 7]])
    again = synth.round_to_bf16(got)
    assert np.array_equal(again, got)
    assert np.all((got.view(np.uint32) & 0xFFFF) == 0)


def test_same_seed_same_values_and_draw_order():
    a = synth.make_inputs(tokens=16, d=32, ffn=64, seed=7, n_mb=2)
    b = synth.make_inputs(tokens=16, d=32, ffn=64, seed=7, n_mb=2)
    for u, v in [(a.gamma, b.gamma), (a.w1, b.w1), (a.w2, b.w2), (a.x[1], b.x[1]), (a.dy[0], b.dy[0])]:
        assert np.array_equal(u, v)
    c = synth.make_inputs(tokens=16, d=32, ffn=64, seed=8, n_mb=2)
    assert not np.array_equal(a.x[0], c.x[0])
    # parameters are drawn first, so a different token count leaves them unchanged
    d = synth.make_inputs(tokens=3, d=32, ffn=64, seed=7, n_mb=1)
    assert np.array_equal(a.w2, d.w2)


@pytest.mark.parametrize("name", sorted(synth.CONFIGS))
def test_config_shapes(name):
    c = synth.CONFIGS[name]
    if c["d"] * c["ffn"] > 4096 * 4096:
        pytest.skip("large workload drawn in the GPU tests")
    inp = synth.config_inputs(name)
    assert inp.gamma.shape == (c["d"],)
    assert inp.w1.shape == (c["ffn"], c["d"]) and inp.w2.shape == (c["d"], c["ffn"])
    assert len(inp.x) == c["n_mb"] and inp.x[0].shape == (c["tokens"], c["d"])
    if c["dtype"] == "bf16":
        assert np.all((inp.x[0].view(np.uint32) & 0xFFFF) == 0)
    assert abs(np.std(inp.w1) * np.sqrt(c["d"]) - 1.0) < 0.05
    assert abs(np.std(inp.dy[0]) / c["dy_std"] - 1.0) < 0.05
    assert abs(np.mean(inp.gamma) - 1.0) < 0.01
