"""Pins of the FP8 (E4M3) oracle (CPU): the format against an independent
conversion (torch.float8_e4m3fn) and the values its definition fixes, the
quantisation error bound, power-of-two scale invariance, the block's FP8
variant against the plain float64 block within the FP8 error, and planted
mistakes that must each fail a pin."""

import numpy as np
import pytest

import oracle
import synth
from oracle import fp8


def test_e4m3_values_fixed_by_the_format():
    cases = {
        1.0: 1.0, 1.0625: 1.0, 1.1875: 1.25,            # ties to even
        448.0: 448.0, 449.0: 448.0, 470.0: 448.0, 1e6: 448.0,   # largest finite, saturation
        2.0 ** -6: 2.0 ** -6,                             # smallest normal
        2.0 ** -9: 2.0 ** -9, 2.0 ** -10: 0.0,           # smallest subnormal; tie to 0
        1.5 * 2.0 ** -9: 2.0 ** -8,                       # subnormal tie to even
        0.3: 0.3125, 3.3: 3.25, 0.0: 0.0,
    }
    for v, q in cases.items():
        assert fp8.e4m3(np.array([v]))[0] == q, v
        assert fp8.e4m3(np.array([-v]))[0] == -q, -v


def test_e4m3_matches_an_independent_conversion():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    v = np.concatenate([rng.standard_normal(4000) * s for s in (1e-3, 0.1, 3.0, 60.0)]).astype(np.float32)
    v = v[np.abs(v) < 448]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(fp8.e4m3(v), ref)


def test_quantisation_error_bound():
    rng = np.random.default_rng(6)
    v = (rng.standard_normal(10000) * 7.0).astype(np.float32)
    q, s = fp8.quantize(v)
    u = v.astype(np.float64) / float(s)
    normal = np.abs(u) >= 2.0 ** -6
    # half a spacing: 2^-4 relative for normals, 2^-10 absolute (scaled) for subnormals
    assert np.all(np.abs(q - v)[normal] <= 2.0 ** -4 * np.abs(v)[normal] * (1 + 1e-6))
    assert np.all(np.abs(q - v)[~normal] <= 2.0 ** -10 * float(s) * (1 + 1e-6))
    assert np.max(np.abs(q)) == pytest.approx(np.max(np.abs(v)), rel=1e-6)  # amax maps to 448


def test_power_of_two_scales_are_absorbed():
    rng = np.random.default_rng(7)
    v = (rng.standard_normal(500)).astype(np.float32)
    q1, s1 = fp8.quantize(v)
    q2, s2 = fp8.quantize(v * np.float32(8.0))
    np.testing.assert_array_equal(q2, 8.0 * q1)
    assert s2 == 8 * s1


def _fp8_vs_plain(inp):
    outs8, g8 = fp8.run_workload(inp)
    outs, g = oracle.run_workload(inp)
    errs = {}
    for i, (a, b) in enumerate(zip(outs8, outs)):
        errs[f"y{i}"] = oracle.scaled_error(a["y"] - inp.x[i], b["y"] - inp.x[i])   # the MLP branch
        errs[f"h{i}"] = oracle.scaled_error(a["h"], b["h"])
        errs[f"dx{i}"] = oracle.scaled_error(a["dx"] - inp.dy[i], b["dx"] - inp.dy[i])
    for k in g:
        errs[k] = oracle.scaled_error(g8[k], g[k])
    return errs


def test_fp8_block_is_the_block_within_fp8_error():
    inp = synth.make_inputs(tokens=96, d=64, ffn=192, dtype="bf16", seed=12, n_mb=2, eps=1e-6)
    # a gamma far from 1, so that a gamma mistake is not hidden in the FP8 error
    inp.gamma = synth.round_to_bf16(np.linspace(0.25, 2.0, inp.d).astype(np.float32))
    errs = _fp8_vs_plain(inp)
    # E4M3 keeps 3 mantissa bits: each operand carries up to 2^-4 relative error,
    # so products and sums stay within a few percent of the exact block
    assert max(errs.values()) < 0.12, errs
    assert min(errs.values()) > 1e-4, errs   # and they do differ: the operands were quantised


def test_block_evaluation_with_whole_tensor_scales_is_the_whole_evaluation():
    """Row blocks quantised with the whole tensors' scales (block_amaxes, then
    forward / backward with a_amax, dy_amax, dh_amax) give the whole
    microbatch's rows and, summed over the blocks, its gradients."""
    inp = synth.make_inputs(tokens=200, d=64, ffn=192, dtype="bf16", seed=23, n_mb=1, eps=1e-6)
    whole_outs, whole_g = fp8.run_workload(inp)
    x, dy = inp.x[0], inp.dy[0]
    dy_amax = np.float32(np.max(np.abs(dy.astype(np.float32))))
    spans = [(i, min(200, i + 64)) for i in range(0, 200, 64)]
    am = [fp8.block_amaxes(x[a:b], dy[a:b], inp.gamma, inp.w1, inp.w2, inp.eps, dy_amax) for a, b in spans]
    a_amax, dh_amax = max(v[0] for v in am), max(v[1] for v in am)
    g = oracle.new_grads(inp.d, inp.ffn)
    rows = {"y": [], "h": [], "dx": []}
    for a, b in spans:
        y, h, a_q, n_q, r = fp8.forward(x[a:b], inp.gamma, inp.w1, inp.w2, inp.eps, a_amax)
        dx = fp8.backward(dy[a:b], x[a:b], inp.gamma, inp.w1, inp.w2, h, a_q, n_q, r, g, dy_amax, dh_amax)
        rows["y"].append(y)
        rows["h"].append(h)
        rows["dx"].append(dx)
    for k in rows:
        assert oracle.scaled_error(np.concatenate(rows[k]), whole_outs[0][k]) <= 1e-12, k
    for k in g:
        assert oracle.scaled_error(g[k], whole_g[k]) <= 1e-12, k
    # and a block's own maxima would not do: the scales differ
    local = fp8.block_amaxes(x[:64], dy[:64], inp.gamma, inp.w1, inp.w2, inp.eps, dy_amax)
    assert local != (a_amax, dh_amax)


# ------------------------------------------ the recipe against a plain recipe

def _q_torch(v):
    """Per-tensor E4M3 quantisation through torch's float8_e4m3fn conversion (an
    implementation independent of oracle.fp8): dequantised values."""
    torch = pytest.importorskip("torch")
    v32 = np.asarray(v, dtype=np.float32)
    amax = np.float32(np.max(np.abs(v32)))
    scale = np.float32(448.0) / amax
    codes = torch.from_numpy((v32 * scale).astype(np.float32)).to(torch.float8_e4m3fn).to(torch.float64)
    return codes.numpy() / np.float64(scale)


def _bf16(a):
    torch = pytest.importorskip("torch")
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def _plain_recipe(x, dy, gamma, w1, w2, eps):
    """The block with every GEMM operand quantised where it plainly stands:
    n = x*r*gamma with its own amax scale, W1 alone, dW1 = dh^T . n.  Written
    here, not taken from oracle.fp8, so that the oracle's recipe (gamma folded
    into W1, n' = x*r at scale 1, dW1 = (dh^T . n') * gamma) is checked against
    a second one."""
    x = np.asarray(x, dtype=np.float64)
    r = (1.0 / np.sqrt(np.mean(x * x, axis=1) + eps)).astype(np.float32).astype(np.float64)
    n = (x * r[:, None] * np.asarray(gamma, np.float64)[None, :]).astype(np.float32)
    n_q, w1_q, w2_q = _q_torch(n), _q_torch(w1), _q_torch(w2)
    h = n_q @ w1_q.T
    a_q = _q_torch(_bf16(np.where(h > 0, h, 0.0) ** 2))
    y = x + a_q @ w2_q.T
    dy_q = _q_torch(dy)
    hk = _bf16(h)
    dh_q = _q_torch(_bf16((dy_q @ w2_q) * 2.0 * np.where(hk > 0, hk, 0.0)))
    dn = dh_q @ w1_q
    dx_norm, dgamma = oracle.rmsnorm_backward(dn, x, gamma, r)
    return {"y": y, "dx": np.asarray(dy, np.float64) + dx_norm,
            "dw1": dh_q.T @ n_q, "dw2": dy_q.T @ a_q, "dgamma": dgamma}


def test_recipe_is_as_accurate_as_the_plain_recipe():
    """Folding gamma into W1 before quantising (and n' at scale 1) is an operand
    choice: against the exact float64 block its error is the plain recipe's,
    tensor by tensor, within a factor of two; the two recipes differ by no more
    than FP8 rounding."""
    inp = synth.make_inputs(tokens=256, d=128, ffn=384, dtype="bf16", seed=14, n_mb=1, eps=1e-6)
    inp.gamma = synth.round_to_bf16(np.linspace(0.3, 1.9, inp.d).astype(np.float32))
    x, dy = inp.x[0], inp.dy[0]
    exact_outs, exact_g = oracle.run_workload(inp)
    fold_outs, fold_g = fp8.run_workload(inp)
    plain = _plain_recipe(x, dy, inp.gamma, inp.w1, inp.w2, inp.eps)
    exact = {"y": exact_outs[0]["y"] - x, "dx": exact_outs[0]["dx"] - dy, **exact_g}
    fold = {"y": fold_outs[0]["y"] - x, "dx": fold_outs[0]["dx"] - dy, **fold_g}
    plain = {**plain, "y": plain["y"] - x, "dx": plain["dx"] - dy}
    for k in exact:
        e_fold = oracle.scaled_error(fold[k], exact[k])
        e_plain = oracle.scaled_error(plain[k], exact[k])
        assert 0.5 * e_plain <= e_fold <= 2.0 * e_plain, (k, e_fold, e_plain)
        assert oracle.scaled_error(fold[k], plain[k]) <= 2.0 * max(e_fold, e_plain), k


# ------------------------------------------------------------- planted mistakes

def _pins_pass():
    try:
        test_e4m3_values_fixed_by_the_format()
        test_quantisation_error_bound()
        test_power_of_two_scales_are_absorbed()
        test_fp8_block_is_the_block_within_fp8_error()
    except AssertionError:
        return False
    return True


def _no_dequant(v):
    q, s = _orig_quantize(v)
    return q / float(s), s          # codes used as values: the scale is dropped


def _no_ties_to_even(u):
    u = np.asarray(u, dtype=np.float64)
    a = np.abs(u)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    sp = np.exp2(np.maximum(ex - 1, -6) - 3)
    return np.copysign(np.minimum(np.floor(a / sp + 0.5) * sp, 448.0), u)


def _no_saturation(u):
    u = np.asarray(u, dtype=np.float64)
    a = np.abs(u)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    sp = np.exp2(np.maximum(ex - 1, -6) - 3)
    return np.copysign(np.rint(a / sp) * sp, u)


_orig_quantize = fp8.quantize
_orig_forward = fp8.forward
_orig_backward = fp8.backward


def _w1_without_gamma(x, gamma, w1, w2, eps):
    return _orig_forward(x, np.ones_like(np.asarray(gamma)), w1, w2, eps)


def _dw1_without_gamma(dy, x, gamma, w1, w2, h, a_q, n_q, r, grads):
    before = grads["dw1"].copy()
    dx = _orig_backward(dy, x, gamma, w1, w2, h, a_q, n_q, r, grads)
    grads["dw1"] = before + (grads["dw1"] - before) / np.asarray(gamma, dtype=np.float64)[None, :]
    return dx


def _gate_sign(dy, x, gamma, w1, w2, h, a_q, n_q, r, grads):
    return _orig_backward(dy, x, gamma, w1, w2, -h, a_q, n_q, r, grads)


@pytest.mark.parametrize("name, attr, bad", [
    ("scale not applied", "quantize", _no_dequant),
    ("ties away from zero", "e4m3", _no_ties_to_even),
    ("no saturation", "e4m3", _no_saturation),
    ("gamma not folded into W1", "forward", _w1_without_gamma),
    ("dW1 without gamma", "backward", _dw1_without_gamma),
    ("gate on -h", "backward", _gate_sign),
])
def test_planted_mistakes_are_caught(monkeypatch, name, attr, bad):
    assert _pins_pass()
    monkeypatch.setattr(fp8, attr, bad)
    assert not _pins_pass(), f"planted mistake not caught: {name}"
