"""Pins of the float64 oracle to things other than itself (CPU only).

Each ``check_*`` function takes an oracle module (the real one, or a copy with a
planted mistake) and raises AssertionError when the pin does not hold:

* the hand-derived worked example in ``golden/worked_example.txt``;
* central finite differences of L = sum(dy * y) for every parameter and input;
* closed forms: relu(h)² and its derivative at special points, the unit RMS of
  the normalised rows, eps = 0 scale invariance;
* the RMSNorm backward invariant x·dx_norm = r³·eps·Σ(ĝ·x) per row;
* the residual rule (W2 = 0 gives y = x, dx = dy and zero dW1, dγ);
* a zero upstream gradient leaves the gradient buffers bitwise unchanged;
* accumulation: microbatch A then B equals the concatenated batch [A; B].

``test_planted_mistakes_are_caught`` plants plausible mistakes into copies of
the oracle's source and requires every one of them to fail at least one pin.
The backward is also compared with torch float64 autograd used as a black box.
"""

import os
import types

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _parse_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, rest = line.split(None, 1)
            rows = [[float(t) for t in part.split()] for part in rest.split("|")]
            vals[key] = np.array(rows if len(rows) > 1 else rows[0])
    return vals


def _tiny_inputs(seed, T, d, F, eps=1e-6, h_margin=1e-3):
    """Random float64 inputs whose pre-activations all stay away from the ReLU² kink."""
    rng = np.random.default_rng(seed)
    for _ in range(1000):
        x = rng.standard_normal((T, d))
        gamma = 1.0 + 0.3 * rng.standard_normal(d)
        w1 = rng.standard_normal((F, d)) / np.sqrt(d)
        w2 = rng.standard_normal((d, F)) / np.sqrt(F)
        dy = rng.standard_normal((T, d))
        _, h, _, _ = oracle.forward(x, gamma, w1, w2, eps)
        if np.min(np.abs(h)) > h_margin:
            return x, gamma, w1, w2, dy
    raise RuntimeError("could not draw inputs away from h = 0")


# ----------------------------------------------------------------------------- pins

def check_worked_example(O):
    g = _parse_golden("worked_example.txt")
    x = g["x"][None, :]
    dy = g["dy"][None, :]
    y, h, a, r = O.forward(x, g["gamma"], g["w1"], g["w2"], float(g["eps"][0]))
    grads = O.new_grads(4, 2)
    dx = O.backward(dy, x, g["gamma"], g["w1"], g["w2"], h, r, grads)
    for name, got, want in [("r", r, g["r"]), ("h", h[0], g["h"]), ("a", a[0], g["a"]),
                            ("y", y[0], g["y"]), ("dx", dx[0], g["dx"]),
                            ("dgamma", grads["dgamma"], g["dgamma"]),
                            ("dw1", grads["dw1"], g["dw1"]), ("dw2", grads["dw2"], g["dw2"])]:
        got = np.asarray(got, dtype=np.float64).reshape(np.shape(want))
        assert np.allclose(got, want, rtol=0, atol=1e-12), (name, got, want)


def _loss(O, x, gamma, w1, w2, dy, eps):
    y, _, _, _ = O.forward(x, gamma, w1, w2, eps)
    return float(np.sum(dy * y))


def check_finite_differences(O, seed=11, T=4, d=8, F=16, eps=1e-6, tol=1e-6):
    x, gamma, w1, w2, dy = _tiny_inputs(seed, T, d, F, eps)
    _, h, _, r = O.forward(x, gamma, w1, w2, eps)
    grads = O.new_grads(d, F)
    dx = O.backward(dy, x, gamma, w1, w2, h, r, grads)
    analytic = {"x": dx, "gamma": grads["dgamma"], "w1": grads["dw1"], "w2": grads["dw2"]}
    params = {"x": x, "gamma": gamma, "w1": w1, "w2": w2}
    for name, p in params.items():
        fd = np.zeros_like(p)
        for idx in np.ndindex(p.shape):
            old = p[idx]
            step = 1e-6 * max(1.0, abs(old))
            p[idx] = old + step
            lp = _loss(O, params["x"], params["gamma"], params["w1"], params["w2"], dy, eps)
            p[idx] = old - step
            lm = _loss(O, params["x"], params["gamma"], params["w1"], params["w2"], dy, eps)
            p[idx] = old
            fd[idx] = (lp - lm) / (2 * step)
        err = oracle.scaled_error(analytic[name], fd)
        assert err <= tol, (name, err)


def check_relu_squared_closed_form(O):
    h = np.array([-1.0, -0.0, 0.0, 1e-300, 2.0, 3.5])
    assert np.array_equal(O.relu_squared(h), [0.0, 0.0, 0.0, 0.0, 4.0, 12.25])
    assert np.array_equal(O.relu_squared_grad(h), [0.0, 0.0, 0.0, 2e-300, 4.0, 7.0])


def check_rmsnorm_closed_forms(O):
    rng = np.random.default_rng(5)
    x = rng.standard_normal((6, 10)) * rng.uniform(0.1, 10.0, size=(6, 1))
    ones = np.ones(10)
    n, r = O.rmsnorm_forward(x, ones, 0.0)
    # unit root-mean-square rows when gamma = 1 and eps = 0
    assert np.allclose(np.mean(n * n, axis=1), 1.0, rtol=0, atol=1e-12)
    # scale invariance with eps = 0
    n2, r2 = O.rmsnorm_forward(3.0 * x, ones, 0.0)
    assert np.allclose(n2, n, rtol=0, atol=1e-12)
    assert np.allclose(r2 * 3.0, r, rtol=1e-12, atol=0)
    # a constant row c with eps: r = 1/sqrt(c² + eps)
    nc, rc = O.rmsnorm_forward(np.full((1, 4), 2.0), ones[:4], 0.5)
    assert abs(rc[0] - 1.0 / np.sqrt(4.5)) < 1e-15
    # d = 1, eps = 0: n = sign(x)·gamma
    n1, _ = O.rmsnorm_forward(np.array([[-7.0], [0.25]]), np.array([1.5]), 0.0)
    assert np.allclose(n1[:, 0], [-1.5, 1.5], rtol=0, atol=1e-15)


def check_rmsnorm_backward_invariant(O):
    rng = np.random.default_rng(6)
    for eps in (0.0, 0.3):
        x = rng.standard_normal((5, 12))
        gamma = 1.0 + 0.2 * rng.standard_normal(12)
        dn = rng.standard_normal((5, 12))
        _, r = O.rmsnorm_forward(x, gamma, eps)
        dxn, _ = O.rmsnorm_backward(dn, x, gamma, r)
        lhs = np.sum(x * dxn, axis=1)
        rhs = r ** 3 * eps * np.sum(dn * gamma[None, :] * x, axis=1)
        assert np.allclose(lhs, rhs, rtol=1e-12, atol=1e-12), (eps, lhs, rhs)


def check_residual_rule(O):
    x, gamma, w1, w2, dy = _tiny_inputs(21, 5, 6, 9)
    w2 = np.zeros_like(w2)
    y, h, a, r = O.forward(x, gamma, w1, w2, 1e-6)
    assert np.array_equal(y, x)
    grads = O.new_grads(6, 9)
    dx = O.backward(dy, x, gamma, w1, w2, h, r, grads)
    assert np.array_equal(dx, dy)
    assert not np.any(grads["dw1"]) and not np.any(grads["dgamma"])
    assert np.allclose(grads["dw2"], dy.T @ a, rtol=1e-12, atol=0)


def check_zero_upstream(O):
    x, gamma, w1, w2, _ = _tiny_inputs(22, 5, 6, 9)
    y, h, a, r = O.forward(x, gamma, w1, w2, 1e-6)
    grads = O.new_grads(6, 9)
    rng = np.random.default_rng(1)
    for k in grads:
        grads[k][...] = rng.standard_normal(grads[k].shape)
    before = {k: v.copy() for k, v in grads.items()}
    dx = O.backward(np.zeros_like(x), x, gamma, w1, w2, h, r, grads)
    assert not np.any(dx)
    for k in grads:
        assert np.array_equal(grads[k], before[k]), k


def check_accumulation(O):
    xa, gamma, w1, w2, dya = _tiny_inputs(31, 4, 6, 10)
    xb, _, _, _, dyb = _tiny_inputs(32, 3, 6, 10)
    eps = 1e-6
    g_seq = O.new_grads(6, 10)
    for x, dy in ((xa, dya), (xb, dyb)):
        _, h, _, r = O.forward(x, gamma, w1, w2, eps)
        O.backward(dy, x, gamma, w1, w2, h, r, g_seq)
    g_cat = O.new_grads(6, 10)
    x = np.concatenate([xa, xb])
    dy = np.concatenate([dya, dyb])
    _, h, _, r = O.forward(x, gamma, w1, w2, eps)
    O.backward(dy, x, gamma, w1, w2, h, r, g_cat)
    for k in g_seq:
        assert oracle.scaled_error(g_seq[k], g_cat[k]) <= 1e-12, k
    # A then A equals 2 x A; the 1/n scale then gives back one A
    g_one = O.new_grads(6, 10)
    _, h, _, r = O.forward(xa, gamma, w1, w2, eps)
    O.backward(dya, xa, gamma, w1, w2, h, r, g_one)
    g_two = O.new_grads(6, 10)
    for _ in range(2):
        O.backward(dya, xa, gamma, w1, w2, h, r, g_two)
    O.scale_grads(g_two, 0.5)
    for k in g_one:
        assert oracle.scaled_error(g_two[k], g_one[k]) <= 1e-15, k


ALL_CHECKS = [check_worked_example, check_finite_differences, check_relu_squared_closed_form,
              check_rmsnorm_closed_forms, check_rmsnorm_backward_invariant, check_residual_rule,
              check_zero_upstream, check_accumulation]


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check(oracle)


def test_finite_differences_ragged_shape_large_eps():
    check_finite_differences(oracle, seed=12, T=3, d=5, F=7, eps=0.1)


# ------------------------------------------------------------- planted mistakes

MUTANTS = {
    "eps_outside_root": ("r = 1.0 / np.sqrt(mean_sq + eps)", "r = 1.0 / (np.sqrt(mean_sq) + eps)"),
    "sum_not_mean": ("mean_sq = np.sum(x * x, axis=1) / d", "mean_sq = np.sum(x * x, axis=1)"),
    "relu_not_squared": ("    return r * r\n", "    return r\n"),
    "gate_missing_2": ("return 2.0 * relu(h)", "return relu(h)"),
    "no_forward_residual": ("y = x + a @ _f64(w2).T", "y = a @ _f64(w2).T"),
    "no_backward_residual": ("return dy + dx_norm", "return dx_norm"),
    "residual_sign": ("return dy + dx_norm", "return dy - dx_norm"),
    "norm_bwd_no_mean_term": ("dx_norm = r[:, None] * (g - xhat * mean_gx[:, None])",
                              "dx_norm = r[:, None] * g"),
    "norm_bwd_mean_term_sign": ("dx_norm = r[:, None] * (g - xhat * mean_gx[:, None])",
                                "dx_norm = r[:, None] * (g + xhat * mean_gx[:, None])"),
    "norm_bwd_no_gamma": ("g = dn * gamma[None, :]", "g = dn"),
    "dgamma_unnormalised_x": ("dgamma = np.sum(dn * xhat, axis=0)", "dgamma = np.sum(dn * x, axis=0)"),
    "dw1_from_x_not_n": ('grads["dw1"] += dh.T @ n', 'grads["dw1"] += dh.T @ x'),
    "dw2_transposed": ('grads["dw2"] += dy.T @ a', 'grads["dw2"] += (a.T @ dy).T.T'),
    "gate_on_activation": ("dh = da * relu_squared_grad(h)", "dh = da * relu_squared_grad(a)"),
    "dn_through_w2": ("dn = dh @ w1", "dn = dh @ w2.T"),
}


def _mutant(old, new):
    src = open(oracle.__file__).read()
    assert src.count(old) == 1, old
    mod = types.ModuleType("oracle_mutant")
    exec(compile(src.replace(old, new), "oracle_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_are_caught(name):
    mod = _mutant(*MUTANTS[name])
    failed = []
    for check in ALL_CHECKS:
        try:
            check(mod)
        except Exception:  # an assertion or a shape error both count as caught
            failed.append(check.__name__)
    assert failed, f"planted mistake {name!r} passes every pin"


# ------------------------------------------------ torch float64 autograd black box

def _torch_grads(x, gamma, w1, w2, dy, eps):
    torch = pytest.importorskip("torch")
    t = {k: torch.tensor(v, dtype=torch.float64, requires_grad=True)
         for k, v in dict(x=x, gamma=gamma, w1=w1, w2=w2).items()}
    xx = t["x"]
    rr = torch.rsqrt(xx.pow(2).mean(dim=1, keepdim=True) + eps)
    n = xx * rr * t["gamma"]
    h = torch.nn.functional.linear(n, t["w1"])
    y = xx + torch.nn.functional.linear(torch.relu(h).pow(2), t["w2"])
    y.backward(torch.tensor(dy, dtype=torch.float64))
    return {k: v.grad.numpy() for k, v in t.items()}, y.detach().numpy()


@pytest.mark.parametrize("case", ["tiny_fp32", "ragged"])
def test_backward_matches_torch_autograd(case):
    if case == "tiny_fp32":
        inp = synth.config_inputs("tiny_fp32")
    else:
        inp = synth.make_inputs(tokens=37, d=24, ffn=40, dtype="f32", seed=9, eps=1e-3)
    x = inp.x[0].astype(np.float64)
    dy = inp.dy[0].astype(np.float64)
    gamma, w1, w2 = (inp.gamma.astype(np.float64), inp.w1.astype(np.float64),
                     inp.w2.astype(np.float64))
    tg, ty = _torch_grads(x, gamma, w1, w2, dy, inp.eps)
    y, h, a, r = oracle.forward(x, gamma, w1, w2, inp.eps)
    grads = oracle.new_grads(inp.d, inp.ffn)
    dx = oracle.backward(dy, x, gamma, w1, w2, h, r, grads)
    assert oracle.scaled_error(y, ty) <= 1e-13
    assert oracle.scaled_error(dx, tg["x"]) <= 1e-12
    assert oracle.scaled_error(grads["dgamma"], tg["gamma"]) <= 1e-12
    assert oracle.scaled_error(grads["dw1"], tg["w1"]) <= 1e-12
    assert oracle.scaled_error(grads["dw2"], tg["w2"]) <= 1e-12


# ------------------------------------------------ why gradient buffers are fp32

def test_bf16_accumulation_loses_contribution():
    g = _parse_golden("bf16_accumulation.txt")
    s = np.float32(g["sum"][0])
    c = np.float32(g["contribution"][0])
    assert synth.round_to_bf16(np.array([s + c], dtype=np.float32))[0] == g["bf16_result"]
    assert np.float32(s + c) == g["f32_result"]
    # 258 is the next bf16 value above 256: one ulp step of 2 at this binade
    assert synth.round_to_bf16(np.array([257.0001], dtype=np.float32))[0] == g["bf16_next_above_256"]
