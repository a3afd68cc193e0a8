"""Pins of the optimizer-side oracle (CPU): library special cases, closed forms,
an independent implementation (torch.optim.AdamW, float64) as a black box, and
planted mistakes that must each fail a pin."""

import copy

import numpy as np
import pytest

from oracle import optim


def _grads(seed, shapes=((7,), (5, 9), (9, 5))):
    rng = np.random.default_rng(seed)
    return [rng.standard_normal(s) * (i + 1) for i, s in enumerate(shapes)]


def test_grad_norm_is_the_l2_norm_of_the_concatenation():
    gs = _grads(1)
    flat = np.concatenate([g.ravel() for g in gs])
    assert optim.grad_norm(gs) == pytest.approx(np.linalg.norm(flat), rel=1e-14)


def test_grad_norm_closed_forms():
    assert optim.grad_norm([np.full(4, 3.0), np.full(9, 4.0 / 3.0)]) == pytest.approx(np.sqrt(36 + 16))
    assert optim.grad_norm([np.zeros(3)]) == 0.0


def test_clip_coefficient():
    assert optim.clip_coefficient(0.5, 1.0) == 1.0          # below the bound: untouched
    assert optim.clip_coefficient(2.0, 1.0) == pytest.approx(0.5, rel=1e-6)
    c = optim.clip_coefficient(10.0, 2.5)
    gs = [np.full(3, 10.0 / np.sqrt(3.0))]                   # global norm 10
    optim.scale(gs, c)
    assert optim.grad_norm(gs) == pytest.approx(2.5, rel=1e-6)


def _torch_adamw(w0, grads, lr, b1, b2, eps, wd):
    torch = pytest.importorskip("torch")
    p = torch.nn.Parameter(torch.tensor(w0, dtype=torch.float64))
    opt = torch.optim.AdamW([p], lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd)
    for g in grads:
        p.grad = torch.tensor(g, dtype=torch.float64)
        opt.step()
    st = opt.state[p]
    return p.detach().numpy(), st["exp_avg"].numpy(), st["exp_avg_sq"].numpy()


@pytest.mark.parametrize("wd", [0.0, 0.1])
def test_adamw_matches_an_independent_implementation(wd):
    rng = np.random.default_rng(7)
    w0 = rng.standard_normal(64)
    grads = [rng.standard_normal(64) * s for s in (1.0, 0.1, 3.0, 1e-3, 0.5)]
    lr, b1, b2, eps = 1e-2, 0.9, 0.95, 1e-8
    w, m, v = w0.copy(), np.zeros(64), np.zeros(64)
    for t, g in enumerate(grads, start=1):
        optim.adamw_step(w, g, m, v, t, lr, b1, b2, eps, wd)
    wt, mt, vt = _torch_adamw(w0, grads, lr, b1, b2, eps, wd)
    np.testing.assert_allclose(w, wt, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(m, mt, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(v, vt, rtol=1e-13, atol=1e-15)


def test_adamw_closed_forms():
    # first step: m_hat = g, v_hat = g^2, so the update is lr * g / (|g| + eps)
    g = np.array([2.0, -0.5, 1e-3, 0.0])
    w, m, v = np.ones(4), np.zeros(4), np.zeros(4)
    optim.adamw_step(w, g, m, v, 1, 0.1, 0.9, 0.999, 1e-8, 0.0)
    np.testing.assert_allclose(w, 1.0 - 0.1 * g / (np.abs(g) + 1e-8), rtol=1e-12)
    # zero gradient, decay only: w_t = w_0 (1 - lr wd)^t
    w, m, v = np.full(3, 2.0), np.zeros(3), np.zeros(3)
    for t in range(1, 6):
        optim.adamw_step(w, np.zeros(3), m, v, t, 0.01, 0.9, 0.999, 1e-8, 0.5)
    np.testing.assert_allclose(w, 2.0 * (1 - 0.005) ** 5, rtol=1e-14)
    # a constant gradient keeps m_hat = g and v_hat = g^2 at every step
    w, m, v = np.zeros(1), np.zeros(1), np.zeros(1)
    for t in range(1, 4):
        optim.adamw_step(w, np.array([4.0]), m, v, t, 0.1, 0.8, 0.9, 0.0, 0.0)
    np.testing.assert_allclose(w, [-0.3], rtol=1e-12)


def test_round_to_bf16():
    one = 1.0
    assert optim.round_to_bf16(np.array([one]))[0] == 1.0
    assert optim.round_to_bf16(np.array([1 + 2.0 ** -8]))[0] == 1.0                 # tie -> even
    assert optim.round_to_bf16(np.array([1 + 3 * 2.0 ** -8]))[0] == 1 + 2.0 ** -6  # tie -> even
    assert optim.round_to_bf16(np.array([1 + 2.0 ** -8 + 2.0 ** -12]))[0] == 1 + 2.0 ** -7
    assert optim.round_to_bf16(np.array([-3.0]))[0] == -3.0
    torch = pytest.importorskip("torch")
    x = np.random.default_rng(3).standard_normal(1000).astype(np.float32) * 37
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(optim.round_to_bf16(x), ref)


# ------------------------------------------------------------- planted mistakes

def _pins_pass():
    """True when every pin above passes for the current optim module."""
    try:
        test_grad_norm_is_the_l2_norm_of_the_concatenation()
        test_grad_norm_closed_forms()
        test_clip_coefficient()
        for wd in (0.0, 0.1):
            test_adamw_matches_an_independent_implementation(wd)
        test_adamw_closed_forms()
    except AssertionError:
        return False
    return True


def _no_bias_correction(w, g, m, v, step, lr, b1, b2, eps, wd):
    w *= 1.0 - lr * wd
    m *= b1; m += (1 - b1) * g
    v *= b2; v += (1 - b2) * g * g
    w -= lr * m / (np.sqrt(v) + eps)


def _decay_after_update(w, g, m, v, step, lr, b1, b2, eps, wd):
    m *= b1; m += (1 - b1) * g
    v *= b2; v += (1 - b2) * g * g
    w -= (lr / (1 - b1 ** step)) * m / (np.sqrt(v) / np.sqrt(1 - b2 ** step) + eps)
    w *= 1.0 - lr * wd


def _eps_inside_root(w, g, m, v, step, lr, b1, b2, eps, wd):
    w *= 1.0 - lr * wd
    m *= b1; m += (1 - b1) * g
    v *= b2; v += (1 - b2) * g * g
    w -= (lr / (1 - b1 ** step)) * m / np.sqrt(v / (1 - b2 ** step) + eps)


def _betas_swapped(w, g, m, v, step, lr, b1, b2, eps, wd):
    w *= 1.0 - lr * wd
    m *= b2; m += (1 - b2) * g
    v *= b1; v += (1 - b1) * g * g
    w -= (lr / (1 - b2 ** step)) * m / (np.sqrt(v) / np.sqrt(1 - b1 ** step) + eps)


def _coupled_l2(w, g, m, v, step, lr, b1, b2, eps, wd):
    g = g + wd * w   # L2 folded into the gradient (Adam, not AdamW)
    m *= b1; m += (1 - b1) * g
    v *= b2; v += (1 - b2) * g * g
    w -= (lr / (1 - b1 ** step)) * m / (np.sqrt(v) / np.sqrt(1 - b2 ** step) + eps)


@pytest.mark.parametrize("name, attr, bad", [
    ("no bias correction", "adamw_step", _no_bias_correction),
    ("decay after the update", "adamw_step", _decay_after_update),
    ("eps inside the root", "adamw_step", _eps_inside_root),
    ("betas swapped", "adamw_step", _betas_swapped),
    ("L2 instead of decoupled decay", "adamw_step", _coupled_l2),
    ("norm without the root", "grad_norm", lambda gs: sum(float(np.sum(np.asarray(g) ** 2)) for g in gs)),
    ("clip not capped at 1", "clip_coefficient", lambda n, mx: mx / (n + 1e-6)),
])
def test_planted_mistakes_are_caught(monkeypatch, name, attr, bad):
    pytest.importorskip("torch")
    assert _pins_pass()
    monkeypatch.setattr(optim, attr, bad)
    assert not _pins_pass(), f"planted mistake not caught: {name}"
