"""Pins of the routed ReLU² expert oracle (CPU): the dense block as the one-expert
special case, linearity in the mixture weights, central finite differences of
L = sum(dy * y) for every input, reverse-mode AD of an independent restatement,
zero gradients for experts nobody selected, slot-order invariance, and planted
mistakes that must each fail a pin."""

import numpy as np
import pytest

import oracle
from oracle import moe


def _case(seed, T=5, d=6, F=8, E=3, k=2, eps=1e-6):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, d))
    gamma = 1.0 + 0.3 * rng.standard_normal(d)
    w1s = rng.standard_normal((E, F, d)) / np.sqrt(d)
    w2s = rng.standard_normal((E, d, F)) / np.sqrt(F)
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)])
    p = rng.uniform(0.2, 1.0, size=(T, k))
    dy = rng.standard_normal((T, d))
    return x, gamma, w1s, w2s, idx, p, dy, eps


def _run(x, gamma, w1s, w2s, idx, p, dy, eps):
    y, h, o, r = moe.forward(x, gamma, w1s, w2s, idx, p, eps)
    g = moe.new_grads(w1s.shape[0], x.shape[1], w1s.shape[1])
    dx, dp = moe.backward(dy, x, gamma, w1s, w2s, idx, p, h, o, r, g)
    return y, h, dx, dp, g


def test_one_expert_is_the_dense_block():
    x, gamma, w1s, w2s, _, _, dy, eps = _case(1, E=1, k=1)
    idx = np.zeros((x.shape[0], 1), dtype=int)
    p = np.ones((x.shape[0], 1))
    y, h, dx, _, g = _run(x, gamma, w1s, w2s, idx, p, dy, eps)
    yd, hd, _, rd = oracle.forward(x, gamma, w1s[0], w2s[0], eps)
    gd = oracle.new_grads(x.shape[1], w1s.shape[1])
    dxd = oracle.backward(dy, x, gamma, w1s[0], w2s[0], hd, rd, gd)
    np.testing.assert_allclose(y, yd, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(h[:, 0], hd, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dx, dxd, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["dw1"][0], gd["dw1"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["dw2"][0], gd["dw2"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["dgamma"], gd["dgamma"], rtol=1e-12, atol=1e-12)


def test_two_identical_experts_add_their_weights():
    x, gamma, w1s, w2s, _, _, dy, eps = _case(2, E=2, k=2)
    w1s[1], w2s[1] = w1s[0], w2s[0]
    T = x.shape[0]
    idx = np.tile([0, 1], (T, 1))
    p = np.random.default_rng(3).uniform(0.1, 1.0, size=(T, 2))
    y, _, _, _, _ = _run(x, gamma, w1s, w2s, idx, p, dy, eps)
    yd, _, _, _ = oracle.forward(x, gamma, w1s[0], w2s[0], eps)
    np.testing.assert_allclose(y - x, (yd - x) * (p[:, 0] + p[:, 1])[:, None], rtol=1e-12, atol=1e-12)


def _loss(args):
    x, gamma, w1s, w2s, idx, p, dy, eps = args
    y, _, _, _ = moe.forward(x, gamma, w1s, w2s, idx, p, eps)
    return float(np.sum(dy * y))


def test_finite_differences():
    args = list(_case(4))
    y, h, dx, dp, g = _run(*args)
    assert np.min(np.abs(h)) > 1e-3   # away from the ReLU² kink
    step = 1e-6
    for pos, name, got in ((0, "x", dx), (5, "p", dp), (1, "gamma", g["dgamma"]), (2, "w1", g["dw1"]),
                           (3, "w2", g["dw2"])):
        base = np.array(args[pos], dtype=np.float64)
        num = np.zeros_like(base)
        it = np.nditer(base, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            plus, minus = list(args), list(args)
            bp, bm = base.copy(), base.copy()
            bp[i] += step
            bm[i] -= step
            plus[pos], minus[pos] = bp, bm
            num[i] = (_loss(plus) - _loss(minus)) / (2 * step)
        np.testing.assert_allclose(got, num, rtol=1e-5, atol=1e-7, err_msg=name)


def test_unselected_experts_get_no_gradient():
    x, gamma, w1s, w2s, _, p, dy, eps = _case(5, E=4, k=2)
    idx = np.tile([2, 0], (x.shape[0], 1))   # experts 1 and 3 unused
    _, _, _, _, g = _run(x, gamma, w1s, w2s, idx, p, dy, eps)
    for e in (1, 3):
        assert not np.any(g["dw1"][e]) and not np.any(g["dw2"][e])
    assert np.any(g["dw1"][0]) and np.any(g["dw2"][2])


def test_slot_order_does_not_matter():
    x, gamma, w1s, w2s, idx, p, dy, eps = _case(6)
    y, _, dx, dp, g = _run(x, gamma, w1s, w2s, idx, p, dy, eps)
    y2, _, dx2, dp2, g2 = _run(x, gamma, w1s, w2s, idx[:, ::-1], p[:, ::-1], dy, eps)
    np.testing.assert_allclose(y2, y, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dx2, dx, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dp2, dp[:, ::-1], rtol=1e-12, atol=1e-12)
    for k in g:
        np.testing.assert_allclose(g2[k], g[k], rtol=1e-12, atol=1e-12)


def test_backward_matches_torch_autograd():
    """Reverse-mode AD (torch, float64) of an independent restatement of the
    routed forward, against the oracle's hand-derived backward for every input,
    at a size where tokens take three of five experts."""
    torch = pytest.importorskip("torch")
    x, gamma, w1s, w2s, idx, p, dy, eps = _case(11, T=29, d=20, F=24, E=5, k=3, eps=1e-5)
    y, _, dx, dp, g = _run(x, gamma, w1s, w2s, idx, p, dy, eps)
    t = {name: torch.tensor(v, dtype=torch.float64, requires_grad=True)
         for name, v in (("x", x), ("gamma", gamma), ("w1s", w1s), ("w2s", w2s), ("p", p))}
    xx = t["x"]
    n = xx * torch.rsqrt(xx.pow(2).mean(dim=1, keepdim=True) + eps) * t["gamma"]
    e = torch.as_tensor(idx, dtype=torch.long)
    hh = torch.einsum("tjfd,td->tjf", t["w1s"][e], n)                   # every slot's expert
    oo = torch.einsum("tjdf,tjf->tjd", t["w2s"][e], torch.relu(hh).pow(2))
    yy = xx + (t["p"].unsqueeze(-1) * oo).sum(dim=1)
    yy.backward(torch.tensor(dy, dtype=torch.float64))
    assert oracle.scaled_error(y, yy.detach().numpy()) <= 1e-13
    for name, got, ref in (("dx", dx, t["x"].grad), ("dp", dp, t["p"].grad), ("dgamma", g["dgamma"], t["gamma"].grad),
                           ("dw1", g["dw1"], t["w1s"].grad), ("dw2", g["dw2"], t["w2s"].grad)):
        assert oracle.scaled_error(got, ref.numpy()) <= 1e-12, name


# ------------------------------------------------------------- planted mistakes

def _pins_pass():
    try:
        test_one_expert_is_the_dense_block()
        test_two_identical_experts_add_their_weights()
        test_finite_differences()
        test_unselected_experts_get_no_gradient()
        test_slot_order_does_not_matter()
        test_backward_matches_torch_autograd()
    except AssertionError:
        return False
    return True


_orig_backward = moe.backward
_orig_forward = moe.forward


def _dp_from_dx(dy, x, gamma, w1s, w2s, idx, p, h, o, r, grads):
    dx, dp = _orig_backward(dy, x, gamma, w1s, w2s, idx, p, h, o, r, grads)
    return dx, dp * 0.5 + 0.5 * np.einsum("td,tjd->tj", dy, o) * p   # weight leaks into its own gradient


def _no_weight_on_expert_grad(dy, x, gamma, w1s, w2s, idx, p, h, o, r, grads):
    return _orig_backward(dy, x, gamma, w1s, w2s, idx, np.ones_like(p), h, o, r, grads)[0], \
        np.einsum("td,tjd->tj", dy, o)


def _last_slot_only(dy, x, gamma, w1s, w2s, idx, p, h, o, r, grads):
    q = np.array(p, dtype=np.float64).copy()
    q[:, :-1] = 0.0                                   # sum rule dropped: one expert reaches dn
    dx, _ = _orig_backward(dy, x, gamma, w1s, w2s, idx, q, h, o, r, grads)
    return dx, np.einsum("td,tjd->tj", dy, o)


def _unweighted_combine(x, gamma, w1s, w2s, idx, p, eps):
    return _orig_forward(x, gamma, w1s, w2s, idx, np.ones_like(np.asarray(p, dtype=np.float64)), eps)


@pytest.mark.parametrize("name, attr, bad", [
    ("d_routing_weights scaled by the weight", "backward", _dp_from_dx),
    ("expert gradient without its weight", "backward", _no_weight_on_expert_grad),
    ("only the last slot reaches dn", "backward", _last_slot_only),
    ("combine without the weights", "forward", _unweighted_combine),
])
def test_planted_mistakes_are_caught(monkeypatch, name, attr, bad):
    assert _pins_pass()
    monkeypatch.setattr(moe, attr, bad)
    assert not _pins_pass(), f"planted mistake not caught: {name}"
