"""Pins for the oracle's V network, expectile loss and policy."""
import os

import numpy as np
import pytest
import scipy.special
import torch

from oracle import iql

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _constants():
    out = {}
    with open(os.path.join(GOLDEN, "constants.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                out[k] = float(v)
    return out


def _net(rng, s, h, scale=1.0):
    p = h * s + h + h * h + h + h + 1
    return rng.uniform(-scale, scale, size=p)


def test_zero_weights_give_constant_v():
    s, h = 6, 5
    flat = np.zeros(h * s + h + h * h + h + h + 1)
    flat[-1] = 0.375
    x = np.random.default_rng(0).standard_normal((9, s))
    v, _ = iql.forward(flat, x, s, h)
    assert np.all(v == 0.375)
    # only b3 receives gradient when every weight is zero (ReLU(0) is inactive)
    qt = np.random.default_rng(1).standard_normal(9)
    _, loss, grad = iql.value_fwd_bwd(flat, x, qt, 0.7, s, h)
    assert np.count_nonzero(grad[:-1]) == 0
    d = qt - 0.375
    w = np.where(d >= 0, 0.7, 0.3)
    assert grad[-1] == pytest.approx(np.sum(-2 * w * d) / 9, rel=1e-12)


def test_linear_regime_closed_form():
    # positive inputs, positive weights and biases: every ReLU is active, the
    # network is affine and V = w3 W2 W1 x + w3 W2 b1 + w3 b2 + b3
    rng = np.random.default_rng(2)
    s, h = 7, 6
    flat = np.abs(_net(rng, s, h)) + 0.01
    x = np.abs(rng.standard_normal((11, s))) + 0.01
    w1, b1, w2, b2, w3, b3 = iql.unflatten(flat, s, h)
    a = w3 @ w2 @ w1
    c = w3 @ w2 @ b1 + w3 @ b2 + b3
    want = (x @ a.T)[:, 0] + c[0]
    v, _ = iql.forward(flat, x, s, h)
    np.testing.assert_allclose(v, want, rtol=1e-12)


def _torch_reference(flat, x, qt, tau, s, h):
    t = torch.tensor(flat, dtype=torch.float64, requires_grad=True)
    o = 0
    w1 = t[o:o + h * s].view(h, s); o += h * s
    b1 = t[o:o + h]; o += h
    w2 = t[o:o + h * h].view(h, h); o += h * h
    b2 = t[o:o + h]; o += h
    w3 = t[o:o + h].view(1, h); o += h
    b3 = t[o:o + 1]
    xx = torch.tensor(x, dtype=torch.float64)
    v = torch.nn.functional.linear(
        torch.relu(torch.nn.functional.linear(torch.relu(torch.nn.functional.linear(xx, w1, b1)), w2, b2)),
        w3, b3).squeeze(1)
    d = torch.tensor(qt, dtype=torch.float64) - v
    wgt = torch.where(d >= 0, torch.full_like(d, tau), torch.full_like(d, 1 - tau))
    loss = (wgt * d * d).mean()
    loss.backward()
    return v.detach().numpy(), float(loss.detach()), t.grad.numpy()


@pytest.mark.parametrize("s,h,b,tau", [(6, 5, 4, 0.7), (48, 64, 33, 0.9), (50, 128, 70, 0.5)])
def test_against_torch_autograd(s, h, b, tau):
    rng = np.random.default_rng(s * 1000 + h)
    flat = _net(rng, s, h, scale=np.sqrt(6.0 / max(s, h)))
    x = rng.standard_normal((b, s))
    qt = rng.standard_normal(b) * 2
    v, loss, grad = iql.value_fwd_bwd(flat, x, qt, tau, s, h)
    tv, tl, tg = _torch_reference(flat, x, qt, tau, s, h)
    np.testing.assert_allclose(v, tv, rtol=1e-12, atol=1e-14)
    assert loss == pytest.approx(tl, rel=1e-12)
    np.testing.assert_allclose(grad, tg, rtol=1e-10, atol=1e-14)


def test_finite_differences_tiny_net():
    rng = np.random.default_rng(4)
    s, h, b, tau = 6, 5, 4, 0.7
    for _ in range(20):
        flat = _net(rng, s, h)
        x = rng.standard_normal((b, s))
        qt = rng.standard_normal(b) * 2
        v, act = iql.forward(flat, x, s, h)
        d = qt - v
        # no ReLU kink or expectile switch within reach of the step
        if (np.abs(act["z1"]).min() > 1e-3 and np.abs(act["z2"]).min() > 1e-3
                and np.abs(d).min() > 1e-3):
            break
    else:
        pytest.skip("no well-conditioned draw")
    _, _, grad = iql.value_fwd_bwd(flat, x, qt, tau, s, h)
    eps = 1e-6
    fd = np.empty_like(flat)
    for i in range(flat.size):
        e = np.zeros_like(flat)
        e[i] = eps
        lp = iql.value_fwd_bwd(flat + e, x, qt, tau, s, h)[1]
        lm = iql.value_fwd_bwd(flat - e, x, qt, tau, s, h)[1]
        fd[i] = (lp - lm) / (2 * eps)
    np.testing.assert_allclose(grad, fd, rtol=1e-6, atol=1e-9)


def test_expectile_half_is_half_mse():
    rng = np.random.default_rng(5)
    q, v = rng.standard_normal(100), rng.standard_normal(100)
    loss, _ = iql.expectile_loss(q, v, 0.5)
    assert loss == pytest.approx(0.5 * np.mean((q - v) ** 2), rel=1e-13)


def test_expectile_asymmetry():
    c = _constants()
    tau = c["tau_default"]
    rng = np.random.default_rng(6)
    d = np.abs(rng.standard_normal(50)) + 0.1
    v = rng.standard_normal(50)
    up, _ = iql.expectile_loss(v + d, v, tau)      # every diff positive
    down, _ = iql.expectile_loss(v - d, v, tau)    # every diff negative
    assert down / up == pytest.approx((1 - tau) / tau, rel=1e-12)
    assert up > down   # tau > 0.5 penalises underestimation of Q more


def test_expectile_hand_example():
    # d = (0, 2, -1): weights (tau, tau, 1 - tau) = (0.8, 0.8, 0.2)
    loss, dv = iql.expectile_loss(np.array([1.0, 2.0, -1.0]), np.array([1.0, 0.0, 0.0]), 0.8)
    assert loss == pytest.approx((0.8 * 4.0 + 0.2 * 1.0) / 3, rel=1e-15)
    np.testing.assert_allclose(dv, [0.0, -2 * 0.8 * 2.0 / 3, -2 * 0.2 * -1.0 / 3], rtol=1e-15)


def test_expectile_dv_by_finite_differences():
    rng = np.random.default_rng(7)
    q, v = rng.standard_normal(8), rng.standard_normal(8)
    _, dv = iql.expectile_loss(q, v, 0.7)
    for i in range(8):
        e = np.zeros(8)
        e[i] = 1e-6
        fd = (iql.expectile_loss(q, v + e, 0.7)[0] - iql.expectile_loss(q, v - e, 0.7)[0]) / 2e-6
        assert dv[i] == pytest.approx(fd, rel=1e-6, abs=1e-12)


def test_policy_properties():
    c = _constants()
    beta, clamp = c["beta_default"], c["adv_clamp"]
    rng = np.random.default_rng(8)
    q = rng.standard_normal((500, 9)) * 6
    v = rng.standard_normal(500) * 3
    pi, am = iql.policy(q, v, beta)
    np.testing.assert_allclose(pi.sum(axis=1), 1.0, atol=1e-14)
    assert (pi > 0).all() and (pi <= 1).all()
    assert (pi.max(axis=1) / pi.min(axis=1)).max() <= np.exp(2 * clamp * beta) * (1 + 1e-12)
    # an independent softmax on the clamped, scaled advantages
    ref = scipy.special.softmax(beta * np.clip(q - v[:, None], -clamp, clamp), axis=1)
    np.testing.assert_allclose(pi, ref, rtol=1e-12, atol=1e-300)
    adv = np.clip(q - v[:, None], -clamp, clamp)
    for r in range(500):
        top = adv[r].max()
        assert am[r] == min(i for i in range(9) if adv[r, i] == top)


def test_policy_degenerate_cases():
    q = np.array([[20.0, 30.0, 40.0], [-50.0, -60.0, -70.0], [0.1, 0.2, 0.3]])
    v = np.zeros(3)
    pi, am = iql.policy(q, v, 3.0)
    # all advantages clamped at +10 (row 0) or -10 (row 1): uniform, lowest index
    np.testing.assert_allclose(pi[0], 1 / 3, rtol=1e-15)
    np.testing.assert_allclose(pi[1], 1 / 3, rtol=1e-15)
    assert am[0] == 0 and am[1] == 0 and am[2] == 2
    pi0, _ = iql.policy(q, v, 0.0)
    np.testing.assert_allclose(pi0, 1 / 3, rtol=1e-15)


def test_backward_abs_bounds_and_equality():
    rng = np.random.default_rng(9)
    s, h, b = 7, 6, 20
    flat = _net(rng, s, h)
    x = rng.standard_normal((b, s))
    qt = rng.standard_normal(b) * 2
    v, act = iql.forward(flat, x, s, h)
    _, dv = iql.expectile_loss(qt, v, 0.7)
    g = iql.backward(flat, act, dv, s, h)
    ga = iql.backward_abs(flat, act, dv, s, h)
    assert (np.abs(g) <= ga * (1 + 1e-12) + 1e-300).all()
    # one-signed terms everywhere: positive inputs, weights and dv -> equality
    flat = np.abs(flat) + 0.01
    x = np.abs(x) + 0.01
    v, act = iql.forward(flat, x, s, h)
    dv = np.abs(rng.standard_normal(b)) + 0.01
    g = iql.backward(flat, act, dv, s, h)
    ga = iql.backward_abs(flat, act, dv, s, h)
    np.testing.assert_allclose(np.abs(g), ga, rtol=1e-12)


# ---- IQL target r + gamma (1 - done) V(s') ----------------------------------

def _target_case(seed=3, b=9, s=6, h=5):
    rng = np.random.default_rng(seed)
    flat = rng.standard_normal(h * s + h + h * h + h + h + 1)
    xs = rng.standard_normal((b, s))
    r = rng.standard_normal(b)
    d = (rng.random(b) < 0.4).astype(np.float64)
    return flat, xs, r, d, s, h


def test_target_terminal_rows_bootstrap_nothing():
    flat, xs, r, _, s, h = _target_case()
    t, _ = iql.iql_target(flat, xs, r, np.ones_like(r), 0.99, s, h)
    assert np.array_equal(t, r)


def test_target_gamma_zero_is_the_reward():
    flat, xs, r, d, s, h = _target_case(seed=4)
    t, _ = iql.iql_target(flat, xs, r, d, 0.0, s, h)
    assert np.array_equal(t, r)


def test_target_zero_weights_closed_form():
    # W1 = W2 = W3 = 0: V = b3 for every state, so target = r + gamma (1 - d) b3
    flat, xs, r, d, s, h = _target_case(seed=5)
    w1, b1, w2, b2, w3, b3 = iql.unflatten(flat, s, h)
    flat0 = iql.flatten(np.zeros_like(w1), b1, np.zeros_like(w2), b2, np.zeros_like(w3), b3)
    t, v = iql.iql_target(flat0, xs, r, d, 0.9, s, h)
    assert np.allclose(v, b3[0], rtol=0, atol=0)
    assert np.allclose(t, r + 0.9 * (1.0 - d) * b3[0], rtol=1e-15, atol=0)


def test_target_mixes_rows_by_done_flag():
    # rows with done = 0 carry gamma V(s'); rows with done = 1 do not
    flat, xs, r, d, s, h = _target_case(seed=6, b=40)
    t, v = iql.iql_target(flat, xs, r, d, 0.5, s, h)
    live = d == 0.0
    assert live.any() and (~live).any()
    assert np.allclose(t[live] - r[live], 0.5 * v[live], rtol=1e-14, atol=1e-15)
    assert np.array_equal(t[~live], r[~live])
