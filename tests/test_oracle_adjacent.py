"""Pins of the adjacent-step oracle (step-size preprocessing and z-gate)
against things other than itself: central finite differences of its own
forward, closed-form values, the identity and clamp special cases, and
library routines (scipy's expit, numpy's log1p on moderate arguments)."""
import math

import numpy as np
import pytest

import oracle.adjacent as adj


def fd(f, x, eps=1e-6):
    g = np.zeros_like(x)
    for i in np.ndindex(x.shape):
        xp, xm = x.copy(), x.copy()
        xp[i] += eps
        xm[i] -= eps
        g[i] = (f(xp) - f(xm)) / (2 * eps)
    return g


@pytest.mark.parametrize("use_softplus,lo,hi", [(True, 0.0, np.inf), (True, 0.05, 1.5), (False, -np.inf, np.inf),
                                                (False, -0.5, 0.7)])
def test_dt_finite_differences(use_softplus, lo, hi):
    rng = np.random.default_rng(3)
    raw = rng.normal(size=(7, 5)) * 2
    bias = rng.normal(size=5)
    w = rng.normal(size=(7, 5))
    # keep every value away from the clamp kinks so the difference quotient is smooth
    s = adj.dt_fwd(raw, bias, use_softplus, -np.inf, np.inf)
    for bound in (lo, hi):
        if np.isfinite(bound):
            raw = np.where(np.abs(s - bound) < 1e-3, raw + 0.01, raw)
    ddt_raw, ddt_bias = adj.dt_bwd(raw, w, bias, use_softplus, lo, hi)
    loss_raw = lambda r: float(np.sum(adj.dt_fwd(r, bias, use_softplus, lo, hi) * w))
    loss_bias = lambda b: float(np.sum(adj.dt_fwd(raw, b, use_softplus, lo, hi) * w))
    np.testing.assert_allclose(ddt_raw, fd(loss_raw, raw), rtol=1e-7, atol=1e-9)
    np.testing.assert_allclose(ddt_bias, fd(loss_bias, bias), rtol=1e-7, atol=1e-9)


def test_dt_closed_forms():
    # softplus(0) = ln 2 with slope 1/2; without bias, softplus or clamp the map is the identity
    assert adj.dt_fwd(np.zeros((1, 1)))[0, 0] == pytest.approx(math.log(2.0), rel=1e-15)
    r, b = adj.dt_bwd(np.zeros((1, 1)), np.ones((1, 1)))
    assert r[0, 0] == pytest.approx(0.5, rel=1e-15) and b[0] == pytest.approx(0.5, rel=1e-15)
    x = np.linspace(-3, 3, 12).reshape(4, 3)
    np.testing.assert_array_equal(adj.dt_fwd(x, None, False, -np.inf, np.inf), x)
    r, b = adj.dt_bwd(x, x, None, False, -np.inf, np.inf)
    np.testing.assert_array_equal(r, x)
    np.testing.assert_allclose(b, x.sum(axis=0), rtol=1e-15)
    # softplus against log1p(exp(v)) where that is well conditioned, and its slope against expit
    scipy_special = pytest.importorskip("scipy.special")
    v = np.linspace(-30, 30, 61)
    np.testing.assert_allclose(adj.softplus(v), np.log1p(np.exp(v)), rtol=1e-14)
    np.testing.assert_allclose(adj.sigmoid(v), scipy_special.expit(v), rtol=1e-15)
    # large arguments: softplus(v) -> v, far below: softplus(v) -> e^v
    assert adj.softplus(np.array([800.0]))[0] == 800.0
    assert adj.softplus(np.array([-800.0]))[0] == pytest.approx(math.exp(-800.0))


def test_dt_clamp_blocks_gradient_outside_only():
    raw = np.array([[-5.0, 0.0, 5.0]])
    lo, hi = 0.1, 2.0
    dt = adj.dt_fwd(raw, None, True, lo, hi)
    np.testing.assert_allclose(dt, [[lo, math.log(2.0), hi]], rtol=1e-15)
    r, _ = adj.dt_bwd(raw, np.ones_like(raw), None, True, lo, hi)
    np.testing.assert_allclose(r, [[0.0, 0.5, 0.0]], rtol=1e-15)
    # exactly on the bound the gradient passes (identity map, bound hit exactly)
    r, _ = adj.dt_bwd(np.array([[0.25, 0.75]]), np.ones((1, 2)), None, False, 0.25, 0.75)
    np.testing.assert_array_equal(r, [[1.0, 1.0]])


def test_gate_finite_differences_and_closed_forms():
    rng = np.random.default_rng(5)
    y = rng.normal(size=(6, 4))
    z = rng.normal(size=(6, 4)) * 3
    g = rng.normal(size=(6, 4))
    dy, dz = adj.gate_bwd(y, z, g)
    np.testing.assert_allclose(dy, fd(lambda a: float(np.sum(adj.gate_fwd(a, z) * g)), y), rtol=1e-7, atol=1e-9)
    np.testing.assert_allclose(dz, fd(lambda a: float(np.sum(adj.gate_fwd(y, a) * g)), z), rtol=1e-7, atol=1e-9)
    # silu(0) = 0 with slope 1/2; silu(z) -> z for large z, -> 0 for very negative z
    one = np.ones((1, 1))
    assert adj.gate_fwd(one, np.zeros((1, 1)))[0, 0] == 0.0
    assert adj.gate_bwd(one, np.zeros((1, 1)), one)[1][0, 0] == pytest.approx(0.5, rel=1e-15)
    assert adj.gate_fwd(one, np.array([[40.0]]))[0, 0] == pytest.approx(40.0, rel=1e-15)
    assert abs(adj.gate_fwd(one, np.array([[-40.0]]))[0, 0]) < 1e-15
