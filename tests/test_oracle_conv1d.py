"""Pins of the causal-conv1d oracle against things other than itself: central
finite differences of its own forward, torch's conv1d differentiated by
autograd (an independent route, fp64 on the CPU), a hand-expanded two-tap
example, closed forms (width 1, an impulse kernel) and the packed-sequence
invariant (a packed batch equals the separate runs)."""
import numpy as np
import pytest
import torch

import oracle.conv1d as cv


def fd(f, x, eps=1e-6):
    g = np.zeros_like(x)
    for i in np.ndindex(x.shape):
        xp, xm = x.copy(), x.copy()
        xp[i] += eps
        xm[i] -= eps
        g[i] = (f(xp) - f(xm)) / (2 * eps)
    return g


def _case(b, T, C, K, seed):
    rng = np.random.default_rng(seed)
    return (rng.normal(size=(b, T, C)), rng.normal(size=(C, K)) * 0.7, rng.normal(size=C) * 0.3,
            rng.normal(size=(b, T, C)))


@pytest.mark.parametrize("activation", ["silu", "none"])
@pytest.mark.parametrize("K", [1, 3, 4])
@pytest.mark.parametrize("with_seq", [False, True])
def test_finite_differences(activation, K, with_seq):
    b = 1 if with_seq else 2
    x, w, bias, dy = _case(b, 10, 3, K, seed=K + 7 * with_seq)
    seq = np.array([[0, 0, 0, 0, 1, 1, 1, 2, 2, 2]], np.int32) if with_seq else None
    dx, dw, db = cv.bwd(x, w, dy, bias, seq, activation)
    loss = lambda xx, ww, bb: float(np.sum(cv.fwd(xx, ww, bb, seq, activation) * dy))
    np.testing.assert_allclose(dx, fd(lambda v: loss(v, w, bias), x), rtol=1e-7, atol=1e-9)
    np.testing.assert_allclose(dw, fd(lambda v: loss(x, v, bias), w), rtol=1e-7, atol=1e-9)
    np.testing.assert_allclose(db, fd(lambda v: loss(x, w, v), bias), rtol=1e-7, atol=1e-9)


@pytest.mark.parametrize("activation", ["silu", "none"])
def test_against_torch_conv1d_autograd(activation):
    # depthwise conv1d (groups = channels) with K-1 zeros of left padding is the causal window
    x, w, bias, dy = _case(3, 37, 5, 4, seed=11)
    xt = torch.tensor(x, requires_grad=True)
    wt = torch.tensor(w, requires_grad=True)
    bt = torch.tensor(bias, requires_grad=True)
    pre = torch.nn.functional.conv1d(torch.nn.functional.pad(xt.transpose(1, 2), (3, 0)), wt.unsqueeze(1), bt,
                                     groups=5).transpose(1, 2)
    y = torch.nn.functional.silu(pre) if activation == "silu" else pre
    (y * torch.tensor(dy)).sum().backward()
    np.testing.assert_allclose(cv.fwd(x, w, bias, None, activation), y.detach().numpy(), rtol=1e-12, atol=1e-12)
    dx, dw, db = cv.bwd(x, w, dy, bias, None, activation)
    np.testing.assert_allclose(dx, xt.grad.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dw, wt.grad.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(db, bt.grad.numpy(), rtol=1e-12, atol=1e-12)


def test_two_taps_by_hand():
    # T = 3, one channel, w = [a, b] (tap 0 reads t-1, tap 1 reads t), no bias or activation:
    # y = [b x0, a x0 + b x1, a x1 + b x2]
    a, bb = 0.5, -2.0
    x = np.array([[[1.0], [3.0], [-1.0]]])
    dy = np.array([[[2.0], [1.0], [4.0]]])
    y = cv.fwd(x, np.array([[a, bb]]), None, None, "none")
    np.testing.assert_array_equal(y.reshape(-1), [-2.0, 0.5 - 6.0, 1.5 + 2.0])
    dx, dw, db = cv.bwd(x, np.array([[a, bb]]), dy, None, None, "none")
    np.testing.assert_array_equal(dx.reshape(-1), [bb * 2 + a * 1, bb * 1 + a * 4, bb * 4])
    np.testing.assert_array_equal(dw.reshape(-1), [1 * 1 + 4 * 3, 2 * 1 + 1 * 3 + 4 * -1])
    np.testing.assert_array_equal(db, [7.0])


def test_width_one_is_elementwise():
    x, w, bias, dy = _case(2, 6, 4, 1, seed=3)
    pre = x * w[:, 0] + bias
    s = 1 / (1 + np.exp(-pre))
    np.testing.assert_allclose(cv.fwd(x, w, bias), pre * s, rtol=1e-14)
    dpre = dy * s * (1 + pre * (1 - s))
    dx, dw, db = cv.bwd(x, w, dy, bias)
    np.testing.assert_allclose(dx, dpre * w[:, 0], rtol=1e-13)
    np.testing.assert_allclose(dw[:, 0], (dpre * x).sum(axis=(0, 1)), rtol=1e-13)
    np.testing.assert_allclose(db, dpre.sum(axis=(0, 1)), rtol=1e-13)


def test_impulse_kernel_is_identity():
    x, _, _, dy = _case(1, 9, 3, 4, seed=5)
    w = np.zeros((3, 4))
    w[:, 3] = 1.0                       # the tap that reads token t itself
    np.testing.assert_array_equal(cv.fwd(x, w, None, None, "none"), x)
    dx, dw, db = cv.bwd(x, w, dy, None, None, "none")
    np.testing.assert_array_equal(dx, dy)
    for k in range(4):                  # dw[c, k] = sum_t dy[t] x[t - 3 + k]
        lag = 3 - k
        ref = (dy[0, lag:, :] * x[0, :9 - lag, :]).sum(axis=0)
        np.testing.assert_allclose(dw[:, k], ref, rtol=1e-13)


def test_packed_sequences_equal_separate_runs():
    lens = (5, 1, 7, 3)
    T = sum(lens)
    x, w, bias, dy = _case(1, T, 3, 4, seed=9)
    seq = np.repeat(np.arange(len(lens)), lens).astype(np.int32)[None, :]
    y = cv.fwd(x, w, bias, seq)
    dx, dw, db = cv.bwd(x, w, dy, bias, seq)
    off, dw_sum, db_sum = 0, np.zeros_like(dw), np.zeros_like(db)
    for L in lens:
        sl = slice(off, off + L)
        np.testing.assert_allclose(y[:, sl], cv.fwd(x[:, sl], w, bias), rtol=1e-14)
        dxs, dws, dbs = cv.bwd(x[:, sl], w, dy[:, sl], bias)
        np.testing.assert_allclose(dx[:, sl], dxs, rtol=1e-13, atol=1e-15)
        dw_sum += dws
        db_sum += dbs
        off += L
    np.testing.assert_allclose(dw, dw_sum, rtol=1e-12)
    np.testing.assert_allclose(db, db_sum, rtol=1e-12)
